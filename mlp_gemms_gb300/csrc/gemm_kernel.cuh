// The grouped block-scaled GEMM kernel template on the 5th-generation tensor core, with
// fused epilogues: BF16 store, SwiGLU forward (BF16 pre-activation save +
// dual-orientation MXFP8 requant) and dSwiGLU backward (dual requant of dz).
//
// torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP fwd/bwd and wgrad
// group gemm":
//   * shared-infrastructure commit: per-expert row counts are multiples of
//     128 so no tile straddles an expert; the expert of a tile is found from
//     its integer row base, with no per-group tensor-map updates; the
//     blocked scale layout has a constant 512-byte K stride per 128-row
//     block, so the scale chunk of (row block, K block) is one address;
//   * correctness-first kernels commit: FC1 grouped GEMM + SwiGLU + dual
//     (1x32 rowwise, 32x1 columnwise) MXFP8 RCEIL quantization + BF16
//     pre-activation save in one launch; FC2 dgrad + dSwiGLU + dual
//     quantization in one launch; ragged-K wgrad with BF16 output where a
//     zero-token expert gets zeros.
//
// Kernel organisation (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: A/B tiles (128-byte swizzled, K-major) and the
//               512-byte scale chunks into a ring of shared-memory stages;
//   warp 1      owns tensor memory; one lane copies each stage's scale
//               chunks into tensor memory (tcgen05.cp 32x128b.warpx4) and
//               issues tcgen05.mma .kind::mxf8f6f4.block_scale (M=128, N=BN,
//               K=32 per instruction, fp32 accumulators in tensor memory),
//               or .kind::mxf4 for packed E2M1 operands (F4: K=64 per
//               instruction, a stage holds 256 K-elements and two scale
//               chunks per 128-row block);
//   warps 2..    epilogue (8 warps, 12 for the dense GELU / dGELU ones at
//               BN = 256): tcgen05.ld of the accumulator (warp w reads
//               lanes 32*(w%4)..+31, the warps of a lane quarter split the
//               columns), then the fused math and stores; dSwiGLU adds a
//               loader warp that streams the saved z by TMA.
// With BN = 256 there is one accumulator buffer; the epilogue copies it to
// registers (plain, SwiGLU) or parks part of it in unused tensor-memory
// columns (dSwiGLU, GELU / dGELU) and releases it before its math, so the
// next tile's MMAs run under the epilogue.  With BN = 128 two accumulator
// buffers alternate.
// Every wait is bounded in time; on expiry the kernel records a device
// status bit and unwinds without leaving copies or MMAs in flight.
#pragma once
#include "mx_common.cuh"
#include "mx_internal.h"
#include "pair_common.cuh"

namespace mx {

// One status word per translation unit that instantiates the kernel.
static __device__ unsigned g_gemm_status = 0;

constexpr int EPI_THREADS = 256;
// Threads of one CTA: the dSwiGLU epilogue adds a warp that streams the saved
// pre-activation z into shared memory.
// Epilogue warps: two per tensor-memory lane quarter, three for the dense
// GELU / dGELU epilogues at BN = 256 (the heaviest per output element; their
// tiles' columns are dealt round-robin to the quarter's warps).
template <int BN, int EPI> constexpr int kEpiWarps() {
  return (BN == 256 && (EPI == EPI_GELU || EPI == EPI_DGELU)) ? 12 : 8;
}
// PAIR (CTA pairs, tcgen05 .cta_group::2): one more warp copies each
// stage's scale chunks into both CTAs' tensor memory, so that the leader's
// MMA thread issues only MMAs.
template <int BN, int EPI, bool PAIR = false> constexpr int kThreads() {
  return 64 + 32 * kEpiWarps<BN, EPI>() + (EPI == EPI_DSWIGLU ? 32 : 0) + (PAIR ? 32 : 0);
}
constexpr int MAX_SORTED_G = 1024;  // wgrad schedules at most this many experts by size
constexpr int MAX_SPLIT = MAX_SPLIT_EXPERTS;  // wgrad: at most this many experts have their K range split

// Wgrad K-splitting of the largest experts (built per CTA in the prologue):
// ranks 0..n-1 (the largest experts) have parts[j] > 1 parts of at most
// split_chunks chunks each.  Their parts >= 1 come first in the tile order
// (xbase[j]: first such tile of rank j), then every expert's part 0 in rank
// order; sbase[j]: first partial slot of rank j (parts[j] slots per tile).
struct SplitInfo {
  int n;
  int extra_total;
  int xbase[MAX_SPLIT + 1];
  int parts[MAX_SPLIT];
  int sbase[MAX_SPLIT];
};

// F4: packed E2M1 operands on .kind::mxf4.  A stage's 128-byte rows then
// hold 256 K-elements, i.e. KC = 2 scale chunks per 128-row block.
// PK: the fused requant epilogues at BN = 256 (dense GELU / dGELU,
// dSwiGLU), which park three of each warp's four 32-column chunks in tensor
// memory past the scale slots so that the single accumulator is handed back
// at once; they take three stages for the room their larger scale-chunk and
// column-sum buffers (GELU / dGELU) or the z ring (dSwiGLU) need.
// PAIR: each CTA of a pair stages its own 128 rows of A and half (BN / 2
// rows) of the tile's B slice, so a stage is 33.5 KB and more of them fit.
template <int BN, bool ZR = false, bool F4 = false, bool PK = false, int EWARPS = 8, bool PAIR = false>
struct Cfg {
  static constexpr int EW = EWARPS;  // epilogue warps
  static constexpr int KC = F4 ? 2 : 1;
  static constexpr int STAGES = PAIR ? (PK ? 4 : 5) : (BN == 256 ? (PK ? 3 : 4) : (ZR ? 4 : 5));
  static constexpr int ACC = BN == 256 ? 1 : 2;
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * 128;
  static constexpr int SF_A_BYTES = KC * 512;  // A's chunks, then B's (chunk-major)
  static constexpr int SF_BYTES = KC * (512 + (BN / 128) * 512);
  static constexpr int SF_COLS = KC * (4 + 4 * (BN / 128));
  static constexpr uint32_t TX = A_BYTES + B_BYTES + SF_BYTES;
  // per-warp staging: a 32x32 BF16 / 32x16 fp32 block (2048 bytes) for the
  // plain epilogues, the [32][17] fp32 transpose for the requant ones;
  // 512-byte multiples (TMA store swizzle atoms).  F4 runs plain epilogues
  // only, and the room goes to a fourth 256-K stage.
  static constexpr int TB_BYTES = F4 ? 2048 : 2560;
  // scale chunks (BN/128 rowwise, BN/128 columnwise, 512 bytes each) and the
  // dense dGELU column-sum partials [4 lane quarters][BN] fp32
  static constexpr int CHUNK_BYTES = F4 ? 0 : ((PK && !ZR) ? 6144 : 4096);
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  // ZR: a ring of z slots, each [128 rows][Z_COLS cols] of gate and of up
  // (BF16): at BN = 128 two slots of 64 columns (128-byte swizzle), read by
  // all 8 epilogue warps; at BN = 256 three slots of 32 columns (64-byte
  // swizzle), each read by the 4 warps of one column half
  static constexpr int Z_COLS = BN == 256 ? 32 : 64;
  static constexpr int Z_SLOT = 2 * 128 * Z_COLS * 2;
  static constexpr int Z_SLOTS = ZR ? (BN == 256 ? 3 : 2) : 0;
  static constexpr int Z_READERS = BN == 256 ? 4 : 8;
  static constexpr int OFF_Z = (OFF_SF + STAGES * SF_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_TB = OFF_Z + Z_SLOTS * Z_SLOT;   // 8 x [32][17] fp32 transpose buffers
  static constexpr int OFF_CHUNK = OFF_TB + EW * TB_BYTES;   // scale chunks + column-sum partials
  static constexpr int OFF_BAR = OFF_CHUNK + CHUNK_BYTES;
  // wgrad with a workspace: tiles claimed from a global counter reach the
  // MMA thread and the epilogue through a TQN-entry queue
  static constexpr int TQN = 4;
  // PAIR adds peer_read, sf_ready[STAGES] and sf_final
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC + 2 + 2 * Z_SLOTS + 2 * TQN + (PAIR ? STAGES + 2 : 0);
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_TQ = OFF_MISC + 16;                 // TQN int32 tile indices
  static constexpr int OFF_ORDER = OFF_TQ + 4 * TQN;           // wgrad: experts by descending size
  static constexpr int OFF_SPLIT = OFF_ORDER + 2 * MAX_SORTED_G;  // wgrad: SplitInfo
  static constexpr int OFF_PREF = OFF_SPLIT + 256;             // PAIR: 256-row tiles before each expert
  static constexpr int SMEM_BYTES = OFF_PREF + (PAIR ? 4 * (MAX_PAIR_G + 1) : 0) + 1024;  // + alignment slack
  static_assert(MAX_PAIR_G == MAX_PAIR_G_HOST, "row-tile table size");
  static_assert(sizeof(SplitInfo) <= 256, "split info must fit");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SF_TMEM_BASE = 256;
  static constexpr uint32_t PARK_COL = 320;  // PK: 2 x 96 parked columns
  static_assert(ACC * BN <= 256, "accumulators live in tensor-memory columns 0..255");
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= (PK ? PARK_COL : TMEM_COLS), "scale slots must fit");
  static_assert(!PK || (BN == 256 && PARK_COL + 192 <= TMEM_COLS), "parked chunks must fit");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(OFF_TB % 1024 == 0, "staging buffers must be swizzle-atom aligned");
  static_assert(OFF_Z % 1024 == 0, "z slots must be swizzle-atom aligned");
};

// The configuration a kernel instantiation uses (launchers size shared
// memory with the same one).
template <int BN, int EPI> constexpr bool kParks() {
  return BN == 256 && (EPI == EPI_GELU || EPI == EPI_DGELU || EPI == EPI_DSWIGLU);
}
template <int BN, int EPI, bool F4 = false, bool PAIR = false>
using KCfg = Cfg<BN, EPI == EPI_DSWIGLU, F4, kParks<BN, EPI>(), kEpiWarps<BN, EPI>(), PAIR>;

struct Tile {
  int active;
  int g;
  int64_t m0, n0;
  int64_t kbeg;
  int nk;  // pipeline stages (K chunks of 128 elements, 256 with F4)
  int nc;  // K chunks of 128 elements
  int parts, part;  // wgrad K-split: parts of this (expert, m, n) tile and which one
  int64_t slot;     // first partial slot of the tile's parts
  int cnt;          // its arrival counter
  int upper;        // PAIR: the 256-row tile's upper 128 rows lie in its expert's segment
};

__device__ __forceinline__ int32_t ldg_i32(const int32_t* p) { return __ldg(p); }

// Tile t -> (expert, row base, column base, K range).  Grouped: tiles are
// row-block-major over all R rows; the expert is the segment holding the
// row base.  Wgrad: tiles are expert-major; K runs over the expert's rows.
// nk counts K chunks of 128 elements here.
template <int NT, int MODE, int MT = 128>
__device__ __forceinline__ Tile get_tile_chunks(const GemmParams& p, int64_t t, bool report, const uint16_t* order,
                                                const SplitInfo* split) {
  Tile T;
  T.active = 0; T.g = 0; T.m0 = 0; T.n0 = 0; T.kbeg = 0; T.nk = 0; T.nc = 0;
  T.parts = 1; T.part = 0; T.slot = 0; T.cnt = 0; T.upper = 1;
  if (MODE == MODE_GROUPED) {
    int64_t mt = t / p.n_tiles, nt = t % p.n_tiles;
    T.m0 = mt * 128;
    T.n0 = nt * NT;
    // no offsets: one dense segment of all R rows
    int64_t total = p.offsets ? ldg_i32(p.offsets + p.G - 1) : p.R;
    if (T.m0 >= total) return T;  // inactive tail
    int lo = 0, hi = p.G - 1;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if ((int64_t)ldg_i32(p.offsets + mid) > T.m0) hi = mid; else lo = mid + 1;
    }
    int64_t end = p.offsets ? ldg_i32(p.offsets + lo) : p.R;
    int64_t start = lo ? ldg_i32(p.offsets + lo - 1) : 0;
    bool bad = (start & 127) || (end & 127) || start > T.m0 || end <= T.m0 || end > p.R || total > p.R;
    if (bad) {
      if (report) atomicOr(&g_gemm_status, DEV_BAD_OFFSETS);
      return T;
    }
    T.g = lo;
    T.nk = (int)(p.K / 128);
    T.active = 1;
  } else {
    int64_t per_g = (int64_t)p.m_tiles * p.n_tiles;
    int64_t tt = t;
    int srank = -1;
    if (split != nullptr && split->n > 0) {
      if (t < split->extra_total) {  // part >= 1 of a split expert
        int j = 0;
        while (j + 1 < split->n && split->xbase[j + 1] <= t) j++;
        const int64_t local = t - split->xbase[j];
        T.part = 1 + (int)(local / per_g);
        tt = (int64_t)j * per_g + local % per_g;
        srank = j;
      } else {
        tt = t - split->extra_total;
        if (tt / per_g < split->n) srank = (int)(tt / per_g);
      }
    }
    // the tile count has headroom for split parts: past the last expert a
    // tile is inactive
    if (tt / per_g >= p.G) return T;
    T.g = (int)(tt / per_g);
    if (order) T.g = order[T.g];
    int64_t rem = tt % per_g;
    T.m0 = (rem / p.n_tiles) * MT;  // MT: 256-row tiles for CTA pairs
    T.n0 = (rem % p.n_tiles) * NT;
    int64_t end = p.offsets ? ldg_i32(p.offsets + T.g) : p.R;
    int64_t start = T.g ? ldg_i32(p.offsets + T.g - 1) : 0;
    bool bad = (start & 127) || (end & 127) || end < start || end > p.R || start < 0;
    if (bad && report) atomicOr(&g_gemm_status, DEV_BAD_OFFSETS);
    T.kbeg = bad ? 0 : start;
    T.nk = bad ? 0 : (int)((end - start) / 128);
    if (srank >= 0 && !bad) {  // this part's share of the chunks, balanced
      T.parts = split->parts[srank];
      const int lo = (int)((int64_t)T.nk * T.part / T.parts), hi = (int)((int64_t)T.nk * (T.part + 1) / T.parts);
      T.kbeg = start + 128ll * lo;
      T.nk = hi - lo;
      T.slot = (int64_t)split->sbase[srank] + rem * T.parts;
      T.cnt = (int)((int64_t)srank * per_g + rem);
    } else {
      T.part = 0;
    }
    T.active = 1;
  }
  return T;
}

// The same with nk in pipeline stages: with F4 a stage covers two chunks
// and a tile with an odd chunk count ends on a half stage.
template <int NT, int MODE, bool F4 = false, int MT = 128>
__device__ __forceinline__ Tile get_tile(const GemmParams& p, int64_t t, bool report, const uint16_t* order,
                                         const SplitInfo* split = nullptr) {
  Tile T = get_tile_chunks<NT, MODE, MT>(p, t, report, order, split);
  T.nc = T.nk;
  if (F4) T.nk = (T.nc + 1) >> 1;
  return T;
}

// get_tile, or with PAIR (grouped only) the 256-row tile of pair tile t:
// row tile t / n_tiles in expert order (the pref table), column tile
// t % n_tiles; m0 is the pair's row base (each CTA adds 128 x its rank).
template <int NT, int MODE, bool F4, bool PAIR>
__device__ __forceinline__ Tile get_tile_x(const GemmParams& p, int64_t t, bool report, const uint16_t* order,
                                           const SplitInfo* split, const int32_t* pref) {
  if constexpr (!PAIR) {
    return get_tile<NT, MODE, F4>(p, t, report, order, split);
  } else if constexpr (MODE == MODE_WGRAD) {
    // wgrad: the weight rows in 256-row tiles (p.m_tiles of them), the rest
    // as for one SM per tile
    return get_tile<NT, MODE, F4, 256>(p, t, report, order, split);
  } else {
    Tile T;
    T.active = 0; T.g = 0; T.m0 = 0; T.n0 = (t % p.n_tiles) * NT; T.kbeg = 0; T.nk = 0; T.nc = 0;
    T.parts = 1; T.part = 0; T.slot = 0; T.cnt = 0; T.upper = 0;
    if (pair_row_tile(p.offsets, p.G, p.R, pref, t / p.n_tiles, &T.g, &T.m0, &T.upper)) {
      T.nk = (int)(p.K / 128);
      T.nc = T.nk;
      T.active = 1;
    }
    return T;
  }
}

// The global tile a CTA handles at its i-th turn.  Grouped: plain round
// robin (neighbouring CTAs share A rows and B panels in L2).  Wgrad: tiles
// are laid out expert by expert in descending size order and dealt to the
// CTAs boustrophedon-wise (forward on even turns, backward on odd), which
// spreads the long reductions of the largest experts across the grid.
template <int MODE>
__device__ __forceinline__ int64_t tile_index(int64_t i) {
  if (MODE == MODE_WGRAD && (i & 1)) return i * gridDim.x + (gridDim.x - 1 - blockIdx.x);
  return i * gridDim.x + blockIdx.x;
}

// With PAIR both CTAs of a cluster take the same tiles: pair p = blockIdx / 2
// of gridDim / 2 takes tiles p, p + gridDim / 2, ...
template <bool PAIR>
__device__ __forceinline__ int64_t tile_slots() { return PAIR ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x; }

template <int MODE, bool PAIR>
__device__ __forceinline__ int64_t tile_index_x(int64_t i) {
  if constexpr (PAIR) {
    const int64_t np = gridDim.x >> 1, pi = blockIdx.x >> 1;
    if (MODE == MODE_WGRAD && (i & 1)) return i * np + (np - 1 - pi);  // boustrophedon, as for one SM
    return i * np + pi;
  }
  return tile_index<MODE>(i);
}


__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(ptr));
}

// ---- epilogue helpers --------------------------------------------------

// sigmoid as 1 / (1 + exp(-x)) with the fast exponential and divide
// intrinsics (exactly 1.0 once exp(-x) vanishes against 1, 0 once it
// overflows).
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Convert 32 fp32 values (this lane's row) to BF16 into the warp's staging
// buffer (row = lane, 64 bytes, 64-byte swizzle) and store the warp's 32x32
// block with one TMA store.  The caller has made sure the buffer's previous
// store has been read (bulk_wait_read by lane 0, then __syncwarp).
__device__ __forceinline__ void store_bf16_block(const float* v, uint8_t* stage, int lane, const CUtensorMap* tm,
                                                 int64_t col0, int64_t row0) {
  uint4* row = reinterpret_cast<uint4*>(stage + lane * 64);
#pragma unroll
  for (int c = 0; c < 4; c++)
    row[c ^ ((lane >> 1) & 3)] = make_uint4(float2_to_bf16x2(v[8 * c], v[8 * c + 1]), float2_to_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                            float2_to_bf16x2(v[8 * c + 4], v[8 * c + 5]), float2_to_bf16x2(v[8 * c + 6], v[8 * c + 7]));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm, stage, (int)col0, (int)row0);
    bulk_commit();
  }
}

// Test instrument: this lane's 32 fp32 pre-quantization values of one row
// (columns col0..col0+31) into the tap [rows, ld] when one is attached.
__device__ __forceinline__ void tap_store32(float* tap, int64_t ld, int64_t row, int64_t col0, const float* v) {
  float4* d = reinterpret_cast<float4*>(tap + row * ld + col0);
#pragma unroll
  for (int i = 0; i < 8; i++) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// fp32 variant: 16 values of this lane's row into the staging buffer (64
// bytes per row, 64-byte swizzle), then one TMA store (or reduce-add into
// what the destination holds) of the warp's 32x16 block.
__device__ __forceinline__ void store_f32_block(const float* v, uint8_t* stage, int lane, const CUtensorMap* tm,
                                                int64_t col0, int64_t row0, bool add) {
  uint4* row = reinterpret_cast<uint4*>(stage + lane * 64);
#pragma unroll
  for (int c = 0; c < 4; c++)
    row[c ^ ((lane >> 1) & 3)] = make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                            __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (add) tma_reduce_add_2d(tm, stage, (int)col0, (int)row0);
    else tma_store_2d(tm, stage, (int)col0, (int)row0);
    bulk_commit();
  }
}

// Before a warp rewrites its staging buffer: the previous TMA store has read it.
__device__ __forceinline__ void stage_reuse_wait(int lane) {
  if (lane == 0) bulk_wait_read();
  __syncwarp();
}

// Rowwise E4M3 requant of 32 fp32 values held by one thread.
__device__ __forceinline__ uint32_t row_quant_store_e4m3(float (&v)[32], uint8_t* dst) {
  uint32_t sb = rceil_scale_byte_sel<E4M3>(amax_abs_bits<32>(v));
  uint32_t w[8];
  quantize_block_words<E4M3>(v, sb, w);
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return sb;
}

__device__ __forceinline__ void store_chunk(uint8_t* dst, const uint8_t* chunk, int lane) {
  reinterpret_cast<uint4*>(dst)[lane] = reinterpret_cast<const uint4*>(chunk)[lane];
}

// Generic requant helpers (element format QF, optional 32-point rotation).

// tanh-GELU and its derivative in fp32 (Primus PR #1064 "feat(mxfp6): MXFP6
// (E2M3) Flux linears, a fused MLP, and the MLPerf recipe": the fused MLP's
// tanh GELU epilogue and its derivative as the backward prologue).
// With u = sqrt(2/pi) (x + 0.044715 x^3), 0.5 (1 + tanh(u)) = sigma(2u), the
// logistic function, so gelu(x) = x sigma(2u): one exponential and one
// reciprocal, and no cancellation in 1 + tanh(u) for negative x.  The
// derivative is s + x s (1 - s) d(2u)/dx with s = sigma(2u), 1 - s taken as
// E s (E = exp(-2u)) where s >= 1/2 and as 1 - s below.  The polynomial is
// evaluated at x clamped to [-100, 100], where the logistic has saturated to
// 0 or 1 in fp32 anyway, so x^3 cannot overflow.
__device__ __forceinline__ float gelu_2u_(float x) {
  const float c1 = 1.5957691216057308f;   // 2 sqrt(2/pi)
  const float c3 = 0.0713548162726009f;   // 2 sqrt(2/pi) 0.044715
  const float xc = fminf(fmaxf(x, -100.0f), 100.0f);
  return xc * fmaf(c3, xc * xc, c1);
}
__device__ __forceinline__ float gelu_tanh_f(float x) { return x * sigmoidf_(gelu_2u_(x)); }
__device__ __forceinline__ float dgelu_tanh_f(float x) {
  const float c1 = 1.5957691216057308f;
  const float c3x3 = 0.2140644488178027f;  // 3 * 2 sqrt(2/pi) 0.044715
  const float v = gelu_2u_(x);
  const float e = __expf(-v);
  const float s = __fdividef(1.0f, 1.0f + e);
  const float oms = v < 0.0f ? 1.0f - s : e * s;
  const float xc = fminf(fmaxf(x, -100.0f), 100.0f);
  return fmaf(x * s * oms, fmaf(c3x3, xc * xc, c1), s);
}

// Rowwise requant of 32 fp32 values held by one thread (rotated first if QH).
template <int QF, bool QH>
__device__ __forceinline__ uint32_t row_quant_store(float (&v)[32], uint8_t* dst) {
  if constexpr (QH) hadamard32(v);
  const uint32_t sb = rceil_scale_byte_sel<QF>(amax_abs_bits<32>(v));
  uint32_t w[8];
  quantize_block_words<QF>(v, sb, w);
  if constexpr (QF == E4M3) {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else if constexpr (QF == E2M1) {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    reinterpret_cast<uint2*>(dst)[0] = make_uint2(w[0], w[1]);
    reinterpret_cast<uint2*>(dst)[1] = make_uint2(w[2], w[3]);
    reinterpret_cast<uint2*>(dst)[2] = make_uint2(w[4], w[5]);
  }
  return sb;
}

// Columnwise requant of 16 columns whose 32-row blocks are spread over the
// warp (lane = row; v = this lane's values of the 16 columns).  The warp
// transposes them through a padded [32][17] fp32 buffer; lane pair (2c, 2c+1)
// then owns column c, rows 0..15 and 16..31: optional rotation (stages 1..8
// inside each lane, stage 16 across the pair), amax over the pair, scale,
// and 16 packed codes per lane stored straight to the transposed payload.
// dst(c) is the payload row of column c at this warp's 32-row block;
// returns nothing, writes column c's scale byte to chunk[(f&31)*16+(f>>5)*4+q]
// for f = f_local0 + c.  colsum (optional): column c's sum over the warp's 32
// rows before any rotation (rows 0..15 and 16..31 each summed in order, then
// the two halves), written to colsum[c] by the lane pair's first lane.
template <int QF, bool QH>
__device__ __forceinline__ void col_quant16(const float* v, float* buf, int lane, uint8_t* q_col, int64_t col_ld,
                                            int64_t col0, int64_t row_byte0, uint8_t* chunk, int f_local0, int q,
                                            float* colsum = nullptr) {
#pragma unroll
  for (int c = 0; c < 16; c++) buf[lane * 17 + c] = v[c];
  __syncwarp();
  const int c = lane >> 1, hh = lane & 1;
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = buf[(hh * 16 + i) * 17 + c];
  __syncwarp();
  if (colsum != nullptr) {
    float sum = x[0];
#pragma unroll
    for (int i = 1; i < 16; i++) sum += x[i];
    const float other = __shfl_xor_sync(0xffffffffu, sum, 1);
    if (hh == 0) colsum[c] = sum + other;
  }
  if constexpr (QH) {
    butterfly_stages<16>(x);
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], 1);
      x[i] = hh ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
    }
    scale_values<16>(x, __uint_as_float(0x3E3504F3u));
  }
  uint32_t amax = amax_abs_bits<16>(x);
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const uint32_t sb = rceil_scale_byte_sel<QF>(amax);
  uint8_t* dst = q_col + (col0 + c) * col_ld + row_byte0 + hh * (BlockBytes<QF>::value / 2);
  if (sb == 0xFFu) {
    const uint32_t nw = nan_block_word<QF>();
    if constexpr (QF == E4M3) reinterpret_cast<uint4*>(dst)[0] = make_uint4(nw, nw, nw, nw);
    else if constexpr (QF == E2M1) reinterpret_cast<uint2*>(dst)[0] = make_uint2(nw, nw);
    else { uint32_t* d = reinterpret_cast<uint32_t*>(dst); d[0] = nw; d[1] = nw; d[2] = nw; }
  } else {
    scale_values<16>(x, inv_scale_from_byte(sb));
    if constexpr (QF == E4M3) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; i++)
        w[i] = cvt_e4m3x2(x[4 * i], x[4 * i + 1]) | (cvt_e4m3x2(x[4 * i + 2], x[4 * i + 3]) << 16);
      reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (QF == E2M1) {
      uint32_t w[2];
#pragma unroll
      for (int i = 0; i < 2; i++)
        w[i] = cvt_e2m1x2(x[8 * i], x[8 * i + 1]) | (cvt_e2m1x2(x[8 * i + 2], x[8 * i + 3]) << 8) |
               (cvt_e2m1x2(x[8 * i + 4], x[8 * i + 5]) << 16) | (cvt_e2m1x2(x[8 * i + 6], x[8 * i + 7]) << 24);
      reinterpret_cast<uint2*>(dst)[0] = make_uint2(w[0], w[1]);
    } else {
      uint32_t g[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const uint32_t p0 = cvt_e2m3x2(x[4 * i], x[4 * i + 1]), p1 = cvt_e2m3x2(x[4 * i + 2], x[4 * i + 3]);
        g[i] = (p0 & 0x3Fu) | (((p0 >> 8) & 0x3Fu) << 6) | ((p1 & 0x3Fu) << 12) | (((p1 >> 8) & 0x3Fu) << 18);
      }
      uint32_t* d = reinterpret_cast<uint32_t*>(dst);
      d[0] = g[0] | (g[1] << 24);
      d[1] = (g[1] >> 8) | (g[2] << 16);
      d[2] = (g[2] >> 16) | (g[3] << 8);
    }
  }
  if (hh == 0) {
    const int f = f_local0 + c;
    chunk[(f & 31) * 16 + (f >> 5) * 4 + q] = (uint8_t)sb;
  }
}

// ---- the kernel ---------------------------------------------------------

// EXT: the dSwiGLU kernel has a separate instantiation with its optional
// extras, the debug tap and the routing probabilities (its register budget is
// tight); the other fused epilogues test those pointers at run time.
template <int BN, int EPI, int MODE, int QF = E4M3, bool QH = false, bool EXT = false, bool F4 = false,
          bool PAIR = false>
__global__ void __launch_bounds__(kThreads<BN, EPI, PAIR>(), 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmSA,
               const __grid_constant__ CUtensorMap tmSB, const GemmParams p) {
  constexpr bool ZR = EPI == EPI_DSWIGLU;  // z streamed by TMA (tmO maps the BF16 z [R, 2F])
  constexpr bool EXT_ON = EPI != EPI_DSWIGLU || EXT;
  static_assert(!F4 || (EPI == EPI_BF16 || EPI == EPI_F32), "mxf4 operands: plain epilogues only");
  using C = KCfg<BN, EPI, F4, PAIR>;
  constexpr bool PK = kParks<BN, EPI>();
  // PAIR: clusters of two CTAs on 256-row tiles (grouped, BN = 256, FP8/FP6
  // operands); tmSA / tmSB map the operands' blocked scales for the 2-SM loads
  static_assert(!PAIR || (BN == 256 && !F4), "CTA pairs: 256-column tiles of FP8 / FP6 operands");
  constexpr int NT = (EPI == EPI_SWIGLU) ? 128 : BN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sSF = smem + C::OFF_SF;
  uint8_t* sTB = smem + C::OFF_TB;
  uint8_t* sChunk = smem + C::OFF_CHUNK;
  uint8_t* sZ = smem + C::OFF_Z;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + C::ACC;
  uint64_t* final_bar = acc_empty + C::ACC;
  uint64_t* epi_bar = final_bar + 1;  // the epilogue warps' own barrier
  uint64_t* z_full = epi_bar + 1;     // ZR: slot loaded
  uint64_t* z_empty = z_full + C::Z_SLOTS;  // ZR: slot read by its Z_READERS epilogue warps
  uint64_t* tq_full = z_empty + C::Z_SLOTS;   // dynamic wgrad schedule: queue entry written
  uint64_t* tq_empty = tq_full + C::TQN;      // ... and read by the MMA thread and every epilogue warp
  uint64_t* peer_read = tq_empty + C::TQN;    // PAIR, peer: its epilogue warps have read the accumulator
  uint64_t* sf_ready = peer_read + 1;         // PAIR, leader: the stage's scales are in tensor memory
  uint64_t* sf_final = sf_ready + C::STAGES;  // PAIR, leader: every scale copy has completed
  int32_t* pref = reinterpret_cast<int32_t*>(smem + C::OFF_PREF);  // PAIR: 256-row tiles before each expert
  volatile int32_t* tq = reinterpret_cast<volatile int32_t*>(smem + C::OFF_TQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;  // PAIR: 0 = leader (issues the MMAs), 1 = peer
  const bool leader = rank == 0;
  // wgrad with a workspace: each CTA's producer claims the next tile (in the
  // order of get_tile: split parts, then experts by descending size) from a
  // counter the host zeroes, so tiles go to whichever CTA is free first
  const bool dyn = MODE == MODE_WGRAD && p.dyn_ctr != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    // PAIR: the leader's accumulator is handed back by its own epilogue
    // warps plus one arrival from the peer
    for (int a = 0; a < C::ACC; a++) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], C::EW + (PAIR ? 1 : 0)); }
    if (PAIR) {
      mbar_init(peer_read, C::EW);
      for (int s = 0; s < C::STAGES; s++) mbar_init(&sf_ready[s], 1);
      mbar_init(sf_final, 1);
    }
    mbar_init(final_bar, 1);
    mbar_init(epi_bar, C::EW);
    for (int z = 0; z < C::Z_SLOTS; z++) { mbar_init(&z_full[z], 1); mbar_init(&z_empty[z], C::Z_READERS); }
    // tile queue: read by the MMA thread and every epilogue warp; with PAIR
    // the leader's entries are also read by its scale-copy warp and by the
    // peer's producer and epilogue warps, which arrive across the pair
    for (int e = 0; e < C::TQN; e++) {
      mbar_init(&tq_full[e], 1);
      mbar_init(&tq_empty[e], PAIR ? 3 + 2 * C::EW : 1 + C::EW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA); prefetch_tensormap(&tmB); prefetch_tensormap(&tmO);
    if (PAIR) { prefetch_tensormap(&tmSA); prefetch_tensormap(&tmSB); }
  }
  if constexpr (PAIR) {
    // tensor memory allocated by both CTAs of the pair at once (each gets the
    // same columns); the row-tile table built before the pair meets
    if (warp == 1) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                   :: "r"(smem_u32(tmem_slot)), "n"(C::TMEM_COLS) : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    if (warp == 0) build_pair_prefix(p.offsets, p.G, p.R, pref, lane, leader ? &g_gemm_status : nullptr);
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised before any remote arrival or 2-SM copy
    tc_fence_after();
  } else {
    if (warp == 1) tmem_alloc<C::TMEM_COLS>(tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  const uint32_t tmem_base = *tmem_slot;
  // wgrad: rank the experts by descending row count (ties by index)
  const uint16_t* order = nullptr;
  const SplitInfo* split = nullptr;
  if (MODE == MODE_WGRAD && p.offsets != nullptr && p.G <= MAX_SORTED_G && p.G > 1) {
    uint16_t* s_order = reinterpret_cast<uint16_t*>(smem + C::OFF_ORDER);
    auto count = [&](int g) -> int64_t {
      const int64_t e = ldg_i32(p.offsets + g), b = g ? ldg_i32(p.offsets + g - 1) : 0;
      return e - b;
    };
    for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
      const int64_t cg = count(g);
      int rank = 0;
      for (int h = 0; h < p.G; h++) {
        const int64_t ch = count(h);
        rank += (ch > cg || (ch == cg && h < g)) ? 1 : 0;
      }
      s_order[rank] = (uint16_t)g;
    }
    __syncthreads();
    order = s_order;
    if (p.split_chunks > 0) {
      // the largest experts (ranks 0..) with more than split_min chunks get
      // ceil(chunks / split_chunks) parts, while the partial slots and
      // counters the host provided last
      SplitInfo* si = reinterpret_cast<SplitInfo*>(smem + C::OFF_SPLIT);
      if (threadIdx.x == 0) {
        const int64_t per_g = (int64_t)p.m_tiles * p.n_tiles;
        int n = 0;
        int64_t x = 0, sb = 0;
        for (int j = 0; j < p.G && n < MAX_SPLIT; j++) {
          const int g = s_order[j];
          const int64_t e = ldg_i32(p.offsets + g), b = g ? ldg_i32(p.offsets + g - 1) : 0;
          const bool ok = e >= b && ((b | e) & 127) == 0 && e <= p.R;
          const int64_t nk = ok ? (e - b) / 128 : 0;
          if (nk <= p.split_min || nk <= p.split_chunks) break;
          const int parts = (int)((nk + p.split_chunks - 1) / p.split_chunks);
          // PAIR: every pair-tile slot is two 128-row slots
          if ((PAIR ? 2 : 1) * (sb + parts * per_g) > p.split_slots || x + (parts - 1) * per_g > p.split_extra) break;
          si->parts[n] = parts;
          si->xbase[n] = (int)x;
          si->sbase[n] = (int)sb;
          x += (parts - 1) * per_g;
          sb += parts * per_g;
          n++;
        }
        si->xbase[n] = (int)x;
        si->n = n;
        si->extra_total = (int)x;
      }
      __syncthreads();
      split = si;
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // A panels are read by the neighbouring CTAs that take the same row
      // block's other column tiles: normal eviction priority for the grouped
      // GEMMs (FC1 + SwiGLU, FC2, FC1 dgrad 1 % faster than evict-first), but
      // evict-first where the kernel streams more data past them (dSwiGLU's
      // z, 3 % slower with normal priority) or reads them once (wgrad); B
      // slices, reused by every row block of an expert, are kept longer
      const uint64_t pol_a = (EPI == EPI_DSWIGLU || MODE == MODE_WGRAD) ? l2_policy_evict_first()
                                                                        : l2_policy_evict_normal();
      const uint64_t pol_b = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int armed_parity[C::STAGES];
      for (int s = 0; s < C::STAGES; s++) armed_parity[s] = -1;
      bool ok = true;
      int qi = 0;
      uint32_t qph = 0;
      int32_t next = (dyn && leader) ? atomicAdd(p.dyn_ctr, 1) : 0;
      for (int64_t i = 0; ok; i++) {
        int64_t t;
        if (dyn && PAIR && !leader) {  // the peer takes the tiles its leader claimed
          if (!mbar_wait_cluster(&tq_full[qi], qph, abort_flag)) { ok = false; break; }
          t = tq[qi];
          arrive_on_leader(leader_addr(&tq_empty[qi]));
          if (++qi == C::TQN) { qi = 0; qph ^= 1u; }
          if (t < 0) break;
        } else if (dyn) {  // claim one tile ahead, queue this one for the MMA thread and the epilogue
          t = next;
          const bool end = t >= p.num_tiles;
          if (!end) next = atomicAdd(p.dyn_ctr, 1);
          if (!(PAIR ? mbar_wait_cluster(&tq_empty[qi], qph ^ 1u, abort_flag)
                     : mbar_wait_bounded(&tq_empty[qi], qph ^ 1u, abort_flag, WAIT_BUDGET_NS))) {
            ok = false;
            break;
          }
          const int32_t v = end ? -1 : (int32_t)t;
          tq[qi] = v;
          mbar_arrive(&tq_full[qi]);
          if (PAIR) {  // the same entry in the peer's queue
            st_cluster_u32(peer_addr((const void*)&tq[qi]), (uint32_t)v);
            arrive_on_leader(peer_addr(&tq_full[qi]));
          }
          if (++qi == C::TQN) { qi = 0; qph ^= 1u; }
          if (end) break;
        } else {
          if (i * tile_slots<PAIR>() >= p.num_tiles) break;
          t = tile_index_x<MODE, PAIR>(i);
          if (t >= p.num_tiles) continue;
        }
        Tile T = get_tile_x<NT, MODE, F4, PAIR>(p, t, false, order, split, pref);
        if (!T.active || T.nk == 0) continue;
        if (PAIR) T.m0 += 128 * rank;  // this CTA's 128 rows of the pair's 256
        int64_t brow[2];
        if (EPI == EPI_SWIGLU) {
          brow[0] = (int64_t)T.g * 2 * p.F + T.n0;
          brow[1] = brow[0] + p.F;
        } else if (MODE == MODE_GROUPED) {
          brow[0] = (int64_t)T.g * p.Nb + T.n0;
          brow[1] = brow[0] + 128;
        } else {
          brow[0] = T.n0;
          brow[1] = T.n0 + 128;
        }
        for (int kb = 0; kb < T.nk; kb++) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          // F4: the stage's first 128-element chunk and how many it holds
          // (the second half of a tile's last stage may lie past its K range;
          // its payload is loaded but no MMA reads it, and its scales are not
          // loaded)
          const int nch = F4 ? ((2 * kb + 1 < T.nc) ? 2 : 1) : 1;
          const int64_t kc = T.kbeg / 128 + (F4 ? 2 * kb : kb);
          const uint32_t tx = F4 ? (uint32_t)(C::A_BYTES + C::B_BYTES + nch * (512 + (BN / 128) * 512))
                                 : p.tx_bytes;
          // x coordinate: elements, or bytes of the packed payload with F4
          const int kx = (int)(F4 ? kc * 64 : kc * 128);
          if constexpr (PAIR) {
            // 2-SM loads: each CTA its 128 rows of A, its 128-row block of
            // the tile's B slice and every scale chunk its tensor memory
            // needs (its A rows', both B blocks'), all counted on the
            // leader's barrier, which expects both CTAs' bytes
            const uint32_t fb = leader_addr(&full[stage]);
            if (leader) {
              mbar_arrive_expect_tx(&full[stage], 2u * tx);
              armed_parity[stage] = (int)phase;
            }
            tma2_load_2d(sA + stage * C::A_BYTES, &tmA, kx, (int)T.m0, fb, pol_a);
            tma2_load_2d(sB + stage * C::B_BYTES, &tmB, kx, (int)brow[rank], fb, pol_b);
            uint8_t* sf = sSF + stage * C::SF_BYTES;
            tma2_load_3d(sf, &tmSA, 0, (int)kc, (int)(T.m0 >> 7), fb);
            tma2_load_3d(sf + 512, &tmSB, 0, (int)kc, (int)(brow[0] >> 7), fb);
            tma2_load_3d(sf + 1024, &tmSB, 0, (int)kc, (int)(brow[1] >> 7), fb);
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            continue;
          }
          mbar_arrive_expect_tx(&full[stage], tx);
          armed_parity[stage] = (int)phase;
          tma_load_2d(sA + stage * C::A_BYTES, &tmA, kx, (int)T.m0, &full[stage], pol_a);
#pragma unroll
          for (int i = 0; i < BN / 128; i++)
            tma_load_2d(sB + stage * C::B_BYTES + i * 16384, &tmB, kx, (int)brow[i], &full[stage], pol_b);
          uint8_t* sf = sSF + stage * C::SF_BYTES;
#pragma unroll
          for (int c = 0; c < C::KC; c++) {
            if (c < nch) {
              bulk_load(sf + c * 512, p.sfa + ((T.m0 >> 7) * p.sfa_kchunks + kc + c) * 512, 512, &full[stage]);
#pragma unroll
              for (int i = 0; i < BN / 128; i++)
                bulk_load(sf + C::SF_A_BYTES + (c * (BN / 128) + i) * 512,
                          p.sfb + ((brow[i] >> 7) * p.sfb_kchunks + kc + c) * 512, 512, &full[stage]);
            }
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Every copy this thread issued must have landed before the CTA exits
      // (also after an abort: the drain ignores the abort flag, not the clock).
      volatile int no_abort = 0;
      for (int s = 0; s < C::STAGES; s++)
        if (armed_parity[s] >= 0) mbar_wait_bounded(&full[s], (uint32_t)armed_parity[s], &no_abort, WAIT_BUDGET_NS);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (PAIR: the leader's, for both CTAs, M = 256)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int qi = 0;
      uint32_t qph = 0;
      for (int64_t i = 0; ok; i++) {
        int64_t t;
        if (dyn) {
          if (!mbar_wait_bounded(&tq_full[qi], qph, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          t = tq[qi];
          mbar_arrive(&tq_empty[qi]);
          if (++qi == C::TQN) { qi = 0; qph ^= 1u; }
          if (t < 0) break;
        } else {
          if (i * tile_slots<PAIR>() >= p.num_tiles) break;
          t = tile_index_x<MODE, PAIR>(i);
          if (t >= p.num_tiles) continue;
        }
        Tile T = get_tile_x<NT, MODE, F4, PAIR>(p, t, false, order, split, pref);
        if (!T.active || T.nk == 0) continue;
        // PAIR: the peer's hand-back arrives across the cluster (acquire at cluster scope)
        if (!(PAIR ? mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1u, abort_flag)
                   : mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag, WAIT_BUDGET_NS))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < T.nk; kb++) {
          // PAIR: the scale warp has seen the stage's bytes land and copied its scales
          if (!mbar_wait_bounded(PAIR ? &sf_ready[stage] : &full[stage], phase, abort_flag, WAIT_BUDGET_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if constexpr (PAIR) {
            const uint32_t sf_t = tmem_base + C::SF_TMEM_BASE + (uint32_t)(stage * C::SF_COLS);
            const uint64_t ad = smem_desc(smem_u32(sA + stage * C::A_BYTES), 16, 1024, 2);
            const uint64_t bd = smem_desc(smem_u32(sB + stage * C::B_BYTES), 16, 1024, 2);
            const uint32_t idesc0 = mma_idesc_mx((uint32_t)p.a_type, (uint32_t)p.b_type, 256, BN, 0, 0);
#pragma unroll
            for (int j = 0; j < 4; j++)
              tc2_mma_mx(d_tmem, ad + 2 * j, bd + 2 * j, idesc0 | ((uint32_t)j << 4) | ((uint32_t)j << 29), sf_t,
                         sf_t + 4, (kb | j) != 0 ? 1u : 0u);
            tc2_commit_both(&empty[stage]);
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            continue;
          }
          const uint32_t sf_t = tmem_base + C::SF_TMEM_BASE + (uint32_t)(stage * C::SF_COLS);
          const uint32_t sf_s = smem_u32(sSF + stage * C::SF_BYTES);
          const uint32_t a_s = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_s = smem_u32(sB + stage * C::B_BYTES);
          if constexpr (F4) {
            // tensor-memory scale columns: A's chunk c at 4c, B's chunk c
            // (BN/128 row blocks) at 8 + 4c(BN/128)
            const int nch = (2 * kb + 1 < T.nc) ? 2 : 1;
#pragma unroll
            for (int c = 0; c < 2; c++) {
              if (c < nch) {
                tc_copy_scales(sf_t + 4 * c, sf_s + 512 * c);
#pragma unroll
                for (int i = 0; i < BN / 128; i++)
                  tc_copy_scales(sf_t + 8 + 4 * (c * (BN / 128) + i), sf_s + C::SF_A_BYTES + 512 * (c * (BN / 128) + i));
              }
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
              if (j < 2 * nch) {
                const uint64_t adesc = smem_desc(a_s + 32 * j, 16, 1024, 2);
                const uint64_t bdesc = smem_desc(b_s + 32 * j, 16, 1024, 2);
                const uint32_t sid = (uint32_t)(j & 1) * 2u;
                const uint32_t idesc = mma_idesc_mx(MXF4_E2M1, MXF4_E2M1, 128, BN, sid, sid);
                tc_mma_mxf4(d_tmem, adesc, bdesc, idesc, sf_t + 4 * (j >> 1), sf_t + 8 + 4 * (j >> 1) * (BN / 128),
                            (kb | j) != 0 ? 1u : 0u);
              }
            }
          } else {
            tc_copy_scales(sf_t, sf_s);
#pragma unroll
            for (int i = 0; i < BN / 128; i++) tc_copy_scales(sf_t + 4 + 4 * i, sf_s + 512 + 512 * i);
#pragma unroll
            for (int j = 0; j < 4; j++) {
              const uint64_t adesc = smem_desc(a_s + 32 * j, 16, 1024, 2);
              const uint64_t bdesc = smem_desc(b_s + 32 * j, 16, 1024, 2);
              const uint32_t idesc = mma_idesc_mx((uint32_t)p.a_type, (uint32_t)p.b_type, 128, BN, j, j);
              tc_mma_mx(d_tmem, adesc, bdesc, idesc, sf_t, sf_t + 4, (kb | j) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (PAIR) tc2_commit_both(&acc_full[acc]);
        else tc_commit(&acc_full[acc]);
        if (++acc == C::ACC) { acc = 0; acc_phase ^= 1u; }
      }
      if (PAIR && !ok) *abort_flag = 1;
      // No MMA may still be writing tensor memory when it is freed.
      volatile int no_abort = 0;
      if (PAIR) tc2_commit_local(final_bar);
      else tc_commit(final_bar);
      mbar_wait_bounded(final_bar, 0, &no_abort, WAIT_BUDGET_NS);
    }
  } else if (PAIR && warp == kThreads<BN, EPI, PAIR>() / 32 - 1) {
    // ------------------------------------------------------------ scale copies (PAIR, leader)
    // In the MMA thread's stage order: wait for the stage's bytes (both
    // CTAs'), copy its three scale chunks into both CTAs' tensor memory
    // (tcgen05.cp .cta_group::2) and signal sf_ready once they completed.  A
    // slot is rewritten only after the producers refilled its stage, i.e.
    // after the MMAs that read it.
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int qi = 0;
      uint32_t qph = 0;
      for (int64_t i = 0; ok; i++) {
        int64_t t;
        if (dyn) {  // the claimed tiles, in queue order
          if (!mbar_wait_bounded(&tq_full[qi], qph, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          t = tq[qi];
          mbar_arrive(&tq_empty[qi]);
          if (++qi == C::TQN) { qi = 0; qph ^= 1u; }
          if (t < 0) break;
        } else {
          if (i * tile_slots<PAIR>() >= p.num_tiles) break;
          t = tile_index_x<MODE, PAIR>(i);
          if (t >= p.num_tiles) continue;
        }
        const Tile T = get_tile_x<NT, MODE, F4, PAIR>(p, t, false, order, split, pref);
        if (!T.active || T.nk == 0) continue;
        for (int kb = 0; kb < T.nk; kb++) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + C::SF_TMEM_BASE + (uint32_t)(stage * C::SF_COLS);
          const uint64_t sd = smem_desc(smem_u32(sSF + stage * C::SF_BYTES), 0, 128, 0);
          tc2_copy_scales(sf_t, sd);                    // A's 128 rows (each CTA its own)
          tc2_copy_scales(sf_t + 4, sd + (512 >> 4));   // B block 0
          tc2_copy_scales(sf_t + 8, sd + (1024 >> 4));  // B block 1
          tc2_commit_local(&sf_ready[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) *abort_flag = 1;
      // No copy may still be writing either CTA's tensor memory when it is freed.
      volatile int no_abort = 0;
      tc2_commit_local(sf_final);
      mbar_wait_bounded(sf_final, 0, &no_abort, WAIT_BUDGET_NS);
    }
  } else if (ZR && warp == 2 + C::EW) {
    // ------------------------------------------------------------ z loader (ZR)
    // Streams the tile's saved pre-activation, Z_COLS columns (gate and up
    // boxes) per slot, in the epilogue's tile order.
    if (ZR && lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int zs = 0;
      uint32_t zph = 0;
      int armed_parity[C::Z_SLOTS > 0 ? C::Z_SLOTS : 1];
      for (int z = 0; z < C::Z_SLOTS; z++) armed_parity[z] = -1;
      bool ok = true;
      for (int64_t i = 0; i * tile_slots<PAIR>() < p.num_tiles && ok; i++) {
        const int64_t t = tile_index_x<MODE, PAIR>(i);
        if (t >= p.num_tiles) continue;
        Tile T = get_tile_x<NT, MODE, F4, PAIR>(p, t, false, order, split, pref);
        if (!T.active || T.nk == 0) continue;
        if (PAIR && rank && !T.upper) continue;  // the epilogue skips a half past its segment
        if (PAIR) T.m0 += 128 * rank;
        for (int hh = 0; hh < BN / C::Z_COLS; hh++) {
          if (!mbar_wait_bounded(&z_empty[zs], zph ^ 1u, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          mbar_arrive_expect_tx(&z_full[zs], (uint32_t)C::Z_SLOT);
          armed_parity[zs] = (int)zph;
          uint8_t* dst = sZ + zs * C::Z_SLOT;
          tma_load_2d(dst, &tmO, (int)(T.n0 + hh * C::Z_COLS), (int)T.m0, &z_full[zs], pol);
          tma_load_2d(dst + C::Z_SLOT / 2, &tmO, (int)(p.F + T.n0 + hh * C::Z_COLS), (int)T.m0, &z_full[zs], pol);
          if (++zs == C::Z_SLOTS) { zs = 0; zph ^= 1u; }
        }
      }
      volatile int no_abort = 0;
      for (int z = 0; z < C::Z_SLOTS; z++)
        if (armed_parity[z] >= 0) mbar_wait_bounded(&z_full[z], (uint32_t)armed_parity[z], &no_abort, WAIT_BUDGET_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;       // 0..EW-1
    const int q = warp & 3;        // tensor-memory lane quarter
    const int half = ew >> 2;      // column half
    float* tb = reinterpret_cast<float*>(sTB + ew * C::TB_BYTES);
    uint8_t* tb_bytes = sTB + ew * C::TB_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t epi_phase = 0;
    int zslot = 0;           // ZR: next z slot and its phase
    uint32_t zphase = 0;
    uint32_t zt = 0;         // ZR, BN = 256: z slots of the tiles done (8 per tile)
    // Hand accumulator a back to the MMA thread (after tc_fence_before and
    // __syncwarp).  PAIR: the leader's warps arrive on its barrier; the
    // peer's warps meet on their own and one of them then arrives across the
    // pair (release at cluster scope), one remote message per tile.
    uint32_t peer_phase = 0;
    const uint32_t acc_empty_cl = PAIR ? leader_addr(acc_empty) : 0u;
    auto release_acc = [&](int a) {
      if (!PAIR || leader) {
        if (lane == 0) mbar_arrive(&acc_empty[a]);
      } else {
        if (lane == 0) mbar_arrive(peer_read);
        if (ew == 0) {
          mbar_wait_bounded(peer_read, peer_phase, abort_flag, WAIT_BUDGET_NS);
          peer_phase ^= 1u;
          if (lane == 0) arrive_on_leader(acc_empty_cl);
        }
      }
    };
    // Barrier among the epilogue warps, bounded like every other wait.
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_bar);
      bool ok = mbar_wait_bounded(epi_bar, epi_phase, abort_flag, WAIT_BUDGET_NS);
      epi_phase ^= 1u;
      return ok;
    };
    // Wgrad K-split: this part's fp32 partial (the thread's row, BN/2
    // columns) goes to its slot; the part whose arrival completes the tile's
    // counter sums every part's slot in part order (its own from registers)
    // into v, so the result does not depend on which part finishes last.
    // A slot is [BN/4 column groups][128 rows] of float4, so a warp's 32 rows
    // of one group are 512 contiguous bytes.
    // Returns 1 when v holds the tile's sum, 0 when another part stores it,
    // -1 when a wait gave up.
    auto split_reduce = [&](const Tile& T, uint32_t (&v)[BN / 64][32]) -> int {
      constexpr int COLS = BN / 2;
      const int64_t row = q * 32 + lane;
      const int64_t tile_floats = 128ll * BN;
      // PAIR: each CTA's 128 rows of a pair tile are a sub-tile of their
      // own: part k of this CTA's rows in slot 2 (slot + k) + rank, its
      // arrival counter at 2 cnt + rank (the workspace holds as many slots
      // and counters as for one SM per 128-row tile)
      const int64_t sl0 = PAIR ? 2 * T.slot + rank : T.slot;  // part 0's slot
      const int64_t sstride = PAIR ? 2 : 1;                     // slots between parts
      const int64_t cnt = PAIR ? 2 * (int64_t)T.cnt + rank : (int64_t)T.cnt;
      // float4 index of (column group grp, this row): grp * 128 + row
      float4* own = reinterpret_cast<float4*>(p.split_ws + (sl0 + sstride * T.part) * tile_floats) +
                    half * (COLS / 4) * 128 + row;
#pragma unroll
      for (int i = 0; i < COLS / 32; i++) {
#pragma unroll
        for (int c = 0; c < 8; c++)
          __stcg(own + (i * 8 + c) * 128,
                 make_float4(__uint_as_float(v[i][4 * c]), __uint_as_float(v[i][4 * c + 1]),
                             __uint_as_float(v[i][4 * c + 2]), __uint_as_float(v[i][4 * c + 3])));
      }
      __threadfence();
      if (!epi_sync()) return -1;
      volatile int* flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
      if (ew == 0 && lane == 0) *flag = atomicAdd(p.split_cnt + cnt, 1) == T.parts - 1 ? 1 : 0;
      if (!epi_sync()) return -1;
      if (*flag == 0) return 0;
      __threadfence();
      const float4* base = reinterpret_cast<const float4*>(p.split_ws + sl0 * tile_floats) + half * (COLS / 4) * 128 + row;
#pragma unroll
      for (int i = 0; i < COLS / 32; i++) {
#pragma unroll
        for (int c = 0; c < 8; c++) {
          const float4 mine = make_float4(__uint_as_float(v[i][4 * c]), __uint_as_float(v[i][4 * c + 1]),
                                          __uint_as_float(v[i][4 * c + 2]), __uint_as_float(v[i][4 * c + 3]));
          float4 sum = T.part == 0 ? mine : __ldcg(base + (i * 8 + c) * 128);
          for (int pp = 1; pp < T.parts; pp++) {
            const float4 x = pp == T.part ? mine : __ldcg(base + pp * sstride * (tile_floats / 4) + (i * 8 + c) * 128);
            sum.x += x.x; sum.y += x.y; sum.z += x.z; sum.w += x.w;
          }
          v[i][4 * c] = __float_as_uint(sum.x); v[i][4 * c + 1] = __float_as_uint(sum.y);
          v[i][4 * c + 2] = __float_as_uint(sum.z); v[i][4 * c + 3] = __float_as_uint(sum.w);
        }
      }
      if (ew == 0 && lane == 0) p.split_cnt[cnt] = 0;  // ready for the next launch
      return 1;
    };
    // dGELU reads a saved activation per tile: prefetch a tile's rows into
    // L2 one tile ahead of its epilogue (dSwiGLU streams z through shared
    // memory instead).
    auto prefetch_aux = [&](int64_t i) {
      if constexpr (EPI == EPI_DGELU) {
        const int64_t t = tile_index_x<MODE, PAIR>(i);
        if (t >= p.num_tiles) return;
        const Tile U = get_tile<NT, MODE, F4>(p, t, false, order, split);
        if (!U.active || U.nk == 0) return;
        const int64_t r = U.m0 + q * 32 + lane;
        // the row's BN columns in 128-byte lines, dealt to the quarter's warps
        for (int l = ew >> 2; l < BN / 64; l += C::EW / 4) prefetch_l2(p.z + r * p.q_cols + U.n0 + 64 * l);
      }
    };
    prefetch_aux(0);
    int tqi = 0;
    uint32_t tqph = 0;
    for (int64_t i = 0;; i++) {
      int64_t t;
      if (dyn) {
        // PAIR peer: the entry was written across the pair, and its slot is
        // handed back to the leader's producer across the pair
        if (!(PAIR && !leader ? mbar_wait_cluster(&tq_full[tqi], tqph, abort_flag)
                              : mbar_wait_bounded(&tq_full[tqi], tqph, abort_flag, WAIT_BUDGET_NS)))
          break;
        t = tq[tqi];
        __syncwarp();
        if (lane == 0) {
          if (PAIR && !leader) arrive_on_leader(leader_addr(&tq_empty[tqi]));
          else mbar_arrive(&tq_empty[tqi]);
        }
        if (++tqi == C::TQN) { tqi = 0; tqph ^= 1u; }
        if (t < 0) break;
      } else {
        if (i * tile_slots<PAIR>() >= p.num_tiles) break;
        t = tile_index_x<MODE, PAIR>(i);
        if (t >= p.num_tiles) continue;
      }
      prefetch_aux(i + 1);
      Tile T = get_tile_x<NT, MODE, F4, PAIR>(p, t, ew == 0 && lane == 0, order, split, pref);
      if (!T.active) continue;
      const bool dead = PAIR && rank && !T.upper;  // PAIR: an upper half past its expert's segment
      if (PAIR) T.m0 += 128 * rank;                // this CTA's 128 rows of the pair's 256
      const int64_t row_in_tile = q * 32 + lane;
      if (T.nk == 0) {
        if (EPI == EPI_BF16) {  // zero-token expert: an exactly zero gradient slice
          const int64_t row = (MODE == MODE_WGRAD ? (int64_t)T.g * p.Mw : 0) + T.m0 + row_in_tile;
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.out_ld + T.n0 + half * (BN / 2));
#pragma unroll
          for (int c = 0; c < BN / 16; c++) dst[c] = make_uint4(0, 0, 0, 0);
        } else if (EPI == EPI_F32 && !p.accumulate) {  // stored zeros; an accumulate adds nothing
          const int64_t row = (MODE == MODE_WGRAD ? (int64_t)T.g * p.Mw : 0) + T.m0 + row_in_tile;
          uint4* dst = reinterpret_cast<uint4*>(p.out_f32 + row * p.out_ld + T.n0 + half * (BN / 2));
#pragma unroll
          for (int c = 0; c < BN / 8; c++) dst[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      if (!mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag, WAIT_BUDGET_NS)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (dead) {  // computed by the pair's MMAs, not stored
        tc_fence_before();
        __syncwarp();
        release_acc(acc);
        if (++acc == C::ACC) { acc = 0; acc_phase ^= 1u; }
        continue;
      }

      if constexpr (EPI == EPI_BF16) {
        constexpr int COLS = BN / 2;
        uint32_t v[COLS / 32][32];
#pragma unroll
        for (int i = 0; i < COLS / 32; i++) tmem_ld32(tbase + half * COLS + 32 * i, v[i]);
        tmem_wait_ld();
        if (C::ACC == 1) {
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
        bool store = true;
        const bool split_tile = MODE == MODE_WGRAD && T.parts > 1;
        if (split_tile) {
          if (C::ACC == 2) {
            tc_fence_before();
            __syncwarp();
            release_acc(acc);
          }
          const int r = split_reduce(T, v);
          if (r < 0) break;
          store = r == 1;
        }
        if (store && p.bias != nullptr) {  // bias added to the fp32 accumulator: one rounding
          const uint4* bp = reinterpret_cast<const uint4*>(p.bias + (int64_t)T.g * p.bias_ld + T.n0 + half * COLS);
#pragma unroll
          for (int i = 0; i < COLS / 32; i++) {
#pragma unroll
            for (int c = 0; c < 4; c++) {
              const uint4 bw = __ldg(bp + i * 4 + c);
              const uint32_t b4[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
              for (int k = 0; k < 8; k++) {
                const float bv = bf16_bits_to_float((k & 1) ? (b4[k >> 1] >> 16) : (b4[k >> 1] & 0xFFFFu));
                v[i][8 * c + k] = __float_as_uint(__uint_as_float(v[i][8 * c + k]) + bv);
              }
            }
          }
        }
        const int64_t row0 = (MODE == MODE_WGRAD ? (int64_t)T.g * p.Mw : 0) + T.m0 + q * 32;
        if (store) {
#pragma unroll
          for (int i = 0; i < COLS / 32; i++) {
            stage_reuse_wait(lane);
            store_bf16_block(reinterpret_cast<const float*>(v[i]), tb_bytes, lane, &tmO, T.n0 + half * COLS + 32 * i,
                             row0);
          }
        }
        if (C::ACC == 2 && !split_tile) {
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
      } else if constexpr (EPI == EPI_F32) {
        // fp32 into the caller's gradient buffer: 32x16 blocks, TMA store
        // (accumulate = 0) or TMA reduce-add (accumulate = 1)
        constexpr int COLS = BN / 2;
        uint32_t v[COLS / 32][32];
#pragma unroll
        for (int i = 0; i < COLS / 32; i++) tmem_ld32(tbase + half * COLS + 32 * i, v[i]);
        tmem_wait_ld();
        if (C::ACC == 1) {
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
        bool store = true;
        const bool split_tile = MODE == MODE_WGRAD && T.parts > 1;
        if (split_tile) {
          if (C::ACC == 2) {
            tc_fence_before();
            __syncwarp();
            release_acc(acc);
          }
          const int r = split_reduce(T, v);
          if (r < 0) break;
          store = r == 1;
        }
        const int64_t row0 = (MODE == MODE_WGRAD ? (int64_t)T.g * p.Mw : 0) + T.m0 + q * 32;
        const bool add = p.accumulate != 0;
        if (store) {
#pragma unroll
          for (int i = 0; i < COLS / 32; i++) {
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
              stage_reuse_wait(lane);
              store_f32_block(reinterpret_cast<const float*>(v[i]) + 16 * hh, tb_bytes, lane, &tmO,
                              T.n0 + half * COLS + 32 * i + 16 * hh, row0, add);
            }
          }
        }
        if (C::ACC == 2 && !split_tile) {
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        // accumulator columns: [0,128) gate of f0..f0+127, [128,256) up
        uint32_t gv[2][32], uv[2][32];
        tmem_ld32(tbase + half * 64, gv[0]);
        tmem_ld32(tbase + half * 64 + 32, gv[1]);
        tmem_ld32(tbase + 128 + half * 64, uv[0]);
        tmem_ld32(tbase + 128 + half * 64 + 32, uv[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        release_acc(acc);

        const int64_t row = T.m0 + row_in_tile;
        const int64_t f0 = T.n0;
        // BF16 pre-activation save: z = [gate | up], 32x32 blocks by TMA store
#pragma unroll
        for (int i = 0; i < 2; i++) {
          stage_reuse_wait(lane);
          store_bf16_block(reinterpret_cast<const float*>(gv[i]), tb_bytes, lane, &tmO, f0 + half * 64 + 32 * i,
                           T.m0 + q * 32);
          stage_reuse_wait(lane);
          store_bf16_block(reinterpret_cast<const float*>(uv[i]), tb_bytes, lane, &tmO, p.F + f0 + half * 64 + 32 * i,
                           T.m0 + q * 32);
        }
        stage_reuse_wait(lane);  // the transpose buffer is reused below
        // h = g * sigmoid(g) * u in fp32
        float h[2][32];
#pragma unroll
        for (int i = 0; i < 2; i++) {
#pragma unroll
          for (int j = 0; j < 32; j++) {
            float g = __uint_as_float(gv[i][j]), u = __uint_as_float(uv[i][j]);
            h[i][j] = g * sigmoidf_(g) * u;
          }
        }
        if (p.probs != nullptr) {  // the routing probability of this row
          const float prob = __ldg(p.probs + row);
#pragma unroll
          for (int i = 0; i < 2; i++) {
#pragma unroll
            for (int j = 0; j < 32; j++) h[i][j] *= prob;
          }
        }
        if (p.tap != nullptr) {
#pragma unroll
          for (int i = 0; i < 2; i++) tap_store32(p.tap, p.q_cols, row, f0 + half * 64 + 32 * i, h[i]);
        }
        uint8_t* chunk_row = sChunk;
        uint8_t* chunk_col = sChunk + 512;
        // rowwise: two thread-local 32-column blocks
#pragma unroll
        for (int i = 0; i < 2; i++) {
          float tmp[32];
#pragma unroll
          for (int j = 0; j < 32; j++) tmp[j] = h[i][j];
          uint32_t sb = row_quant_store_e4m3(tmp, p.q_row + row * p.q_cols + f0 + half * 64 + 32 * i);
          chunk_row[lane * 16 + q * 4 + half * 2 + i] = (uint8_t)sb;
        }
        // columnwise: 64 columns, each a 32-row block across the warp
#pragma unroll
        for (int i = 0; i < 2; i++) {
#pragma unroll
          for (int k = 0; k < 2; k++) {
            const int fl = half * 64 + 32 * i + 16 * k;
            col_quant16<E4M3, false>(&h[i][16 * k], tb, lane, p.q_col, p.R, f0 + fl, T.m0 + q * 32, chunk_col, fl, q);
          }
        }
        if (!epi_sync()) break;
        if (ew == 0) {
          int64_t ck = (T.m0 >> 7) * ((p.q_cols / 32 + 3) / 4) + (f0 >> 7);
          store_chunk(p.q_row_scale + ck * 512, chunk_row, lane);
        } else if (ew == 1) {
          int64_t ck = (f0 >> 7) * ((p.R / 32 + 3) / 4) + (T.m0 >> 7);
          store_chunk(p.q_col_scale + ck * 512, chunk_col, lane);
        }
        if (!epi_sync()) break;
      } else if constexpr (EPI == EPI_DSWIGLU) {
        // accumulator columns [0,BN): dh for f0..f0+BN-1.  Warp (q, half)
        // takes 32-column chunks j = 0..NST-1 at fc = 64j + 32*half for its
        // 32 rows.  BN = 128: chunk j is the warp's half of z slot j (two
        // 64-column slots per tile, every warp reads every slot).  BN = 256:
        // chunk j is z slot 2j + half of the tile (eight 32-column slots per
        // tile, a three-slot ring), and chunks 1..3 are parked in tensor
        // memory at the tile boundary so that the accumulator goes back at
        // once.
        constexpr int NST = BN / 64;
        constexpr int NCK = BN / 128;  // scale chunks per orientation and half of z
        const int64_t row = T.m0 + row_in_tile;
        const int64_t f0 = T.n0;
        uint8_t* ch_gr = sChunk;
        uint8_t* ch_ur = sChunk + 512 * NCK;
        uint8_t* ch_gc = sChunk + 1024 * NCK;
        uint8_t* ch_uc = sChunk + 1536 * NCK;
        const int zrow = q * 32 + lane;
        bool zok = true;
        float dps = 0.0f;  // routing-probability gradient: this row, this warp's columns
        const float prob = (EXT_ON && p.probs != nullptr) ? __ldg(p.probs + row) : 1.0f;
        uint32_t dh[32];
        const uint32_t park = tmem_base + ((uint32_t)(q * 32) << 16) + C::PARK_COL + (uint32_t)(half * 96);
        if constexpr (PK) {
          uint32_t t1[32], t2[32], t3[32];
          tmem_ld32(tbase + 64 + half * 32, t1);
          tmem_ld32(tbase + 128 + half * 32, t2);
          tmem_ld32(tbase + 192 + half * 32, t3);
          tmem_wait_ld();
          tmem_st32(park, t1);
          tmem_st32(park + 32, t2);
          tmem_st32(park + 64, t3);
          tmem_ld32(tbase + half * 32, dh);
          tmem_wait_ld();
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
#pragma unroll 1
        for (int j = 0; j < NST; j++) {
          const int fc = 64 * j + 32 * half;  // tile-local column of this chunk
          int zs;
          uint32_t zph;
          if constexpr (PK) {
            if (j > 0) tmem_ld32(park + (uint32_t)(j - 1) * 32u, dh);
            const uint32_t zi = zt + 2u * (uint32_t)j + (uint32_t)half;  // slot sequence number
            zs = (int)(zi % (uint32_t)C::Z_SLOTS);
            zph = (zi / (uint32_t)C::Z_SLOTS) & 1u;
          } else {
            tmem_ld32(tbase + fc, dh);
            zs = zslot;
            zph = zphase;
          }
          if (!mbar_wait_bounded(&z_full[zs], zph, abort_flag, WAIT_BUDGET_NS)) { zok = false; break; }
          // this row's 32 gate and 32 up values of the chunk
          const uint8_t* grow = sZ + zs * C::Z_SLOT + zrow * (2 * C::Z_COLS);
          const uint8_t* urow = grow + C::Z_SLOT / 2;
          uint4 zgw[4], zuw[4];
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int off = BN == 256 ? (i ^ ((zrow >> 1) & 3)) << 4           // 64-byte swizzle
                                      : ((half * 4 + i) ^ (zrow & 7)) << 4;   // 128-byte swizzle
            zgw[i] = *reinterpret_cast<const uint4*>(grow + off);
            zuw[i] = *reinterpret_cast<const uint4*>(urow + off);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&z_empty[zs]);
          if (!PK) {
            if (++zslot == C::Z_SLOTS) { zslot = 0; zphase ^= 1u; }
          }
          tmem_wait_ld();
          float dg[32], du[32];
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const uint32_t gw[4] = {zgw[i].x, zgw[i].y, zgw[i].z, zgw[i].w};
            const uint32_t uw[4] = {zuw[i].x, zuw[i].y, zuw[i].z, zuw[i].w};
#pragma unroll
            for (int k = 0; k < 8; k++) {
              const int jj = i * 8 + k;
              const float g = bf16_bits_to_float((k & 1) ? (gw[k >> 1] >> 16) : (gw[k >> 1] & 0xFFFFu));
              const float u = bf16_bits_to_float((k & 1) ? (uw[k >> 1] >> 16) : (uw[k >> 1] & 0xFFFFu));
              float d = __uint_as_float(dh[jj]);
              const float s = sigmoidf_(g);
              if (EXT_ON && p.probs != nullptr) {  // dprobs += dh * swiglu(g, u); then dh * p
                dps = fmaf(d, g * s * u, dps);
                d *= prob;
              }
              dg[jj] = d * u * s * (1.0f + g * (1.0f - s));
              du[jj] = d * g * s;
            }
          }
          if (EXT_ON && p.tap != nullptr) {
            tap_store32(p.tap, p.q_cols, row, f0 + fc, dg);
            tap_store32(p.tap, p.q_cols, row, p.F + f0 + fc, du);
          }
          // columnwise first (the rowwise packer scales its input in place)
#pragma unroll
          for (int k = 0; k < 2; k++) {
            col_quant16<E4M3, false>(&dg[16 * k], tb, lane, p.q_col, p.R, f0 + fc + 16 * k, T.m0 + q * 32,
                                     ch_gc + (fc >> 7) * 512, (fc & 127) + 16 * k, q);
            col_quant16<E4M3, false>(&du[16 * k], tb, lane, p.q_col, p.R, p.F + f0 + fc + 16 * k, T.m0 + q * 32,
                                     ch_uc + (fc >> 7) * 512, (fc & 127) + 16 * k, q);
          }
          uint32_t sbg = row_quant_store_e4m3(dg, p.q_row + row * p.q_cols + f0 + fc);
          uint32_t sbu = row_quant_store_e4m3(du, p.q_row + row * p.q_cols + p.F + f0 + fc);
          const int cb = (fc >> 7) * 512 + lane * 16 + q * 4 + ((fc >> 5) & 3);
          ch_gr[cb] = (uint8_t)sbg;
          ch_ur[cb] = (uint8_t)sbu;
        }
        if (!zok) break;
        if (PK) zt += (uint32_t)(BN / C::Z_COLS);
        if (EXT_ON && p.probs != nullptr) p.dprobs_part[row * p.dprobs_ld + (f0 / BN) * 2 + half] = dps;
        if (!PK) {
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
        if (!epi_sync()) break;
        if (ew < 4 * NCK) {
          const int64_t rcp = (p.q_cols / 32 + 3) / 4;   // row-scale chunks per 128-row block
          const int64_t ccp = (p.R / 32 + 3) / 4;        // column-scale chunks per 128-row block
          const int kind = ew / NCK, jc = ew % NCK;      // dg row, du row, dg col, du col
          const int64_t fb = (((kind & 1) ? p.F : 0) + f0) >> 7;
          const uint8_t* src = (kind == 0 ? ch_gr : kind == 1 ? ch_ur : kind == 2 ? ch_gc : ch_uc) + jc * 512;
          if (kind < 2) store_chunk(p.q_row_scale + ((T.m0 >> 7) * rcp + fb + jc) * 512, src, lane);
          else store_chunk(p.q_col_scale + ((fb + jc) * ccp + (T.m0 >> 7)) * 512, src, lane);
        }
        if (!epi_sync()) break;
      } else if constexpr (EPI == EPI_GELU || EPI == EPI_DGELU) {
        // Dense MLP epilogues, accumulator columns [0,BN) = output columns
        // n0..n0+BN-1 in 32-column chunks, chunk c of lane quarter q taken
        // by the quarter's warp c mod (EW / 4).  GELU: pre = acc + b1 (saved in
        // BF16), act = gelu(pre); dGELU: dpre = acc * gelu'(pre from the BF16
        // save), plus per-column sums of dpre (the bias gradient).  Both
        // requantize rowwise and columnwise with optional rotation.
        constexpr int BB = BlockBytes<QF>::value;
        constexpr int EPQ = C::EW / 4;                     // epilogue warps per lane quarter
        constexpr int NCHMAX = (BN / 32 + EPQ - 1) / EPQ;  // most 32-column chunks a warp takes
        const int wq = ew >> 2;                            // this warp's index within its quarter
        const int nchw = (BN / 32 - wq + EPQ - 1) / EPQ;   // its chunks: wq, wq + EPQ, ... (warp-uniform)
        const int64_t row = T.m0 + row_in_tile;
        const int64_t n0 = T.n0;
        uint8_t* ch_row = sChunk;                   // BN/128 rowwise scale chunks
        uint8_t* ch_col = sChunk + 4 * BN;          // BN/128 columnwise scale chunks
        float* part = reinterpret_cast<float*>(sChunk + 8 * BN);  // [4 lane quarters][BN columns]
        uint32_t accr[32];
        // PK: the warp's chunks after its first go to tensor-memory columns
        // past the scale slots and the first to registers; then the
        // accumulator is free for the next tile's MMAs while this one is
        // requantized.
        const uint32_t park =
            tmem_base + ((uint32_t)(q * 32) << 16) + C::PARK_COL + (uint32_t)(wq * (NCHMAX - 1) * 32);
        if constexpr (PK) {
          static_assert(!PK || C::PARK_COL + EPQ * (NCHMAX - 1) * 32 <= C::TMEM_COLS, "parked chunks must fit");
          // one chunk at a time through accr (its registers are reused only
          // after the store has completed)
#pragma unroll 1
          for (int k = 1; k < nchw; k++) {
            tmem_ld32(tbase + 32 * (wq + EPQ * k), accr);
            tmem_wait_ld();
            tmem_st32(park + 32 * (k - 1), accr);
            tmem_wait_st();
          }
          tmem_ld32(tbase + 32 * wq, accr);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
#pragma unroll 1
        for (int ch = 0; ch < nchw; ch++) {
          const int fc = 32 * (wq + EPQ * ch);
          if (!PK) tmem_ld32(tbase + fc, accr);
          else if (ch > 0) tmem_ld32(park + (uint32_t)(ch - 1) * 32u, accr);
          float aux[32];  // GELU: bias; dGELU: saved pre-activation
          if (EPI == EPI_GELU && p.bias == nullptr) {
#pragma unroll
            for (int j = 0; j < 32; j++) aux[j] = 0.f;
          } else {
            const uint4* src = EPI == EPI_GELU ? reinterpret_cast<const uint4*>(p.bias + n0 + fc)
                                               : reinterpret_cast<const uint4*>(p.z + row * p.q_cols + n0 + fc);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const uint4 w = EPI == EPI_GELU ? __ldg(src + i) : src[i];
              const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 8; k++)
                aux[i * 8 + k] = bf16_bits_to_float((k & 1) ? (w4[k >> 1] >> 16) : (w4[k >> 1] & 0xFFFFu));
            }
          }
          tmem_wait_ld();
          float val[32];
          if constexpr (EPI == EPI_GELU) {
            float pre[32];
#pragma unroll
            for (int j = 0; j < 32; j++) pre[j] = __uint_as_float(accr[j]) + aux[j];
            stage_reuse_wait(lane);
            store_bf16_block(pre, tb_bytes, lane, &tmO, n0 + fc, T.m0 + q * 32);
            stage_reuse_wait(lane);  // the transpose buffer is reused below
#pragma unroll
            for (int j = 0; j < 32; j++) val[j] = gelu_tanh_f(pre[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; j++) val[j] = __uint_as_float(accr[j]) * dgelu_tanh_f(aux[j]);
          }
          if (p.tap != nullptr) tap_store32(p.tap, p.q_cols, row, n0 + fc, val);
          // columnwise first (the rowwise packer rotates and scales in place)
#pragma unroll
          for (int k = 0; k < 2; k++)  // dGELU: this warp's 32-row column sums from the transpose
            col_quant16<QF, QH>(&val[16 * k], tb, lane, p.q_col, p.q_col_ld, n0 + fc + 16 * k,
                                (T.m0 + q * 32) / 32 * BB, ch_col + (fc >> 7) * 512, (fc & 127) + 16 * k, q,
                                EPI == EPI_DGELU ? part + q * BN + fc + 16 * k : nullptr);
          const uint32_t sbr = row_quant_store<QF, QH>(val, p.q_row + row * p.q_row_ld + (n0 + fc) / 32 * BB);
          ch_row[(fc >> 7) * 512 + lane * 16 + q * 4 + ((fc >> 5) & 3)] = (uint8_t)sbr;
        }
        if (!PK) {
          tc_fence_before();
          __syncwarp();
          release_acc(acc);
        }
        if (!epi_sync()) break;
        constexpr int NCK = BN / 128;  // scale chunks per orientation
        if (ew < NCK)
          store_chunk(p.q_row_scale + ((T.m0 >> 7) * ((p.q_cols / 32 + 3) / 4) + (n0 >> 7) + ew) * 512,
                      ch_row + ew * 512, lane);
        else if (ew < 2 * NCK)
          store_chunk(p.q_col_scale + (((n0 >> 7) + ew - NCK) * ((p.R / 32 + 3) / 4) + (T.m0 >> 7)) * 512,
                      ch_col + (ew - NCK) * 512, lane);
        if constexpr (EPI == EPI_DGELU) {
          // BN columns: epilogue warps 0..7 at BN = 256, 2..5 at 128
          const int c = BN == 256 ? ew * 32 + lane : ew * 32 + lane - 64;
          if (c >= 0 && c < BN) {
            float s4 = part[c];
            s4 += part[BN + c];
            s4 += part[2 * BN + c];
            s4 += part[3 * BN + c];
            p.colsum_partials[(T.m0 >> 7) * p.q_cols + n0 + c] = s4;
          }
        }
        if (!epi_sync()) break;
      }
      if (++acc == C::ACC) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores have landed
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_gemm_status, DEV_TIMEOUT);
  if constexpr (PAIR) {
    cluster_sync_all();  // neither CTA frees tensor memory or exits while the other still uses the pair
    tc_fence_after();
    if (warp == 1)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem_base), "n"(C::TMEM_COLS)
                   : "memory");
    cluster_sync_all();
  } else if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<C::TMEM_COLS>(tmem_base);
  }
}

}  // namespace mx
