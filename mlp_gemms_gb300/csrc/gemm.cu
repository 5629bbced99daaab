// Ragged grouped block-scaled GEMM on the 5th-generation tensor core, with
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
//               K=32 per instruction, fp32 accumulators in tensor memory);
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//               32*(w%4)..+31, two warps per lane quarter split the
//               columns), then the fused math and stores.
// With BN = 256 there is one accumulator buffer; the epilogue copies it to
// registers and releases it before its math, so the next tile's MMAs run
// under the epilogue.  With BN = 128 two accumulator buffers alternate.
// Every wait is bounded in time; on expiry the kernel records a device
// status bit and unwinds without leaving copies or MMAs in flight.
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

__device__ unsigned g_gemm_status = 0;

constexpr int NUM_THREADS = 320;
constexpr int EPI_THREADS = 256;
constexpr uint64_t WAIT_BUDGET_NS = 2000000000ull;

template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : 5;
  static constexpr int ACC = BN == 256 ? 1 : 2;
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SF_BYTES = 512 + (BN / 128) * 512;
  static constexpr int SF_COLS = 4 + 4 * (BN / 128);
  static constexpr uint32_t TX = A_BYTES + B_BYTES + SF_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_TB = OFF_SF + STAGES * SF_BYTES;  // 8 x 2 KB transpose buffers
  static constexpr int OFF_CHUNK = OFF_TB + 8 * 2048;        // 4 scale chunks
  static constexpr int OFF_BAR = OFF_CHUNK + 4 * 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC + 2;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;    // + slack for 1024-byte alignment
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SF_TMEM_BASE = 256;
  static_assert(ACC * BN <= 256, "accumulators live in tensor-memory columns 0..255");
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "scale slots must fit");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

struct Tile {
  int active;
  int g;
  int64_t m0, n0;
  int64_t kbeg;
  int nk;
};

__device__ __forceinline__ int32_t ldg_i32(const int32_t* p) { return __ldg(p); }

// Tile t -> (expert, row base, column base, K range).  Grouped: tiles are
// row-block-major over all R rows; the expert is the segment holding the
// row base.  Wgrad: tiles are expert-major; K runs over the expert's rows.
template <int NT, int MODE>
__device__ __forceinline__ Tile get_tile(const GemmParams& p, int64_t t, bool report) {
  Tile T;
  T.active = 0; T.g = 0; T.m0 = 0; T.n0 = 0; T.kbeg = 0; T.nk = 0;
  if (MODE == MODE_GROUPED) {
    int64_t mt = t / p.n_tiles, nt = t % p.n_tiles;
    T.m0 = mt * 128;
    T.n0 = nt * NT;
    int64_t total = ldg_i32(p.offsets + p.G - 1);
    if (T.m0 >= total) return T;  // inactive tail
    int lo = 0, hi = p.G - 1;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if ((int64_t)ldg_i32(p.offsets + mid) > T.m0) hi = mid; else lo = mid + 1;
    }
    int64_t end = ldg_i32(p.offsets + lo);
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
    T.g = (int)(t / per_g);
    int64_t rem = t % per_g;
    T.m0 = (rem / p.n_tiles) * 128;
    T.n0 = (rem % p.n_tiles) * NT;
    int64_t end = ldg_i32(p.offsets + T.g);
    int64_t start = T.g ? ldg_i32(p.offsets + T.g - 1) : 0;
    bool bad = (start & 127) || (end & 127) || end < start || end > p.R || start < 0;
    if (bad && report) atomicOr(&g_gemm_status, DEV_BAD_OFFSETS);
    T.kbeg = bad ? 0 : start;
    T.nk = bad ? 0 : (int)((end - start) / 128);
    T.active = 1;
  }
  return T;
}

// ---- epilogue helpers --------------------------------------------------

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Rowwise E4M3 requant of 32 fp32 values held by one thread.
__device__ __forceinline__ uint32_t row_quant_store_e4m3(float (&v)[32], uint8_t* dst) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 32; i++) amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  uint32_t sb = rceil_scale_byte<E4M3>(amax);
  uint32_t w[8];
  quantize_block_words<E4M3>(v, sb, w);
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return sb;
}

// Columnwise E4M3 requant of two columns whose 32-row block is spread over
// the warp's lanes (lane = row): warp-wide integer max of |bits| gives each
// column's amax; both codes go to the transpose buffer tb[col][lane].
__device__ __forceinline__ void col_quant_pair_e4m3(float v0, float v1, uint8_t* tb_col0, uint8_t* tb_col1,
                                                    uint32_t& sb0, uint32_t& sb1, int lane) {
  uint32_t a0 = __reduce_max_sync(0xffffffffu, __float_as_uint(v0) & 0x7FFFFFFFu);
  uint32_t a1 = __reduce_max_sync(0xffffffffu, __float_as_uint(v1) & 0x7FFFFFFFu);
  sb0 = rceil_scale_byte<E4M3>(a0);
  sb1 = rceil_scale_byte<E4M3>(a1);
  uint32_t c = cvt_e4m3x2(v0 * inv_scale_from_byte(sb0), v1 * inv_scale_from_byte(sb1));
  uint32_t c0 = sb0 == 0xFFu ? 0x7Fu : (c & 0xFFu);
  uint32_t c1 = sb1 == 0xFFu ? 0x7Fu : (c >> 8);
  tb_col0[lane] = (uint8_t)c0;
  tb_col1[lane] = (uint8_t)c1;
}

__device__ __forceinline__ void store_chunk(uint8_t* dst, const uint8_t* chunk, int lane) {
  reinterpret_cast<uint4*>(dst)[lane] = reinterpret_cast<const uint4*>(chunk)[lane];
}

// ---- the kernel ---------------------------------------------------------

template <int BN, int EPI, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const GemmParams p) {
  using C = Cfg<BN>;
  constexpr int NT = (EPI == EPI_SWIGLU) ? 128 : BN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sSF = smem + C::OFF_SF;
  uint8_t* sTB = smem + C::OFF_TB;
  uint8_t* sChunk = smem + C::OFF_CHUNK;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + C::ACC;
  uint64_t* final_bar = acc_empty + C::ACC;
  uint64_t* epi_bar = final_bar + 1;  // the 8 epilogue warps' own barrier
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; s++) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < C::ACC; a++) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], 8); }
    mbar_init(final_bar, 1);
    mbar_init(epi_bar, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) { prefetch_tensormap(&tmA); prefetch_tensormap(&tmB); }
  if (warp == 1) tmem_alloc<C::TMEM_COLS>(tmem_slot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_first();
      const uint64_t pol_b = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int armed_parity[C::STAGES];
      for (int s = 0; s < C::STAGES; s++) armed_parity[s] = -1;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        Tile T = get_tile<NT, MODE>(p, t, false);
        if (!T.active || T.nk == 0) continue;
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
          mbar_arrive_expect_tx(&full[stage], C::TX);
          armed_parity[stage] = (int)phase;
          const int64_t kc = T.kbeg / 128 + kb;
          const int kx = (int)(kc * 128);
          tma_load_2d(sA + stage * C::A_BYTES, &tmA, kx, (int)T.m0, &full[stage], pol_a);
#pragma unroll
          for (int i = 0; i < BN / 128; i++)
            tma_load_2d(sB + stage * C::B_BYTES + i * 16384, &tmB, kx, (int)brow[i], &full[stage], pol_b);
          uint8_t* sf = sSF + stage * C::SF_BYTES;
          bulk_load(sf, p.sfa + ((T.m0 >> 7) * p.sfa_kchunks + kc) * 512, 512, &full[stage]);
#pragma unroll
          for (int i = 0; i < BN / 128; i++)
            bulk_load(sf + 512 + i * 512, p.sfb + ((brow[i] >> 7) * p.sfb_kchunks + kc) * 512, 512, &full[stage]);
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
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        Tile T = get_tile<NT, MODE>(p, t, false);
        if (!T.active || T.nk == 0) continue;
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < T.nk; kb++) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, WAIT_BUDGET_NS)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + C::SF_TMEM_BASE + (uint32_t)(stage * C::SF_COLS);
          const uint32_t sf_s = smem_u32(sSF + stage * C::SF_BYTES);
          tc_copy_scales(sf_t, sf_s);
#pragma unroll
          for (int i = 0; i < BN / 128; i++) tc_copy_scales(sf_t + 4 + 4 * i, sf_s + 512 + 512 * i);
          const uint32_t a_s = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_s = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const uint64_t adesc = smem_desc(a_s + 32 * j, 16, 1024, 2);
            const uint64_t bdesc = smem_desc(b_s + 32 * j, 16, 1024, 2);
            const uint32_t idesc = mma_idesc_mx((uint32_t)p.a_type, (uint32_t)p.b_type, 128, BN, j, j);
            tc_mma_mx(d_tmem, adesc, bdesc, idesc, sf_t, sf_t + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::ACC) { acc = 0; acc_phase ^= 1u; }
      }
      // No MMA may still be writing tensor memory when it is freed.
      volatile int no_abort = 0;
      tc_commit(final_bar);
      mbar_wait_bounded(final_bar, 0, &no_abort, WAIT_BUDGET_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;       // 0..7
    const int q = warp & 3;        // tensor-memory lane quarter
    const int half = ew >> 2;      // column half
    uint8_t* tb = sTB + ew * 2048;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t epi_phase = 0;
    // Barrier among the epilogue warps, bounded like every other wait.
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_bar);
      bool ok = mbar_wait_bounded(epi_bar, epi_phase, abort_flag, WAIT_BUDGET_NS);
      epi_phase ^= 1u;
      return ok;
    };
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      Tile T = get_tile<NT, MODE>(p, t, ew == 0 && lane == 0);
      if (!T.active) continue;
      const int64_t row_in_tile = q * 32 + lane;
      if (T.nk == 0) {
        if (EPI == EPI_BF16) {  // zero-token expert: an exactly zero gradient slice
          const int64_t row = (MODE == MODE_WGRAD ? (int64_t)T.g * p.Mw : 0) + T.m0 + row_in_tile;
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.out_ld + T.n0 + half * (BN / 2));
#pragma unroll
          for (int c = 0; c < BN / 16; c++) dst[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      if (!mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag, WAIT_BUDGET_NS)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);

      if constexpr (EPI == EPI_BF16) {
        constexpr int COLS = BN / 2;
        uint32_t v[COLS / 32][32];
#pragma unroll
        for (int i = 0; i < COLS / 32; i++) tmem_ld32(tbase + half * COLS + 32 * i, v[i]);
        tmem_wait_ld();
        if (C::ACC == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
        const int64_t row = (MODE == MODE_WGRAD ? (int64_t)T.g * p.Mw : 0) + T.m0 + row_in_tile;
        uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.out_ld + T.n0 + half * COLS);
#pragma unroll
        for (int i = 0; i < COLS / 32; i++) {
#pragma unroll
          for (int c = 0; c < 4; c++) {
            const uint32_t* s = &v[i][8 * c];
            dst[i * 4 + c] = make_uint4(
                float2_to_bf16x2(__uint_as_float(s[0]), __uint_as_float(s[1])),
                float2_to_bf16x2(__uint_as_float(s[2]), __uint_as_float(s[3])),
                float2_to_bf16x2(__uint_as_float(s[4]), __uint_as_float(s[5])),
                float2_to_bf16x2(__uint_as_float(s[6]), __uint_as_float(s[7])));
          }
        }
        if (C::ACC == 2) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
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
        if (lane == 0) mbar_arrive(&acc_empty[acc]);

        const int64_t row = T.m0 + row_in_tile;
        const int64_t f0 = T.n0;
        // BF16 pre-activation save: z = [gate | up]
        uint16_t* zr = p.z + row * (2 * p.F);
        uint4* zg = reinterpret_cast<uint4*>(zr + f0 + half * 64);
        uint4* zu = reinterpret_cast<uint4*>(zr + p.F + f0 + half * 64);
#pragma unroll
        for (int i = 0; i < 2; i++) {
#pragma unroll
          for (int c = 0; c < 4; c++) {
            const uint32_t* s = &gv[i][8 * c];
            zg[i * 4 + c] = make_uint4(float2_to_bf16x2(__uint_as_float(s[0]), __uint_as_float(s[1])),
                                       float2_to_bf16x2(__uint_as_float(s[2]), __uint_as_float(s[3])),
                                       float2_to_bf16x2(__uint_as_float(s[4]), __uint_as_float(s[5])),
                                       float2_to_bf16x2(__uint_as_float(s[6]), __uint_as_float(s[7])));
            const uint32_t* u = &uv[i][8 * c];
            zu[i * 4 + c] = make_uint4(float2_to_bf16x2(__uint_as_float(u[0]), __uint_as_float(u[1])),
                                       float2_to_bf16x2(__uint_as_float(u[2]), __uint_as_float(u[3])),
                                       float2_to_bf16x2(__uint_as_float(u[4]), __uint_as_float(u[5])),
                                       float2_to_bf16x2(__uint_as_float(u[6]), __uint_as_float(u[7])));
          }
        }
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
          for (int j = 0; j < 32; j += 2) {
            const int col = i * 32 + j;  // 0..63 within this thread's half
            uint32_t sb0, sb1;
            col_quant_pair_e4m3(h[i][j], h[i][j + 1], tb + col * 32, tb + (col + 1) * 32, sb0, sb1, lane);
            if (lane == 0) {
              const int f = half * 64 + col;
              chunk_col[(f & 31) * 16 + (f >> 5) * 4 + q] = (uint8_t)sb0;
              chunk_col[((f + 1) & 31) * 16 + ((f + 1) >> 5) * 4 + q] = (uint8_t)sb1;
            }
          }
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; k++) {
          const int col = lane + 32 * k;
          const uint4* s = reinterpret_cast<const uint4*>(tb + col * 32);
          uint4* d = reinterpret_cast<uint4*>(p.q_col + (f0 + half * 64 + col) * p.R + T.m0 + q * 32);
          d[0] = s[0];
          d[1] = s[1];
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
        // accumulator columns [0,128): dh for f0..f0+127
        const int64_t row = T.m0 + row_in_tile;
        const int64_t f0 = T.n0;
        const uint16_t* zr = p.z + row * (2 * p.F);
        uint8_t* ch_gr = sChunk;
        uint8_t* ch_ur = sChunk + 512;
        uint8_t* ch_gc = sChunk + 1024;
        uint8_t* ch_uc = sChunk + 1536;
#pragma unroll 1
        for (int ch = 0; ch < 2; ch++) {
          const int fc = half * 64 + ch * 32;  // tile-local column of this chunk
          uint32_t dh[32];
          tmem_ld32(tbase + fc, dh);
          uint4 zgw[4], zuw[4];
          const uint4* zgp = reinterpret_cast<const uint4*>(zr + f0 + fc);
          const uint4* zup = reinterpret_cast<const uint4*>(zr + p.F + f0 + fc);
#pragma unroll
          for (int i = 0; i < 4; i++) { zgw[i] = zgp[i]; zuw[i] = zup[i]; }
          tmem_wait_ld();
          float dg[32], du[32];
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const uint32_t gw[4] = {zgw[i].x, zgw[i].y, zgw[i].z, zgw[i].w};
            const uint32_t uw[4] = {zuw[i].x, zuw[i].y, zuw[i].z, zuw[i].w};
#pragma unroll
            for (int k = 0; k < 8; k++) {
              const int j = i * 8 + k;
              const float g = bf16_bits_to_float((k & 1) ? (gw[k >> 1] >> 16) : (gw[k >> 1] & 0xFFFFu));
              const float u = bf16_bits_to_float((k & 1) ? (uw[k >> 1] >> 16) : (uw[k >> 1] & 0xFFFFu));
              const float d = __uint_as_float(dh[j]);
              const float s = sigmoidf_(g);
              dg[j] = d * u * s * (1.0f + g * (1.0f - s));
              du[j] = d * g * s;
            }
          }
          // columnwise first (the rowwise packer scales its input in place)
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            uint32_t sb0, sb1, sb2, sb3;
            col_quant_pair_e4m3(dg[j], dg[j + 1], tb + j * 32, tb + (j + 1) * 32, sb0, sb1, lane);
            col_quant_pair_e4m3(du[j], du[j + 1], tb + (32 + j) * 32, tb + (33 + j) * 32, sb2, sb3, lane);
            if (lane == 0) {
              const int f = fc + j;
              ch_gc[(f & 31) * 16 + (f >> 5) * 4 + q] = (uint8_t)sb0;
              ch_gc[((f + 1) & 31) * 16 + ((f + 1) >> 5) * 4 + q] = (uint8_t)sb1;
              ch_uc[(f & 31) * 16 + (f >> 5) * 4 + q] = (uint8_t)sb2;
              ch_uc[((f + 1) & 31) * 16 + ((f + 1) >> 5) * 4 + q] = (uint8_t)sb3;
            }
          }
          __syncwarp();
          {
            const uint4* sg = reinterpret_cast<const uint4*>(tb + lane * 32);
            uint4* dgc = reinterpret_cast<uint4*>(p.q_col + (f0 + fc + lane) * p.R + T.m0 + q * 32);
            dgc[0] = sg[0];
            dgc[1] = sg[1];
            const uint4* su = reinterpret_cast<const uint4*>(tb + (32 + lane) * 32);
            uint4* duc = reinterpret_cast<uint4*>(p.q_col + (p.F + f0 + fc + lane) * p.R + T.m0 + q * 32);
            duc[0] = su[0];
            duc[1] = su[1];
          }
          __syncwarp();
          uint32_t sbg = row_quant_store_e4m3(dg, p.q_row + row * p.q_cols + f0 + fc);
          uint32_t sbu = row_quant_store_e4m3(du, p.q_row + row * p.q_cols + p.F + f0 + fc);
          ch_gr[lane * 16 + q * 4 + (fc >> 5)] = (uint8_t)sbg;
          ch_ur[lane * 16 + q * 4 + (fc >> 5)] = (uint8_t)sbu;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        if (!epi_sync()) break;
        {
          const int64_t rcp = (p.q_cols / 32 + 3) / 4;   // row-scale chunks per 128-row block
          const int64_t ccp = (p.R / 32 + 3) / 4;        // column-scale chunks per 128-row block
          if (ew == 0) store_chunk(p.q_row_scale + ((T.m0 >> 7) * rcp + (f0 >> 7)) * 512, ch_gr, lane);
          else if (ew == 1) store_chunk(p.q_row_scale + ((T.m0 >> 7) * rcp + ((p.F + f0) >> 7)) * 512, ch_ur, lane);
          else if (ew == 2) store_chunk(p.q_col_scale + ((f0 >> 7) * ccp + (T.m0 >> 7)) * 512, ch_gc, lane);
          else if (ew == 3) store_chunk(p.q_col_scale + (((p.F + f0) >> 7) * ccp + (T.m0 >> 7)) * 512, ch_uc, lane);
        }
        if (!epi_sync()) break;
      }
      if (++acc == C::ACC) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_gemm_status, DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<C::TMEM_COLS>(tmem_base);
  }
}

template <int BN, int EPI, int MODE>
static cudaError_t launch_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              cudaStream_t s, int num_sms) {
  auto kern = mx_gemm_kernel<BN, EPI, MODE>;
  constexpr int smem = Cfg<BN>::SMEM_BYTES;
  static bool configured = false;  // per instantiation; attribute set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int64_t grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, NUM_THREADS, smem, s>>>(ta, tb, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb, int bn,
                        cudaStream_t s, int num_sms) {
  if (p.epi == EPI_SWIGLU) return launch_one<256, EPI_SWIGLU, MODE_GROUPED>(p, ta, tb, s, num_sms);
  if (p.epi == EPI_DSWIGLU) return launch_one<128, EPI_DSWIGLU, MODE_GROUPED>(p, ta, tb, s, num_sms);
  if (p.mode == MODE_WGRAD) {
    if (bn == 128) return launch_one<128, EPI_BF16, MODE_WGRAD>(p, ta, tb, s, num_sms);
    return launch_one<256, EPI_BF16, MODE_WGRAD>(p, ta, tb, s, num_sms);
  }
  if (bn == 128) return launch_one<128, EPI_BF16, MODE_GROUPED>(p, ta, tb, s, num_sms);
  return launch_one<256, EPI_BF16, MODE_GROUPED>(p, ta, tb, s, num_sms);
}

cudaError_t read_gemm_status(unsigned* out) {
  return cudaMemcpyFromSymbol(out, g_gemm_status, sizeof(unsigned));
}
cudaError_t reset_gemm_status() {
  unsigned z = 0;
  return cudaMemcpyToSymbol(g_gemm_status, &z, sizeof(unsigned));
}

// A bounded wait that nothing completes: the self-test of the timeout path.
__global__ void wait_selftest_kernel(uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0, &abort_flag, budget_ns)) atomicOr(&g_gemm_status, DEV_TIMEOUT);
  }
}

cudaError_t launch_wait_selftest(uint64_t budget_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(budget_ns);
  return cudaGetLastError();
}

}  // namespace mx
