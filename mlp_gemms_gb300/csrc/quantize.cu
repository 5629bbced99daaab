// MX quantizer: BF16 [batch, rows, cols] -> rowwise 1x32 and/or columnwise
// 32x1 MX payload with E8M0 RCEIL scales in the blocked 128x4 layout,
// optional 32-point Hadamard rotation per block and optional per-column sums.
//
// torchao PR #5 "MXFP8 cudnn-fe Swiglu fused Grouped MLP fwd/bwd and wgrad
// group gemm": shared-infrastructure commit (RCEIL E8M0, NaN-propagating
// amax, blocked-scale indexing; rowwise 1x32 and columnwise 32x1
// quantization) and the correctness-first kernels commit (dual-orientation
// quantization).  Primus PR #1064 "feat(mxfp6): MXFP6 (E2M3) Flux linears, a
// fused MLP, and the MLPerf recipe": Hadamard folded into the packer; the
// per-column sum (bias gradient) returned by the packer and finished by a
// separate reduction.
//
// One CTA (256 threads) owns a 128-row x 128-column tile: it stages the BF16
// tile in shared memory with 16-byte coalesced loads, then
//   * rowwise: warp lanes take 32 consecutive rows, each thread one 32-column
//     block -- thread-local amax, scale, pack, 32-byte store;
//   * columnwise: each thread takes a pair of columns over one 32-row block
//     (word loads from shared memory, conflict-free) -- the pair's amax comes
//     from packed 16-bit integer max, the two blocks are packed and stored as
//     rows of the transposed payload.
// The tile's 128x4 scales of each orientation form exactly one 512-byte
// blocked chunk, assembled in shared memory and written with one coalesced
// store.  Column sums are fp32 per tile ([ceil(rows/128), cols] partials),
// reduced in a fixed order by a second kernel: deterministic, no atomics.
#include <mutex>

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

__device__ unsigned g_quant_status = 0;

struct QuantParams {
  const uint16_t* x;
  int64_t rows, cols, ld, x_batch_stride;  // elements
  uint8_t* row_data;
  uint8_t* row_scale;
  int64_t row_ld, row_batch_stride, row_scale_batch_stride;  // bytes
  uint8_t* col_data;
  uint8_t* col_scale;
  int64_t col_ld, col_batch_stride, col_scale_batch_stride;  // bytes
  float* colsum_partials;  // [ceil(rows/128), cols] or null
  int tiles_x;             // ceil(cols / 128)
  int batch;
  uint64_t seed;           // stochastic rounding: the generator's key
  // gather (token permute): output row r quantizes x row src[r] (a zero row
  // where src[r] < 0); rows from offsets[G-1] on are not produced
  const int32_t* src;
  int64_t src_rows;        // rows of x
  const int32_t* offsets;
  int G;
};

// Non-bulk asynchronous 16-byte copy global -> shared; src_bytes = 0 writes
// 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on the barrier once this thread's earlier cp.async copies have
// landed; counts against the barrier's expected arrivals.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr int QT = 128;          // tile edge

// NaN-propagating amax of BF16 pairs, per 16-bit half: a tree of
// max.NaN.xorsign.abs.bf16x2 (magnitude max(|a|, |b|), NaN if either is
// NaN), sign bits cleared at the end; a NaN shows as a pattern above Inf.
__device__ __forceinline__ uint32_t absmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <int N>
__device__ __forceinline__ uint32_t amax_bf16_pairs(const uint32_t* w) {
  uint32_t t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; i++) t[i] = absmax2(w[2 * i], w[2 * i + 1]);
#pragma unroll
  for (int n = N / 4; n >= 1; n >>= 1) {
#pragma unroll
    for (int i = 0; i < n; i++) t[i] = absmax2(t[i], t[i + n]);
  }
  return t[0] & 0x7FFF7FFFu;
}

template <int FMT>
__device__ __forceinline__ void store_block(uint8_t* dst, const uint32_t (&w)[8]) {
  if constexpr (FMT == E4M3) {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else if constexpr (FMT == E2M1) {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  } else {  // 24 bytes, 8-byte aligned
    reinterpret_cast<uint2*>(dst)[0] = make_uint2(w[0], w[1]);
    reinterpret_cast<uint2*>(dst)[1] = make_uint2(w[2], w[3]);
    reinterpret_cast<uint2*>(dst)[2] = make_uint2(w[4], w[5]);
  }
}

// ---- stochastic rounding ----------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC 2011): ten rounds of two 32x32->64 multiplies and xors, the
// key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; round++) {
    if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Grid of an element format for stochastic rounding: mantissa bits, the
// smallest normal exponent (the subnormal spacing is 2^(emin - m)) and the
// largest finite value.
template <int FMT> struct SrGrid;
template <> struct SrGrid<E2M3> { static constexpr int M = 3, EMIN = 0; static constexpr float VMAX = 7.5f; };
template <> struct SrGrid<E2M1> { static constexpr int M = 1, EMIN = 0; static constexpr float VMAX = 6.0f; };

// A scaled value rounded stochastically onto the format's grid: saturating
// at +-max; otherwise the lower neighbour lo = floor(|a| / spacing) * spacing
// (spacing = 2^es, es = max(E, emin) - m, E the fp32 exponent of |a|) or
// lo + spacing, the latter when (u >> 8) < frac * 2^24 with frac = (|a| - lo)
// / spacing.  Evaluated with full-rate operations only, every step exact:
// lo = (|a| + 2^(es+23)) rounded toward zero, minus 2^(es+23); the
// comparison as (u >> 8) * 2^(es-24) < |a| - lo, that threshold assembled
// from the bits of u (2^(es-1) + (bits 8..30) * 2^(es-24), less 2^(es-1)
// unless bit 31 is set).  The result is on the grid, so the
// round-to-nearest conversion that follows is exact; the sign (of zero too)
// is kept.
template <int FMT>
__device__ __forceinline__ float sr_round(float a_signed, uint32_t u) {
  constexpr int M = SrGrid<FMT>::M;
  const float a = fabsf(a_signed);
  const uint32_t bc = max(__float_as_uint(a) >> 23, (uint32_t)(127 + SrGrid<FMT>::EMIN));  // biased max(E, emin)
  const float c = __uint_as_float((bc - M + 23) << 23);                  // 2^(es+23)
  const float lo = __fadd_rz(a, c) - c;
  const float rem = a - lo;
  const uint32_t h = (bc - M - 1) << 23;                                 // 2^(es-1)
  const float hp = __uint_as_float(h | ((u >> 8) & 0x7FFFFFu));
  const float thr = (u >> 31) ? hp : hp - __uint_as_float(h);
  const float sp = __uint_as_float((bc - M) << 23);
  const float r = thr < rem ? lo + sp : lo;
  return copysignf(a < SrGrid<FMT>::VMAX ? r : SrGrid<FMT>::VMAX, a_signed);
}

// Stochastic-rounding variant of the block packer: element i of the block is
// element idx0 + i of its output grid (idx0 a multiple of 32); its bits are
// word (idx % 4) of Philox at counter (idx / 4, orient, 0), key the seed.
template <int FMT>
__device__ __forceinline__ void quantize_block_words_sr(float (&v)[32], uint32_t sb, uint32_t (&w)[8],
                                                        uint64_t seed, uint64_t idx0, uint32_t orient) {
  if (sb == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; i++) w[i] = nan_block_word<FMT>();
    return;
  }
  scale_values<32>(v, inv_scale_from_byte(sb));
#pragma unroll
  for (int g = 0; g < 8; g++) {
    const uint64_t n = (idx0 >> 2) + (uint64_t)g;
    const uint4 r = philox4x32_10((uint32_t)n, (uint32_t)(n >> 32), orient, 0u, (uint32_t)seed,
                                  (uint32_t)(seed >> 32));
    v[4 * g] = sr_round<FMT>(v[4 * g], r.x);
    v[4 * g + 1] = sr_round<FMT>(v[4 * g + 1], r.y);
    v[4 * g + 2] = sr_round<FMT>(v[4 * g + 2], r.z);
    v[4 * g + 3] = sr_round<FMT>(v[4 * g + 3], r.w);
  }
  pack_block<FMT>(v, w);
}

// Quantize 32 fp32 values (rotating first if HAD) and return the scale byte.
template <int FMT, bool HAD, bool SR = false>
__device__ __forceinline__ uint32_t quantize32(float (&v)[32], uint32_t amax_bits_prerot, uint32_t (&w)[8],
                                               uint64_t seed = 0, uint64_t idx0 = 0, uint32_t orient = 0) {
  uint32_t amax_bits = amax_bits_prerot;
  if constexpr (HAD) {
    hadamard32(v);
    amax_bits = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  }
  uint32_t sb = rceil_scale_byte<FMT>(amax_bits);
  if constexpr (SR) quantize_block_words_sr<FMT>(v, sb, w, seed, idx0, orient);
  else quantize_block_words<FMT>(v, sb, w);
  return sb;
}

// Byte offset of BF16 element (r, c) of a 128x128 tile held as two
// 128-byte-swizzled TMA boxes of 64 columns: the 16-byte chunk index within
// each 128-byte row is XORed with (r % 8), so both the row-major 16-byte
// reads (8 consecutive rows) and the word reads along one row are free of
// bank conflicts.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  const int byte = (c & 63) * 2;
  return (uint32_t)((c >> 6) * 16384 + r * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15)));
}

constexpr int Q_STAGE = 32768;                 // one BF16 tile

// E4M3 and E2M1 tiles are staged in shared memory ([128][128] bytes per
// orientation with the 128-byte swizzle, or [128][64] bytes with the
// 64-byte swizzle) and written with two TMA stores; E2M3 (24-byte blocks)
// stores its blocks directly.
template <int FMT> struct QCfg {
  static constexpr bool STAGED = FMT == E4M3 || FMT == E2M1;
  static constexpr int ROW_BYTES = FMT == E4M3 ? 128 : 64;    // staged payload bytes per tile row
  static constexpr int OUT_BYTES = STAGED ? 128 * ROW_BYTES : 0;  // one orientation
  static constexpr int NST = STAGED ? 2 : 3;   // tiles in the load ring
  static constexpr int OFF_OUT = NST * Q_STAGE;
  static constexpr int OFF_SC = OFF_OUT + 2 * OUT_BYTES;
  static constexpr int SMEM = OFF_SC + 2048 + 4096 + 64 + 1024;
};

// Byte offset of (row r, byte b) in a staging tile of 128-byte rows with the
// 128-byte swizzle, or of 64-byte rows with the 64-byte swizzle, as the TMA
// store undoes it: the 16-byte chunk index is XORed with (r % 8), or with
// (r / 2) % 4.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t stage_off(int r, int b) {
  const int x = ROW_BYTES == 128 ? (r & 7) : ((r >> 1) & 3);
  return (uint32_t)(r * ROW_BYTES + ((((b >> 4) ^ x) << 4) | (b & 15)));
}

// GATHER: the token-permute form.  Every thread copies 8 of the tile's 2048
// 16-byte chunks from the routed rows' tokens (cp.async into the same
// swizzled layout the TMA boxes produce) and arrives on the stage's barrier
// when they land (expected arrivals: 256).
template <int FMT, bool HAD, bool ROW, bool COL, bool COLSUM, bool SR = false, bool GATHER = false>
__global__ void __launch_bounds__(256, 2)
quantize_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap rowmap,
                const __grid_constant__ CUtensorMap colmap, const QuantParams p) {
  using QC = QCfg<FMT>;
  constexpr int Q_NST = QC::NST;
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsm_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* out_row = sm + QC::OFF_OUT;                                    // staged payload tiles
  uint8_t* out_col = out_row + QC::OUT_BYTES;
  uint8_t* sc_all = sm + QC::OFF_SC;                                      // [2 parity][row, col][512]
  float* part_all = reinterpret_cast<float*>(sm + QC::OFF_SC + 2048);     // [2 parity][4][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + QC::OFF_SC + 2048 + 4096);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + Q_NST);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // gather: only the rows of the routed segments are produced
  const int64_t rows_out = (GATHER && p.offsets) ? min((int64_t)__ldg(p.offsets + p.G - 1), p.rows) : p.rows;
  const int64_t tiles_y = (rows_out + QT - 1) / QT;
  const int64_t per_batch = tiles_y * p.tiles_x;
  const int64_t total = per_batch * p.batch;
  const uint64_t budget = 2000000000ull;

  if (tid == 0) {
    for (int k = 0; k < Q_NST; k++) mbar_init(&full[k], GATHER ? 256 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // tile t -> (batch entry, row base, column base)
  auto coords = [&](int64_t t, int& b, int64_t& r0, int64_t& c0) {
    b = (int)(t / per_batch);
    const int64_t rem = t % per_batch;
    r0 = (rem / p.tiles_x) * QT;
    c0 = (rem % p.tiles_x) * QT;
  };
  auto issue = [&](int64_t t, int s) {  // thread 0: both 64-column boxes of tile t
    int b;
    int64_t r0, c0;
    coords(t, b, r0, c0);
    const int gy = (int)(b * p.rows + r0);
    mbar_arrive_expect_tx(&full[s], Q_STAGE);
    const uint64_t pol = l2_policy_evict_first();
    tma_load_2d(sm + s * Q_STAGE, &xmap, (int)c0, gy, &full[s], pol);
    tma_load_2d(sm + s * Q_STAGE + 16384, &xmap, (int)c0 + 64, gy, &full[s], pol);
  };
  // gather: thread tid copies chunk (tid % 16) of rows tid / 16 + 16 j,
  // j = 0..7.  The source rows of a tile are read one tile ahead of its
  // copies, so the index loads' latency hides behind the current tile.
  auto gather_rows = [&](int64_t t, int32_t (&tok)[8]) {
    int b;
    int64_t r0, c0;
    coords(t, b, r0, c0);
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int64_t gr = r0 + (tid >> 4) + 16 * j;
      tok[j] = gr < p.rows ? __ldg(p.src + gr) : -1;
    }
  };
  auto gather = [&](int64_t t, int s, const int32_t (&tok)[8]) {
    int b;
    int64_t r0, c0;
    coords(t, b, r0, c0);
    uint8_t* dst = sm + s * Q_STAGE;
    const int c = (tid & 15) * 8;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int r = (tid >> 4) + 16 * j;
      int64_t tk = tok[j];
      if (tk >= p.src_rows) {
        atomicOr(&g_quant_status, DEV_BAD_INDEX);
        tk = -1;
      }
      const bool ok = tk >= 0 && c0 + c < p.cols;
      cp_async16(smem_u32(dst + tile_off(r, c)), ok ? (const void*)(p.x + tk * p.ld + c0 + c) : (const void*)p.x,
                 ok ? 16u : 0u);
    }
    cp_async_arrive_noinc(&full[s]);
  };
  int32_t next_tok[8];
  if (GATHER) {
    for (int k = 0; k < Q_NST; k++) {
      if (blockIdx.x + (int64_t)k * gridDim.x < total) {
        gather_rows(blockIdx.x + (int64_t)k * gridDim.x, next_tok);
        gather(blockIdx.x + (int64_t)k * gridDim.x, k, next_tok);
      }
    }
  } else if (tid == 0) {
    for (int k = 0; k < Q_NST; k++)
      if (blockIdx.x + (int64_t)k * gridDim.x < total) issue(blockIdx.x + (int64_t)k * gridDim.x, k);
  }

  int it = 0;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x, it++) {
    const int s = it % Q_NST;
    if (!mbar_wait_bounded(&full[s], (uint32_t)((it / Q_NST) & 1), abort_flag, budget)) break;
    if (GATHER && t + Q_NST * (int64_t)gridDim.x < total) gather_rows(t + Q_NST * (int64_t)gridDim.x, next_tok);
    int b;
    int64_t r0, c0;
    coords(t, b, r0, c0);
    const int vrows = (int)((p.rows - r0) < QT ? (p.rows - r0) : QT);
    const int vcols = (int)((p.cols - c0) < QT ? (p.cols - c0) : QT);
    const uint8_t* tile = sm + s * Q_STAGE;
    if constexpr (QC::STAGED) {  // the previous tile's TMA stores have read the staging tiles
      if (tid == 0) bulk_wait_read();
      __syncthreads();
    }
    uint8_t* sc_row = sc_all + (it & 1) * 1024;
    uint8_t* sc_col = sc_row + 512;
    float* part = part_all + (it & 1) * 512;

    // ---- rowwise: blocks of 32 columns (every chunk slot gets written) ----
    if constexpr (ROW) {
      const int r = (warp & 3) * 32 + lane;
#pragma unroll 1
      for (int j = 0; j < 2; j++) {
        const int cb = (warp >> 2) * 2 + j;
        uint32_t sb = 0;
        if (r < vrows && cb * 32 < vcols) {
          uint32_t wv[16];
#pragma unroll
          for (int k = 0; k < 4; k++) {
            const uint4 q = *reinterpret_cast<const uint4*>(tile + tile_off(r, cb * 32 + 8 * k));
            wv[4 * k] = q.x; wv[4 * k + 1] = q.y; wv[4 * k + 2] = q.z; wv[4 * k + 3] = q.w;
          }
          const uint32_t m2 = amax_bf16_pairs<16>(wv);
          const uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16) << 16;
          float v[32];
#pragma unroll
          for (int i = 0; i < 16; i++) {
            v[2 * i] = bf16_bits_to_float(wv[i] & 0xFFFFu);
            v[2 * i + 1] = bf16_bits_to_float(wv[i] >> 16);
          }
          uint32_t w[8];
          // stochastic rounding: element index in the rowwise output grid [batch * rows, cols]
          sb = quantize32<FMT, HAD, SR>(v, amax, w, p.seed,
                                        (uint64_t)((int64_t)b * p.rows + r0 + r) * (uint64_t)p.cols +
                                            (uint64_t)(c0 + cb * 32), 0u);
          if constexpr (FMT == E4M3) {
            *reinterpret_cast<uint4*>(out_row + stage_off<128>(r, cb * 32)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(out_row + stage_off<128>(r, cb * 32 + 16)) = make_uint4(w[4], w[5], w[6], w[7]);
          } else if constexpr (FMT == E2M1) {
            *reinterpret_cast<uint4*>(out_row + stage_off<64>(r, cb * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            uint8_t* dst = p.row_data + (int64_t)b * p.row_batch_stride + (r0 + r) * p.row_ld +
                           (c0 + cb * 32) / 32 * BlockBytes<FMT>::value;
            store_block<FMT>(dst, w);
          }
        }
        sc_row[(r & 31) * 16 + (r >> 5) * 4 + cb] = (uint8_t)sb;
      }
    }

    // ---- columnwise: blocks of 32 rows, stored transposed ----
    if constexpr (COL) {
      const int cp = (warp & 1) * 32 + lane;  // column pair 0..63
      const int rb = warp >> 1;               // 32-row block 0..3
      const int c = 2 * cp;
      const bool valid = c < vcols && rb * 32 < vrows;
      uint32_t wv[32];
      if (valid) {
#pragma unroll
        for (int i = 0; i < 32; i++) wv[i] = *reinterpret_cast<const uint32_t*>(tile + tile_off(rb * 32 + i, c));
      }
      const uint32_t m2 = valid ? amax_bf16_pairs<32>(wv) : 0u;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int cc = c + h;
        uint32_t sb = 0;
        float sum = 0.f;
        if (valid) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; i++) {
            v[i] = bf16_bits_to_float(h ? (wv[i] >> 16) : (wv[i] & 0xFFFFu));
            if (COLSUM) sum += v[i];
          }
          const uint32_t amax = (h ? (m2 >> 16) : (m2 & 0xFFFFu)) << 16;
          uint32_t w[8];
          // stochastic rounding: element index in the columnwise output grid [batch * cols, rows]
          sb = quantize32<FMT, HAD, SR>(v, amax, w, p.seed,
                                        (uint64_t)((int64_t)b * p.cols + c0 + cc) * (uint64_t)p.rows +
                                            (uint64_t)(r0 + rb * 32), 1u);
          if constexpr (FMT == E4M3) {
            *reinterpret_cast<uint4*>(out_col + stage_off<128>(cc, rb * 32)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(out_col + stage_off<128>(cc, rb * 32 + 16)) = make_uint4(w[4], w[5], w[6], w[7]);
          } else if constexpr (FMT == E2M1) {
            *reinterpret_cast<uint4*>(out_col + stage_off<64>(cc, rb * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            uint8_t* dst = p.col_data + (int64_t)b * p.col_batch_stride + (c0 + cc) * p.col_ld +
                           (r0 + rb * 32) / 32 * BlockBytes<FMT>::value;
            store_block<FMT>(dst, w);
          }
        }
        if (COLSUM) part[rb * QT + cc] = sum;
        sc_col[(cc & 31) * 16 + (cc >> 5) * 4 + rb] = (uint8_t)sb;
      }
    }
    if constexpr (QC::STAGED) fence_proxy_async_smem();  // staging writes -> visible to the TMA store
    __syncthreads();  // stage s fully read; staging, chunks and partial sums complete

    if (tid == 0) {
      if constexpr (QC::STAGED) {
        // x in payload bytes: one per element (E4M3), one per two (E2M1)
        constexpr int SH = FMT == E4M3 ? 0 : 1;
        if constexpr (ROW) tma_store_2d(&rowmap, out_row, (int)(c0 >> SH), (int)(b * p.rows + r0));
        if constexpr (COL) tma_store_2d(&colmap, out_col, (int)(r0 >> SH), (int)(b * p.cols + c0));
        bulk_commit();
      }
      if (!GATHER && t + Q_NST * (int64_t)gridDim.x < total) issue(t + Q_NST * (int64_t)gridDim.x, s);
    }
    if (GATHER && t + Q_NST * (int64_t)gridDim.x < total) gather(t + Q_NST * (int64_t)gridDim.x, s, next_tok);
    if (tid < 32) {
      if constexpr (ROW) {
        const int64_t chunk = (r0 / 128) * ((p.cols / 32 + 3) / 4) + c0 / 128;
        reinterpret_cast<uint4*>(p.row_scale + (int64_t)b * p.row_scale_batch_stride + chunk * 512)[tid] =
            reinterpret_cast<const uint4*>(sc_row)[tid];
      }
    } else if (tid < 64) {
      if constexpr (COL) {
        const int64_t chunk = (c0 / 128) * ((p.rows / 32 + 3) / 4) + r0 / 128;
        reinterpret_cast<uint4*>(p.col_scale + (int64_t)b * p.col_scale_batch_stride + chunk * 512)[tid - 32] =
            reinterpret_cast<const uint4*>(sc_col)[tid - 32];
      }
    }
    if constexpr (COLSUM) {
      if (tid >= 128 && tid - 128 < vcols) {
        const int c = tid - 128;
        float sum = part[c];
        sum += part[QT + c];
        sum += part[2 * QT + c];
        sum += part[3 * QT + c];
        p.colsum_partials[(r0 / 128) * p.cols + c0 + c] = sum;
      }
    }
  }
  if (QC::STAGED && tid == 0) bulk_wait_all();  // this CTA's TMA stores have completed
  if (GATHER) cp_async_wait_all();              // no copy of this thread still in flight
  if (*abort_flag) {
    // a wait ran out: let every copy this CTA issued land before exiting
    if (tid == 0) {
      volatile int no_abort = 0;
      atomicOr(&g_quant_status, DEV_TIMEOUT);
      for (int k = 0; k < (GATHER ? 0 : Q_NST); k++) {
        const int64_t t = blockIdx.x + (int64_t)(it + k) * gridDim.x;
        if (t < total)
          mbar_wait_bounded(&full[(it + k) % Q_NST], (uint32_t)(((it + k) / Q_NST) & 1), &no_abort, budget);
      }
    }
    __syncthreads();
  }
}

// colsum[c] = sum over tile rows t (in order) of partials[t, c].
__global__ void colsum_reduce_kernel(const float* __restrict__ partials, int64_t tiles, int64_t cols,
                                     float* __restrict__ out) {
  int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  float s = 0.f;
  for (int64_t t = 0; t < tiles; t++) s += partials[t * cols + c];
  out[c] = s;
}

// ---------------------------------------------------------------------------
// Fixed scratch for the column-sum partials of the no-allocation entry point
// (mx_quantize_colsum_noalloc).  Every GPU that loads this library holds it
// until the process exits; all calls share it.
// ---------------------------------------------------------------------------

static __device__ __align__(256) float g_colsum_scratch[kNoAllocColsumFloats];

static std::mutex g_scratch_mu;
static float* g_scratch_ptr[64] = {};

// Device address of the scratch on the current device, looked up once per
// device (the array's host-side name is not a device address).
cudaError_t colsum_scratch(float** out, size_t* floats) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_colsum_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  *floats = kNoAllocColsumFloats;
  return cudaSuccess;
}

cudaError_t read_quant_status(unsigned* out) {
  return cudaMemcpyFromSymbol(out, g_quant_status, sizeof(unsigned));
}
cudaError_t reset_quant_status() {
  unsigned z = 0;
  return cudaMemcpyToSymbol(g_quant_status, &z, sizeof(unsigned));
}

cudaError_t launch_colsum_reduce(const float* partials, int64_t tiles, int64_t cols, float* out, cudaStream_t s) {
  colsum_reduce_kernel<<<(unsigned)((cols + 255) / 256), 256, 0, s>>>(partials, tiles, cols, out);
  return cudaGetLastError();
}

template <int FMT, bool HAD, bool ROW, bool COL, bool COLSUM, bool SR = false, bool GATHER = false>
static cudaError_t launch_q(const QuantLaunch& q, const QuantParams& p, cudaStream_t s) {
  auto kern = quantize_kernel<FMT, HAD, ROW, COL, COLSUM, SR, GATHER>;
  constexpr int smem = QCfg<FMT>::SMEM;
  {
    const cudaError_t e = ensure_smem_attr<quantize_kernel<FMT, HAD, ROW, COL, COLSUM, SR, GATHER>>(smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t tiles = (int64_t)p.tiles_x * ((p.rows + QT - 1) / QT) * p.batch;
  const int64_t cap = 2ll * q.num_sms;
  kern<<<(unsigned)(tiles < cap ? tiles : cap), 256, smem, s>>>(q.xmap, q.rowmap, q.colmap, p);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t dispatch_orient_gather(const QuantLaunch& q, const QuantParams& p, bool row, bool col,
                                          cudaStream_t s) {
  if (row && col) return launch_q<FMT, false, true, true, false, false, true>(q, p, s);
  if (row) return launch_q<FMT, false, true, false, false, false, true>(q, p, s);
  return launch_q<FMT, false, false, true, false, false, true>(q, p, s);
}

template <int FMT, bool HAD>
static cudaError_t dispatch_orient_sr(const QuantLaunch& q, const QuantParams& p, bool row, bool col,
                                      cudaStream_t s) {
  if (row && col) return launch_q<FMT, HAD, true, true, false, true>(q, p, s);
  if (row) return launch_q<FMT, HAD, true, false, false, true>(q, p, s);
  return launch_q<FMT, HAD, false, true, false, true>(q, p, s);
}

template <int FMT, bool HAD>
static cudaError_t dispatch_orient(const QuantLaunch& q, const QuantParams& p, bool row, bool col, bool colsum,
                                   cudaStream_t s) {
  if (colsum) {
    if (row && col) return launch_q<FMT, HAD, true, true, true>(q, p, s);
    if (col) return launch_q<FMT, HAD, false, true, true>(q, p, s);
    return cudaErrorInvalidValue;  // column sums come from the columnwise pass
  }
  if (row && col) return launch_q<FMT, HAD, true, true, false>(q, p, s);
  if (row) return launch_q<FMT, HAD, true, false, false>(q, p, s);
  return launch_q<FMT, HAD, false, true, false>(q, p, s);
}

cudaError_t launch_quantize(const QuantLaunch& q, cudaStream_t s) {
  QuantParams p;
  p.x = static_cast<const uint16_t*>(q.x);
  p.rows = q.rows; p.cols = q.cols; p.ld = q.ld; p.x_batch_stride = q.rows * q.ld;
  const int bb = q.fmt == E4M3 ? 32 : (q.fmt == E2M3 ? 24 : 16);
  p.row_data = q.row_data; p.row_scale = q.row_scale;
  p.row_ld = q.cols / 32 * bb;
  p.row_batch_stride = q.rows * p.row_ld;
  p.row_scale_batch_stride = q.row_data ? (int64_t)scale_bytes(q.rows, q.cols / 32) : 0;
  p.col_data = q.col_data; p.col_scale = q.col_scale;
  p.col_ld = q.rows / 32 * bb;
  p.col_batch_stride = q.cols * p.col_ld;
  p.col_scale_batch_stride = q.col_data ? (int64_t)scale_bytes(q.cols, q.rows / 32) : 0;
  p.colsum_partials = q.colsum_partials;
  p.tiles_x = (int)((q.cols + QT - 1) / QT);
  p.batch = (int)q.batch;
  p.seed = q.seed;
  p.src = q.src; p.src_rows = q.src_rows; p.offsets = q.offsets; p.G = q.G;
  const bool row = q.row_data != nullptr, col = q.col_data != nullptr, cs = q.colsum_partials != nullptr;
  cudaError_t e;
  if (q.src) {  // gather (token permute): no rotation, rounding variant or column sums
    switch (q.fmt) {
      case E4M3: return dispatch_orient_gather<E4M3>(q, p, row, col, s);
      case E2M3: return dispatch_orient_gather<E2M3>(q, p, row, col, s);
      case E2M1: return dispatch_orient_gather<E2M1>(q, p, row, col, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (q.stochastic) {  // E2M3 / E2M1 without column sums (checked by the caller)
    switch (q.fmt * 2 + (q.hadamard ? 1 : 0)) {
      case 2: return dispatch_orient_sr<E2M3, false>(q, p, row, col, s);
      case 3: return dispatch_orient_sr<E2M3, true>(q, p, row, col, s);
      case 4: return dispatch_orient_sr<E2M1, false>(q, p, row, col, s);
      case 5: return dispatch_orient_sr<E2M1, true>(q, p, row, col, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (q.fmt * 2 + (q.hadamard ? 1 : 0)) {
    case 0: e = dispatch_orient<E4M3, false>(q, p, row, col, cs, s); break;
    case 1: e = dispatch_orient<E4M3, true>(q, p, row, col, cs, s); break;
    case 2: e = dispatch_orient<E2M3, false>(q, p, row, col, cs, s); break;
    case 3: e = dispatch_orient<E2M3, true>(q, p, row, col, cs, s); break;
    case 4: e = dispatch_orient<E2M1, false>(q, p, row, col, cs, s); break;
    default: e = dispatch_orient<E2M1, true>(q, p, row, col, cs, s); break;
  }
  if (e != cudaSuccess || !cs) return e;
  int64_t tiles = (q.rows + QT - 1) / QT;
  colsum_reduce_kernel<<<(unsigned)((q.cols + 255) / 256), 256, 0, s>>>(q.colsum_partials, tiles, q.cols,
                                                                        q.colsum);
  return cudaGetLastError();
}

}  // namespace mx
