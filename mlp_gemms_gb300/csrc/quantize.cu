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
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

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
};

constexpr int QT = 128;          // tile edge
constexpr int QPAD = QT + 8;     // smem row pitch in bf16 (272 bytes)

// NaN-propagating amax of 32 BF16 values given as 16 packed pairs: integer
// max of |bits| (a NaN pattern is larger than every other pattern).
__device__ __forceinline__ uint32_t amax_bf16_pairs(const uint32_t* w, int n) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < n; i++) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  return m;
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

// Quantize 32 fp32 values (rotating first if HAD) and return the scale byte.
template <int FMT, bool HAD>
__device__ __forceinline__ uint32_t quantize32(float (&v)[32], uint32_t amax_bits_prerot, uint32_t (&w)[8]) {
  uint32_t amax_bits = amax_bits_prerot;
  if constexpr (HAD) {
    hadamard32(v);
    amax_bits = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  }
  uint32_t sb = rceil_scale_byte<FMT>(amax_bits);
  quantize_block_words<FMT>(v, sb, w);
  return sb;
}

template <int FMT, bool HAD, bool ROW, bool COL, bool COLSUM>
__global__ void __launch_bounds__(256) quantize_kernel(const QuantParams p) {
  __shared__ __align__(16) uint16_t tile[QT * QPAD];
  __shared__ __align__(16) uint8_t sc_row[512];
  __shared__ __align__(16) uint8_t sc_col[512];
  __shared__ float part[4][QT];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.y;
  const int tx = blockIdx.x % p.tiles_x, ty = blockIdx.x / p.tiles_x;
  const int64_t r0 = (int64_t)ty * QT, c0 = (int64_t)tx * QT;
  const int vrows = (int)((p.rows - r0) < QT ? (p.rows - r0) : QT);
  const int vcols = (int)((p.cols - c0) < QT ? (p.cols - c0) : QT);
  const uint16_t* xb = p.x + (int64_t)b * p.x_batch_stride;

  // ---- stage the tile: 16 threads cover one 256-byte row ----
  {
    uint4 v[8];
    const int chunk = tid & 15;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      int r = i * 16 + (tid >> 4);
      if (r < vrows && chunk * 8 < vcols) {
        const uint4* src = reinterpret_cast<const uint4*>(xb + (r0 + r) * p.ld + c0 + chunk * 8);
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w) : "l"(src));
      }
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
      int r = i * 16 + (tid >> 4);
      if (r < vrows && chunk * 8 < vcols) *reinterpret_cast<uint4*>(&tile[r * QPAD + chunk * 8]) = v[i];
    }
    for (int i = tid; i < 512 / 4; i += 256) {
      reinterpret_cast<uint32_t*>(sc_row)[i] = 0u;
      reinterpret_cast<uint32_t*>(sc_col)[i] = 0u;
    }
    if (COLSUM) for (int i = tid; i < 4 * QT; i += 256) (&part[0][0])[i] = 0.f;
  }
  __syncthreads();

  // ---- rowwise: blocks of 32 columns ----
  if constexpr (ROW) {
    const int r = (warp & 3) * 32 + lane;
#pragma unroll 1
    for (int j = 0; j < 2; j++) {
      const int cb = (warp >> 2) * 2 + j;
      if (r < vrows && cb * 32 < vcols) {
        uint32_t wv[16];
        const uint4* s = reinterpret_cast<const uint4*>(&tile[r * QPAD + cb * 32]);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          uint4 q = s[i];
          wv[4 * i] = q.x; wv[4 * i + 1] = q.y; wv[4 * i + 2] = q.z; wv[4 * i + 3] = q.w;
        }
        uint32_t m2 = amax_bf16_pairs(wv, 16);
        uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16) << 16;
        float v[32];
#pragma unroll
        for (int i = 0; i < 16; i++) {
          v[2 * i] = bf16_bits_to_float(wv[i] & 0xFFFFu);
          v[2 * i + 1] = bf16_bits_to_float(wv[i] >> 16);
        }
        uint32_t w[8];
        uint32_t sb = quantize32<FMT, HAD>(v, amax, w);
        uint8_t* dst = p.row_data + (int64_t)b * p.row_batch_stride + (r0 + r) * p.row_ld +
                       (c0 + cb * 32) / 32 * BlockBytes<FMT>::value;
        store_block<FMT>(dst, w);
        sc_row[(r & 31) * 16 + (r >> 5) * 4 + cb] = (uint8_t)sb;
      }
    }
  }

  // ---- columnwise: blocks of 32 rows, stored transposed ----
  if constexpr (COL) {
    const int cp = (warp & 1) * 32 + lane;  // column pair 0..63
    const int rb = warp >> 1;               // 32-row block 0..3
    const int c = 2 * cp;
    if (c < vcols && rb * 32 < vrows) {
      uint32_t wv[32];
#pragma unroll
      for (int i = 0; i < 32; i++) wv[i] = *reinterpret_cast<const uint32_t*>(&tile[(rb * 32 + i) * QPAD + c]);
      uint32_t m2 = amax_bf16_pairs(wv, 32);
#pragma unroll
      for (int h = 0; h < 2; h++) {
        float v[32];
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i++) {
          v[i] = bf16_bits_to_float(h ? (wv[i] >> 16) : (wv[i] & 0xFFFFu));
          if (COLSUM) sum += v[i];
        }
        if (COLSUM) part[rb][c + h] = sum;
        uint32_t amax = (h ? (m2 >> 16) : (m2 & 0xFFFFu)) << 16;
        uint32_t w[8];
        uint32_t sb = quantize32<FMT, HAD>(v, amax, w);
        const int cc = c + h;
        uint8_t* dst = p.col_data + (int64_t)b * p.col_batch_stride + (c0 + cc) * p.col_ld +
                       (r0 + rb * 32) / 32 * BlockBytes<FMT>::value;
        store_block<FMT>(dst, w);
        sc_col[(cc & 31) * 16 + (cc >> 5) * 4 + rb] = (uint8_t)sb;
      }
    }
  }
  __syncthreads();

  // ---- scale chunks (one 512-byte chunk per orientation) and column sums ----
  if (tid < 32) {
    if constexpr (ROW) {
      int64_t sc_cols = p.cols / 32;
      int64_t chunk = (r0 / 128) * ((sc_cols + 3) / 4) + c0 / 128;
      uint4* dst = reinterpret_cast<uint4*>(p.row_scale + (int64_t)b * p.row_scale_batch_stride + chunk * 512);
      dst[tid] = reinterpret_cast<const uint4*>(sc_row)[tid];
    }
  } else if (tid < 64) {
    if constexpr (COL) {
      int64_t sc_cols = p.rows / 32;
      int64_t chunk = (c0 / 128) * ((sc_cols + 3) / 4) + r0 / 128;
      uint4* dst = reinterpret_cast<uint4*>(p.col_scale + (int64_t)b * p.col_scale_batch_stride + chunk * 512);
      dst[tid - 32] = reinterpret_cast<const uint4*>(sc_col)[tid - 32];
    }
  }
  if constexpr (COLSUM) {
    if (tid < QT && tid < vcols) {
      float s = part[0][tid];
      s += part[1][tid];
      s += part[2][tid];
      s += part[3][tid];
      p.colsum_partials[(r0 / 128) * p.cols + c0 + tid] = s;
    }
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

cudaError_t launch_colsum_reduce(const float* partials, int64_t tiles, int64_t cols, float* out, cudaStream_t s) {
  colsum_reduce_kernel<<<(unsigned)((cols + 255) / 256), 256, 0, s>>>(partials, tiles, cols, out);
  return cudaGetLastError();
}

template <int FMT, bool HAD, bool ROW, bool COL, bool COLSUM>
static cudaError_t launch_q(const QuantParams& p, int batch, cudaStream_t s) {
  int64_t tiles = (int64_t)p.tiles_x * ((p.rows + QT - 1) / QT);
  dim3 grid((unsigned)tiles, (unsigned)batch);
  quantize_kernel<FMT, HAD, ROW, COL, COLSUM><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

template <int FMT, bool HAD>
static cudaError_t dispatch_orient(const QuantParams& p, int batch, bool row, bool col, bool colsum,
                                   cudaStream_t s) {
  if (colsum) {
    if (row && col) return launch_q<FMT, HAD, true, true, true>(p, batch, s);
    if (col) return launch_q<FMT, HAD, false, true, true>(p, batch, s);
    return cudaErrorInvalidValue;  // column sums come from the columnwise pass
  }
  if (row && col) return launch_q<FMT, HAD, true, true, false>(p, batch, s);
  if (row) return launch_q<FMT, HAD, true, false, false>(p, batch, s);
  return launch_q<FMT, HAD, false, true, false>(p, batch, s);
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
  const bool row = q.row_data != nullptr, col = q.col_data != nullptr, cs = q.colsum_partials != nullptr;
  cudaError_t e;
  switch (q.fmt * 2 + (q.hadamard ? 1 : 0)) {
    case 0: e = dispatch_orient<E4M3, false>(p, q.batch, row, col, cs, s); break;
    case 1: e = dispatch_orient<E4M3, true>(p, q.batch, row, col, cs, s); break;
    case 2: e = dispatch_orient<E2M3, false>(p, q.batch, row, col, cs, s); break;
    case 3: e = dispatch_orient<E2M3, true>(p, q.batch, row, col, cs, s); break;
    case 4: e = dispatch_orient<E2M1, false>(p, q.batch, row, col, cs, s); break;
    default: e = dispatch_orient<E2M1, true>(p, q.batch, row, col, cs, s); break;
  }
  if (e != cudaSuccess || !cs) return e;
  int64_t tiles = (q.rows + QT - 1) / QT;
  colsum_reduce_kernel<<<(unsigned)((q.cols + 255) / 256), 256, 0, s>>>(q.colsum_partials, tiles, q.cols,
                                                                        q.colsum);
  return cudaGetLastError();
}

}  // namespace mx
