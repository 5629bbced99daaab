// Token permute support for the expert MLP: the routing index (top-k expert
// ids -> 128- (or 256-) row padded expert segments, the source token of every routed
// row and the routed row of every (token, choice)) and the un-permute (the
// weighted sum of a token's routed rows).  Primus PR #1247 "Qwen3-30B-A3B
// FP8 on MI355X to 40k tokens/s/GPU", DeepEP permute section: the permute
// hands the grouped MLP its tokens already quantized, and the un-permute's
// backward hands back the output gradient the same way.  The quantizing
// gather itself is the quantizer kernel's gather form (quantize.cu).
//
// Order of the routed rows: experts ascending; within an expert, (token,
// choice) ascending; each segment padded with empty rows (source -1) to a
// multiple of 128 (256 for the CTA-pair GEMM).  Built as a stable counting sort with no floating point
// and no order-dependent atomics, so the index is deterministic.
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

static __device__ unsigned g_perm_status = 0;

constexpr int ROUTE_CHUNK = 1024;  // (token, choice) entries per counting chunk

// Pass 1: per-chunk expert histograms, expert-major: counts[e][chunk].
__global__ void route_count_kernel(const int32_t* __restrict__ topk, int64_t n, int G, int nchunks,
                                   int32_t* __restrict__ counts) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < G; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t b0 = (int64_t)blockIdx.x * ROUTE_CHUNK;
  const int64_t b1 = b0 + ROUTE_CHUNK < n ? b0 + ROUTE_CHUNK : n;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
    const int e = __ldg(topk + i);
    if (e >= 0 && e < G) atomicAdd(&hist[e], 1);
    else atomicOr(&g_perm_status, DEV_BAD_INDEX);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) counts[(int64_t)e * nchunks + blockIdx.x] = hist[e];
}

// Pass 2 (one block of 1024 threads): per expert, the chunk counts become
// absolute first rows of each chunk's entries (a warp scans an expert's
// chunks 256 at a time, 8 per lane, with a shuffle scan across lanes);
// padded segment ends go to offsets; padding rows and the rows past the
// last segment get source -1.
__global__ void route_scan_kernel(int32_t* __restrict__ counts, int nchunks, int G, int32_t* __restrict__ offsets,
                                  int32_t* __restrict__ src, int64_t R_cap, int32_t pad) {
  __shared__ int32_t tot[1024];
  __shared__ int32_t first[1024];
  __shared__ int32_t end[1024];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int e = warp; e < G; e += nwarps) {
    int32_t* ce = counts + (int64_t)e * nchunks;
    int32_t carry = 0;
    for (int base = 0; base < nchunks; base += 256) {
      int32_t v[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const int c = base + lane * 8 + j;
        v[j] = c < nchunks ? ce[c] : 0;
      }
      int32_t run = 0;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const int32_t t = v[j];
        v[j] = run;
        run += t;
      }
      int32_t incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      const int32_t excl = incl - run;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const int c = base + lane * 8 + j;
        if (c < nchunks) ce[c] = carry + excl + v[j];
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) tot[e] = carry;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int e = 0; e < G; e++) {
      const int32_t padded = (tot[e] + pad - 1) / pad * pad;
      first[e] = acc;
      acc += padded;
      end[e] = acc;
      offsets[e] = acc;
    }
  }
  __syncthreads();
  for (int64_t idx = threadIdx.x; idx < (int64_t)G * nchunks; idx += blockDim.x)
    counts[idx] += first[idx / nchunks];
  for (int e = warp; e < G; e += nwarps)
    for (int32_t r = first[e] + tot[e] + lane; r < end[e]; r += 32) src[r] = -1;
  for (int64_t r = (int64_t)end[G - 1] + threadIdx.x; r < R_cap; r += blockDim.x) src[r] = -1;
}

// Pass 3: one warp per chunk walks its entries in order, 32 at a time
// (all of the chunk's expert ids loaded first); lanes routed to the same
// expert take consecutive rows in lane order.
__global__ void route_scatter_kernel(const int32_t* __restrict__ topk, int64_t n, int k, int G, int nchunks,
                                     const int32_t* __restrict__ counts, int32_t* __restrict__ src,
                                     int32_t* __restrict__ row_of) {
  extern __shared__ int32_t next[];
  const int lane = threadIdx.x;
  for (int e = lane; e < G; e += 32) next[e] = counts[(int64_t)e * nchunks + blockIdx.x];
  const int64_t b0 = (int64_t)blockIdx.x * ROUTE_CHUNK;
  const int64_t b1 = b0 + ROUTE_CHUNK < n ? b0 + ROUTE_CHUNK : n;
  int ev[ROUTE_CHUNK / 32];
#pragma unroll
  for (int it = 0; it < ROUTE_CHUNK / 32; it++) {
    const int64_t i = b0 + it * 32 + lane;
    ev[it] = i < b1 ? __ldg(topk + i) : -1;
  }
  __syncwarp();
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < ROUTE_CHUNK / 32; it++) {
    const int64_t i = b0 + it * 32 + lane;
    const bool in = i < b1;
    const int e = ev[it];
    const bool ok = in && e >= 0 && e < G;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, ok ? e : -1) & __ballot_sync(0xFFFFFFFFu, ok);
    int32_t pos = -1;
    if (ok) {
      pos = next[e] + __popc(peers & below);
      src[pos] = (int32_t)(i / k);
    }
    if (in) row_of[i] = pos;
    __syncwarp();
    if (ok && (peers & below) == 0) next[e] += __popc(peers);
    __syncwarp();
  }
}

cudaError_t launch_route_index(const int32_t* topk, int64_t T, int k, int G, int32_t* offsets, int32_t* src,
                               int64_t R_cap, int32_t* row_of, int32_t* counts, int32_t pad, cudaStream_t s) {
  const int64_t n = T * k;
  const int nchunks = (int)((n + ROUTE_CHUNK - 1) / ROUTE_CHUNK);
  const size_t hist = (size_t)G * sizeof(int32_t);
  if (nchunks > 0) {
    route_count_kernel<<<nchunks, 256, hist, s>>>(topk, n, G, nchunks, counts);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  route_scan_kernel<<<1, 1024, 0, s>>>(counts, nchunks, G, offsets, src, R_cap, pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || nchunks == 0) return e;
  route_scatter_kernel<<<nchunks, 32, hist, s>>>(topk, n, k, G, nchunks, counts, src, row_of);
  return cudaGetLastError();
}

// out[t, :] = sum over j of w[t, j] * in[row_of[t, j], :] (w = 1 without
// weights; choices with row -1 skipped), accumulated in fp32 in choice
// order, one rounding to BF16.  Each thread owns 8 columns (16 bytes).
__global__ void unpermute_kernel(const uint16_t* __restrict__ in, int64_t R, int64_t D,
                                 const int32_t* __restrict__ row_of, const float* __restrict__ w, int64_t T, int k,
                                 uint16_t* __restrict__ out) {
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    for (int64_t c = (int64_t)threadIdx.x * 8; c < D; c += (int64_t)blockDim.x * 8) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; i++) acc[i] = 0.f;
      for (int j = 0; j < k; j++) {
        const int32_t r = __ldg(row_of + t * k + j);
        if (r < 0) continue;
        if (r >= R) {
          atomicOr(&g_perm_status, DEV_BAD_INDEX);
          continue;
        }
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(in + (int64_t)r * D + c));
        const uint32_t h[4] = {q.x, q.y, q.z, q.w};
        if (w != nullptr) {
          const float wj = __ldg(w + t * k + j);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            acc[2 * i] = fmaf(wj, bf16_bits_to_float(h[i] & 0xFFFFu), acc[2 * i]);
            acc[2 * i + 1] = fmaf(wj, bf16_bits_to_float(h[i] >> 16), acc[2 * i + 1]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; i++) {
            acc[2 * i] += bf16_bits_to_float(h[i] & 0xFFFFu);
            acc[2 * i + 1] += bf16_bits_to_float(h[i] >> 16);
          }
        }
      }
      uint4 o;
      o.x = float2_to_bf16x2(acc[0], acc[1]);
      o.y = float2_to_bf16x2(acc[2], acc[3]);
      o.z = float2_to_bf16x2(acc[4], acc[5]);
      o.w = float2_to_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(out + t * D + c) = o;
    }
  }
}

cudaError_t launch_unpermute(const uint16_t* in, int64_t R, int64_t D, const int32_t* row_of, const float* w,
                             int64_t T, int k, uint16_t* out, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int threads = D >= 2048 ? 256 : (int)((D / 8 + 31) / 32 * 32);
  const int64_t cap = (int64_t)num_sms * 8;
  unpermute_kernel<<<(unsigned)(T < cap ? T : cap), threads, 0, s>>>(in, R, D, row_of, w, T, k, out);
  return cudaGetLastError();
}

cudaError_t read_perm_status(unsigned* out) {
  return cudaMemcpyFromSymbol(out, g_perm_status, sizeof(unsigned));
}
cudaError_t reset_perm_status() {
  unsigned z = 0;
  return cudaMemcpyToSymbol(g_perm_status, &z, sizeof(unsigned));
}

}  // namespace mx
