// Instantiations of the grouped block-scaled GEMM for the expert MLP: the
// plain BF16-out grouped GEMM, the ragged-K wgrad, and the SwiGLU forward /
// dSwiGLU backward fused epilogues (torchao PR #5 "MXFP8 cudnn-fe Swiglu fused
// Grouped MLP fwd/bwd and wgrad group gemm", correctness-first kernels
// commit).  The kernel itself is in gemm_kernel.cuh.
#include "gemm_kernel.cuh"

namespace mx {

template <int BN, int EPI, int MODE, bool EXT = false>
static cudaError_t launch_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& to, cudaStream_t s, int num_sms) {
  auto kern = mx_gemm_kernel<BN, EPI, MODE, E4M3, false, EXT>;
  constexpr int smem = KCfg<BN, EPI>::SMEM_BYTES;
  {
    const cudaError_t e = ensure_smem_attr<mx_gemm_kernel<BN, EPI, MODE, E4M3, false, EXT>>(smem);
    if (e != cudaSuccess) return e;
  }
  int64_t grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads<BN, EPI>(), smem, s>>>(ta, tb, to, ta, tb, p);
  return cudaGetLastError();
}

// The fused SwiGLU / dSwiGLU epilogues on CTA pairs (256-row tiles, two SMs
// per tile): clusters of two CTAs, one pair per two SMs.
template <int EPI, int MODE, bool EXT>
static cudaError_t launch_pair_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                                   const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& to,
                                   cudaStream_t s, int num_sms) {
  constexpr int smem = KCfg<256, EPI, false, true>::SMEM_BYTES;
  {
    const cudaError_t e = ensure_smem_attr<mx_gemm_kernel<256, EPI, MODE, E4M3, false, EXT, false, true>>(smem);
    if (e != cudaSuccess) return e;
  }
  int64_t pairs = p.num_tiles < num_sms / 2 ? p.num_tiles : num_sms / 2;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads<256, EPI, true>(), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<256, EPI, MODE, E4M3, false, EXT, false, true>, ta, tb, to, tsa,
                            tsb, p);
}

cudaError_t launch_gemm_pair_fused(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                                   const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& to,
                                   cudaStream_t s, int num_sms) {
  const bool ext = p.tap != nullptr || p.probs != nullptr;
  if (p.mode == MODE_WGRAD) {
    if (p.epi == EPI_F32) return launch_pair_one<EPI_F32, MODE_WGRAD, false>(p, ta, tb, tsa, tsb, to, s, num_sms);
    if (p.epi == EPI_BF16) return launch_pair_one<EPI_BF16, MODE_WGRAD, false>(p, ta, tb, tsa, tsb, to, s, num_sms);
    return cudaErrorInvalidValue;
  }
  if (p.epi == EPI_SWIGLU) return launch_pair_one<EPI_SWIGLU, MODE_GROUPED, false>(p, ta, tb, tsa, tsb, to, s, num_sms);
  if (p.epi == EPI_DSWIGLU)
    return ext ? launch_pair_one<EPI_DSWIGLU, MODE_GROUPED, true>(p, ta, tb, tsa, tsb, to, s, num_sms)
               : launch_pair_one<EPI_DSWIGLU, MODE_GROUPED, false>(p, ta, tb, tsa, tsb, to, s, num_sms);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                        int bn, cudaStream_t s, int num_sms) {
  if (p.f4) return launch_gemm_f4(p, ta, tb, to, bn, s, num_sms);
  if (p.epi == EPI_SWIGLU) return launch_one<256, EPI_SWIGLU, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
  if (p.epi == EPI_DSWIGLU) {  // 256-column tiles where F allows (bn), else 128
    const bool ext = p.tap != nullptr || p.probs != nullptr;
    if (bn == 256)
      return ext ? launch_one<256, EPI_DSWIGLU, MODE_GROUPED, true>(p, ta, tb, to, s, num_sms)
                 : launch_one<256, EPI_DSWIGLU, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
    return ext ? launch_one<128, EPI_DSWIGLU, MODE_GROUPED, true>(p, ta, tb, to, s, num_sms)
               : launch_one<128, EPI_DSWIGLU, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
  }
  if (p.epi == EPI_F32) {
    if (p.mode != MODE_WGRAD) return cudaErrorInvalidValue;
    if (bn == 128) return launch_one<128, EPI_F32, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
    return launch_one<256, EPI_F32, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
  }
  if (p.mode == MODE_WGRAD) {
    if (bn == 128) return launch_one<128, EPI_BF16, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
    return launch_one<256, EPI_BF16, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
  }
  if (bn == 128) return launch_one<128, EPI_BF16, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
  return launch_one<256, EPI_BF16, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
}

__global__ void dprobs_reduce_kernel(const float* __restrict__ part, int64_t R, int64_t ld,
                                     const int32_t* __restrict__ offsets, int G, float* __restrict__ out) {
  const int64_t rows = offsets ? (int64_t)__ldg(offsets + G - 1) : R;
  for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < rows && r < R;
       r += (int64_t)gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int64_t k = 0; k < ld; k++) s += part[r * ld + k];
    out[r] = s;
  }
}

cudaError_t launch_dprobs_reduce(const float* part, int64_t R, int64_t ld, const int32_t* offsets, int G,
                                 float* dprobs, cudaStream_t s) {
  const int64_t blocks = (R + 255) / 256;
  dprobs_reduce_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(part, R, ld, offsets, G, dprobs);
  return cudaGetLastError();
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
