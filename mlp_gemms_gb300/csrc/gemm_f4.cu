// Instantiations of the block-scaled GEMM for packed E2M1 (MXFP4) operands
// on tcgen05 .kind::mxf4: the BF16-out grouped / dense GEMM, the ragged-K
// wgrad and the fp32 main-grad wgrad.  ROCm Primus guide "MXFP4 training for
// Flux models" (the linears run on MXFP4 operands, E2M1 elements with one
// E8M0 scale per 32); the operands are the quantizer's E2M1 payloads as they
// are, two elements per byte, which is the layout .kind::mxf4 reads.  The
// kernel itself is in gemm_kernel.cuh.
#include "gemm_kernel.cuh"

namespace mx {

template <int BN, int EPI, int MODE>
static cudaError_t launch_f4_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                                 const CUtensorMap& to, cudaStream_t s, int num_sms) {
  auto kern = mx_gemm_kernel<BN, EPI, MODE, E4M3, false, false, true>;
  constexpr int smem = KCfg<BN, EPI, true>::SMEM_BYTES;
  {
    const cudaError_t e = ensure_smem_attr<mx_gemm_kernel<BN, EPI, MODE, E4M3, false, false, true>>(smem);
    if (e != cudaSuccess) return e;
  }
  int64_t grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads<BN, EPI>(), smem, s>>>(ta, tb, to, ta, tb, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_f4(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                           int bn, cudaStream_t s, int num_sms) {
  if (p.epi == EPI_F32) {
    if (p.mode != MODE_WGRAD) return cudaErrorInvalidValue;
    if (bn == 128) return launch_f4_one<128, EPI_F32, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
    return launch_f4_one<256, EPI_F32, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
  }
  if (p.epi != EPI_BF16) return cudaErrorInvalidValue;
  if (p.mode == MODE_WGRAD) {
    if (bn == 128) return launch_f4_one<128, EPI_BF16, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
    return launch_f4_one<256, EPI_BF16, MODE_WGRAD>(p, ta, tb, to, s, num_sms);
  }
  if (bn == 128) return launch_f4_one<128, EPI_BF16, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
  return launch_f4_one<256, EPI_BF16, MODE_GROUPED>(p, ta, tb, to, s, num_sms);
}

cudaError_t read_f4_status(unsigned* out) {
  return cudaMemcpyFromSymbol(out, g_gemm_status, sizeof(unsigned));
}
cudaError_t reset_f4_status() {
  unsigned z = 0;
  return cudaMemcpyToSymbol(g_gemm_status, &z, sizeof(unsigned));
}

}  // namespace mx
