// Instantiations of the block-scaled GEMM for the dense MXFP6 MLP: FC1 with
// the bias + tanh-GELU epilogue that saves the BF16 pre-activation and packs
// the activation rowwise and columnwise (rotated), and FC2 dgrad with the
// dGELU epilogue that packs the pre-activation gradient and sums its columns
// (the bias gradient).  Primus PR #1064 "feat(mxfp6): MXFP6 (E2M3) Flux
// linears, a fused MLP, and the MLPerf recipe": fused-MLP commit (the packer
// takes the epilogue as a prologue in both directions, the pre-activation
// gradient is never assembled, the bias gradient comes back as a per-column
// sum) and the first commit (E2M3 with the Hadamard rotation in the packer).
#include "gemm_kernel.cuh"

namespace mx {

template <int BN, int EPI, int QF, bool QH>
static cudaError_t launch_dense_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                                    const CUtensorMap& to, cudaStream_t s, int num_sms) {
  auto kern = mx_gemm_kernel<BN, EPI, MODE_GROUPED, QF, QH>;
  constexpr int smem = KCfg<BN, EPI>::SMEM_BYTES;
  {
    const cudaError_t e = ensure_smem_attr<mx_gemm_kernel<BN, EPI, MODE_GROUPED, QF, QH>>(smem);
    if (e != cudaSuccess) return e;
  }
  int64_t grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads<BN, EPI>(), smem, s>>>(ta, tb, to, ta, tb, p);
  return cudaGetLastError();
}

template <int BN, int EPI>
static cudaError_t dispatch_q(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& to, cudaStream_t s, int num_sms) {
  if (p.q_fmt == E2M3 && p.q_had) return launch_dense_one<BN, EPI, E2M3, true>(p, ta, tb, to, s, num_sms);
  if (p.q_fmt == E2M3) return launch_dense_one<BN, EPI, E2M3, false>(p, ta, tb, to, s, num_sms);
  if (p.q_fmt == E4M3 && p.q_had) return launch_dense_one<BN, EPI, E4M3, true>(p, ta, tb, to, s, num_sms);
  if (p.q_fmt == E4M3) return launch_dense_one<BN, EPI, E4M3, false>(p, ta, tb, to, s, num_sms);
  return cudaErrorInvalidValue;
}

// bn = 256 where the output width allows (the 128x256 MMA, tensor-memory
// parking in the epilogue), else 128.
cudaError_t launch_gemm_dense(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& to, int bn, cudaStream_t s, int num_sms) {
  if (p.epi == EPI_GELU)
    return bn == 256 ? dispatch_q<256, EPI_GELU>(p, ta, tb, to, s, num_sms)
                     : dispatch_q<128, EPI_GELU>(p, ta, tb, to, s, num_sms);
  if (p.epi == EPI_DGELU)
    return bn == 256 ? dispatch_q<256, EPI_DGELU>(p, ta, tb, to, s, num_sms)
                     : dispatch_q<128, EPI_DGELU>(p, ta, tb, to, s, num_sms);
  return cudaErrorInvalidValue;
}

cudaError_t read_dense_status(unsigned* out) {
  return cudaMemcpyFromSymbol(out, g_gemm_status, sizeof(unsigned));
}
cudaError_t reset_dense_status() {
  unsigned z = 0;
  return cudaMemcpyToSymbol(g_gemm_status, &z, sizeof(unsigned));
}

}  // namespace mx
