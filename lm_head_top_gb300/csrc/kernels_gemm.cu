// Instantiations and launchers of the tcgen05 GEMM kernel for the four
// contractions of the fused KL loss (forward logsumexp, backward recompute,
// dH = G W, dW = G^T H).
#include "kdkl_internal.h"
#include "tc_gemm.cuh"

namespace kdkl {

namespace {

constexpr int kMaxDevices = 64;

template <int EPI, bool A_MN, bool B_MN>
cudaError_t launch_one(const char* name, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const GemmShape& sh, const EpiParams& ep, int* status, int grid,
                       cudaStream_t stream) {
  auto kern = tc_gemm_kernel<EPI, A_MN, B_MN>;
  static bool attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_kernel(name, kern, dim3(grid), dim3(GEMM_THREADS), (size_t)GEMM_SMEM_BYTES,
                       stream, tmA, tmB, sh, ep, status);
}

}  // namespace

cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const GemmShape& sh, const EpiParams& ep, int* status, int grid,
                        cudaStream_t stream) {
  switch (kind) {
    case GEMM_FWD_LSE:
      return launch_one<EPI_LSE, false, false>("fwd_lse_gemm", tmA, tmB, sh, ep, status, grid,
                                               stream);
    case GEMM_BWD_GRAD:
      return launch_one<EPI_GRAD, false, false>("bwd_grad_gemm", tmA, tmB, sh, ep, status, grid,
                                                stream);
    case GEMM_DH:
      return launch_one<EPI_STORE, false, true>("dH_gemm", tmA, tmB, sh, ep, status, grid, stream);
    case GEMM_DW:
      return launch_one<EPI_STORE, true, true>("dW_gemm", tmA, tmB, sh, ep, status, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kdkl
