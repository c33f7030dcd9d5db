// Instantiations and launchers of the tcgen05 GEMM kernel for the four
// contractions of the fused KL loss (forward logsumexp, backward recompute,
// dH = G W, dW = G^T H).
#include <atomic>

#include "kdkl_internal.h"
#include "tc_gemm.cuh"

namespace kdkl {

namespace {

constexpr int kMaxDevices = 64;

template <int EPI, bool A_MN, bool B_MN, int BN, bool PAIR, bool DUAL>
cudaError_t launch_one(const char* name, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const CUtensorMap& tmA1, const CUtensorMap& tmB1, const GemmShape& sh,
                       const GemmShape& sh1, const EpiParams& ep, const EpiParams& ep1,
                       int* status, int grid, cudaStream_t stream) {
  auto kern = tc_gemm_kernel<EPI, A_MN, B_MN, BN, PAIR, DUAL>;
  constexpr int smem = TileCfg<BN, PAIR>::SMEM_BYTES;
  // Per device and instantiation; concurrent first calls may both set the
  // attribute, which is harmless (same value).
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  if (PAIR)
    return launch_kernel_cluster(name, kern, dim3(grid), dim3(GEMM_THREADS), (size_t)smem, stream,
                                 2u, tmA, tmB, tmA1, tmB1, sh, sh1, ep, ep1, status);
  return launch_kernel(name, kern, dim3(grid), dim3(GEMM_THREADS), (size_t)smem, stream, tmA,
                       tmB, tmA1, tmB1, sh, sh1, ep, ep1, status);
}

// One job per launch: the second job's parameters repeat the first's and are
// not read.
template <int EPI, bool A_MN, bool B_MN, int BN>
cudaError_t launch_pick(bool pair, const char* name, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const GemmShape& sh, const EpiParams& ep, int* status, int grid,
                        cudaStream_t stream) {
  if (pair)
    return launch_one<EPI, A_MN, B_MN, BN, true, false>(name, tmA, tmB, tmA, tmB, sh, sh, ep, ep,
                                                        status, grid, stream);
  return launch_one<EPI, A_MN, B_MN, BN, false, false>(name, tmA, tmB, tmA, tmB, sh, sh, ep, ep,
                                                       status, grid, stream);
}

}  // namespace

int pair_max_active_clusters() {
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int known = cached[dev].load(std::memory_order_acquire);
  if (known > 0) return known;
  // Every pair instantiation has the same block size and shared memory, so one
  // of them stands for all.
  auto kern = tc_gemm_kernel<EPI_LSE, false, false, LOGIT_BN, true, false>;
  constexpr int smem = TileCfg<LOGIT_BN, true>::SMEM_BYTES;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(GEMM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  cached[dev].store(n, std::memory_order_release);
  return n;
}

cudaError_t launch_gemm(GemmKind kind, int bn, bool pair, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const GemmShape& sh, const EpiParams& ep,
                        int* status, int grid, cudaStream_t stream) {
  if (pair && (grid % 2) != 0) return cudaErrorInvalidValue;
  switch (kind) {
    case GEMM_FWD_LSE:
      if (bn != LOGIT_BN) break;
      return launch_pick<EPI_LSE, false, false, LOGIT_BN>(pair, "fwd_lse_gemm", tmA, tmB, sh, ep,
                                                          status, grid, stream);
    case GEMM_BWD_GRAD:
      if (bn != LOGIT_BN) break;
      return launch_pick<EPI_GRAD, false, false, LOGIT_BN>(pair, "bwd_grad_gemm", tmA, tmB, sh,
                                                           ep, status, grid, stream);
    case GEMM_FWD_LSE_MIX:
      if (bn != LOGIT_BN) break;
      return launch_pick<EPI_LSE_MIX, false, false, LOGIT_BN>(pair, "fwd_lse_mix_gemm", tmA, tmB,
                                                              sh, ep, status, grid, stream);
    case GEMM_BWD_GRAD_MIX:
      if (bn != LOGIT_BN) break;
      return launch_pick<EPI_GRAD_MIX, false, false, LOGIT_BN>(pair, "bwd_grad_mix_gemm", tmA,
                                                               tmB, sh, ep, status, grid, stream);
    case GEMM_TOPK:
      if (bn != LOGIT_BN) break;
      return launch_pick<EPI_TOPK, false, false, LOGIT_BN>(pair, "topk_gemm", tmA, tmB, sh, ep,
                                                           status, grid, stream);
    case GEMM_DH:
      if (bn != 256) break;
      return launch_pick<EPI_STORE, false, true, 256>(pair, "dH_gemm", tmA, tmB, sh, ep, status,
                                                      grid, stream);
    case GEMM_DW:
      if (bn != 256) break;
      return launch_pick<EPI_STORE, true, true, 256>(pair, "dW_gemm", tmA, tmB, sh, ep, status,
                                                     grid, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_dw_dh(bool pair, bool dh_first, const CUtensorMap& tmG_MN,
                              const CUtensorMap& tmH_MN, const GemmShape& sh_dw,
                              const EpiParams& ep_dw, const CUtensorMap& tmG_K,
                              const CUtensorMap& tmW_MN, const GemmShape& sh_dh,
                              const EpiParams& ep_dh, int* status, int grid, cudaStream_t stream) {
  if (pair && (grid % 2) != 0) return cudaErrorInvalidValue;
  if (dh_first) {  // job 0 = dH (A K-major), job 1 = dW
    if (pair)
      return launch_one<EPI_STORE, false, true, 256, true, true>(
          "dW_dH_gemm", tmG_K, tmW_MN, tmG_MN, tmH_MN, sh_dh, sh_dw, ep_dh, ep_dw, status, grid,
          stream);
    return launch_one<EPI_STORE, false, true, 256, false, true>(
        "dW_dH_gemm", tmG_K, tmW_MN, tmG_MN, tmH_MN, sh_dh, sh_dw, ep_dh, ep_dw, status, grid,
        stream);
  }
  if (pair)  // job 0 = dW (A MN-major), job 1 = dH
    return launch_one<EPI_STORE, true, true, 256, true, true>(
        "dW_dH_gemm", tmG_MN, tmH_MN, tmG_K, tmW_MN, sh_dw, sh_dh, ep_dw, ep_dh, status, grid,
        stream);
  return launch_one<EPI_STORE, true, true, 256, false, true>(
      "dW_dH_gemm", tmG_MN, tmH_MN, tmG_K, tmW_MN, sh_dw, sh_dh, ep_dw, ep_dh, status, grid,
      stream);
}

}  // namespace kdkl
