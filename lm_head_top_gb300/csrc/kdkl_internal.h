// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace kdkl {

struct GemmShape;
struct EpiParams;

// Launch bookkeeping: counts every kernel launch and, while timing is on,
// brackets it with CUDA events on its stream.
void note_launch_begin(const char* name, cudaStream_t stream, void** token);
void note_launch_end(void* token, cudaStream_t stream);

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block,
                          size_t smem, cudaStream_t stream, Args&&... args) {
  void* token = nullptr;
  note_launch_begin(name, stream, &token);
  kern<<<grid, block, smem, stream>>>(std::forward<Args>(args)...);
  const cudaError_t e = cudaGetLastError();
  note_launch_end(token, stream);
  return e;
}

// Same, launched as clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block,
                                  size_t smem, cudaStream_t stream, unsigned cluster_x,
                                  Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* token = nullptr;
  note_launch_begin(name, stream, &token);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e == cudaSuccess) e = cudaGetLastError();
  note_launch_end(token, stream);
  return e;
}

// kernels_small.cu
// rowmap == nullptr: row t <- token t, and the mask is counted into *n_count.
// Else row r <- token rowmap[r] for r < *n_count (set by launch_mask_scan).
cudaError_t launch_teacher_prep(const int32_t* idx, const float* logit, const uint8_t* mask,
                                const int32_t* labels, const int* rowmap, int T, int K, int V,
                                float inv_tau, int32_t* sidx, float* sp, float* ent, int* n_count,
                                int* status, cudaStream_t stream);
// Counted-token compaction: rowmap [T], invmap [T], *n_count = N.
cudaError_t launch_mask_scan(const uint8_t* mask, int T, int* rowmap, int* invmap, int* n_count,
                             cudaStream_t stream);
// Hc rows [0, N) <- H rows rowmap[0..N); rows up to N rounded up to `round`
// (at most rows_cap) zeroed.
cudaError_t launch_gather_rows(const uint16_t* H, int d, const int* rowmap, const int* n_count,
                               long long rows_cap, int round, uint16_t* Hc, int num_sms,
                               cudaStream_t stream);
int combine_blocks(int T);
cudaError_t launch_lse_combine(const float* pm, const float* ps, const float* pd, int nsplit, int T,
                               const float* ent, const uint8_t* mask, const int* invmap,
                               float cl2, float inv_tau, float* lse, float* token_kl,
                               double* block_sums, cudaStream_t stream);
cudaError_t launch_lse_combine_mix(const float* pm, const float* ps, const float* pd,
                                   const float* ps1, const float* pzl, int nsplit, int T,
                                   const float* ent, const uint8_t* mask, const int* invmap,
                                   float cl2, float inv_tau, float kl_w, float ce_w, float* lse,
                                   float* lse1, float* token_loss, double* block_sums,
                                   cudaStream_t stream);
cudaError_t launch_loss_finalize(const double* block_sums, int nblocks, const int* n_count,
                                 float* loss, cudaStream_t stream);
// out [T, d] bf16 <- in rows (invmap[t], or t when invmap is nullptr; zeros
// for invmap[t] < 0); n = T * d.
cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, long long n, int d,
                               const int* invmap, int num_sms, cudaStream_t stream);
// merge of per-split top-K lists; shared memory = topk_merge_p2() * 8 bytes
int topk_merge_p2(int nsplit, int K);
cudaError_t launch_topk_merge(const float* unit_val, const int32_t* unit_id, const int* unit_cnt,
                              const uint32_t* row_key, int nsplit, int T, int K, int32_t* out_id,
                              float* out_val, cudaStream_t stream);

// kernels_rkl.cu — reverse KL over the cached ids (CUDA cores; see the file)
struct RklLayout {
  long long n;        // T * K (id, position) pairs
  long long n_tiles;  // radix-sort tiles
  long long n_seg;    // dW segments
  int passes, bits, nbins;
  size_t off_bsum;
  size_t off_G, off_z, off_keys[2], off_vals[2], off_hist, off_scan, off_bstart, off_bend, off_part;
  size_t total;
};
RklLayout rkl_layout(long long T, long long d, int K, long long V, size_t header);
// count -> sort by id -> z per (token, id) pair -> per-token RKL (+ grad_z) -> loss.
// *n_count must start at 0.
cudaError_t rkl_forward(const RklLayout& L, const uint16_t* H, const uint16_t* W,
                        const int32_t* idx, const float* logit, const uint8_t* mask, int T, int d,
                        int K, int V, float inv_tau, float* token_rkl, float* grad_z, float* loss,
                        void* ws, int* status, int* n_count, int num_sms, cudaStream_t stream);
// [recompute G, or sort by id] -> dH -> dW segments -> dW fix-up. *n_count must start at 0.
cudaError_t rkl_backward(const RklLayout& L, const uint16_t* H, const uint16_t* W,
                         const int32_t* idx, const float* logit, const uint8_t* mask, int T, int d,
                         int K, int V, float inv_tau, const float* grad_z, float grad_loss,
                         uint16_t* dH, float* dW, int accumulate, void* ws, int* status,
                         int* n_count, int num_sms, cudaStream_t stream);

// kernels_gemm.cu — tcgen05 GEMMs (see tc_gemm.cuh for the epilogues)
enum GemmKind {
  GEMM_FWD_LSE = 0,   // A = H (K-major), B = W (K-major), online logsumexp + gather
  GEMM_BWD_GRAD = 1,  // A = H (K-major), B = W (K-major), softmax - P into the bf16 buffer
  GEMM_DH = 2,        // A = G (K-major), B = W (MN-major), fp32 out
  GEMM_DW = 3,        // A = G (MN-major), B = H (MN-major), fp32 out
  GEMM_TOPK = 4,      // A = H (K-major), B = W (K-major), per-split top-K lists
  GEMM_FWD_LSE_MIX = 5,   // forward with the temperature-1 sum and the label logit
  GEMM_BWD_GRAD_MIX = 6   // backward gradient of the mixed soft + hard-label loss
};
// How many 2-CTA clusters of the GEMM kernel fit on the current device at once
// (0 if unknown). The persistent grid must not exceed it.
int pair_max_active_clusters();

// bn: N tile width (LOGIT_BN for the logit GEMMs; 256 for dH/dW).
// pair: 2-CTA clusters sharing one 256 x bn tile (grid must be even).
cudaError_t launch_gemm(GemmKind kind, int bn, bool pair, const CUtensorMap& tmA,
                        const CUtensorMap& tmB,
                        const GemmShape& sh, const EpiParams& ep, int* status, int grid,
                        cudaStream_t stream);

// dW (A = G^T, B = H, both MN-major) and dH (A = G K-major, B = W MN-major)
// of one backward block in one persistent launch, their units in one
// sequence: dW's first, or dH's first when dh_first. 256-wide N tiles.
cudaError_t launch_gemm_dw_dh(bool pair, bool dh_first, const CUtensorMap& tmG_MN,
                              const CUtensorMap& tmH_MN, const GemmShape& sh_dw,
                              const EpiParams& ep_dw, const CUtensorMap& tmG_K,
                              const CUtensorMap& tmW_MN, const GemmShape& sh_dh,
                              const EpiParams& ep_dh, int* status, int grid, cudaStream_t stream);

}  // namespace kdkl
