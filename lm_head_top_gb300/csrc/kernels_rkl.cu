// Reverse KL restricted to the cached ids: a loss-choice variant whose
// gradient lives only on the K cached ids of each token, so it needs no
// vocabulary-wide GEMM. Per token (one warp): gather the K rows of W, form the
// logits z[t, idx_k] = H_t . W[idx_k] (fp32 sums of bf16 products), then
//   qt = softmax_k(z_idx / tau), p = softmax_k(topk_logit / tau)   (entries with
//   a -inf teacher logit are outside the support and dropped from both)
//   RKL_t = sum_k qt_k (log qt_k - log p_k)
//   dRKL/dz_k = qt_k (log qt_k - log p_k - RKL_t) / tau.
// The backward writes dH_t = sum_k g_k W[idx_k] (bf16) and adds g_k H_t into
// dW[idx_k] with vector reductions (fp32; the order of the adds across tokens
// is not fixed, so dW is not bitwise reproducible).
//
// Loss-choice ablation: "Making knowledge distillation cheap enough to run at
// scale", closing section (the paper's ablations over the choice of loss).
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "kdkl_internal.h"
#include "tc_primitives.cuh"

namespace kdkl {

constexpr int RKL_WARPS = 8;
constexpr int RKL_MAX_K = 512;  // entries per warp kept in shared memory

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_sum_f(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max_f(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// z[k] = H_t . W[idx_k] for the warp's token into zs (shared); returns false
// (and flags the status) if an id is out of range, in which case that entry
// reads no memory and its z is 0.
__device__ bool rkl_gather_logits(const uint16_t* __restrict__ Ht, const uint16_t* __restrict__ W,
                                  const int32_t* __restrict__ irow, int d, int K, int V,
                                  float* zs, int* status) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  for (int k = 0; k < K; ++k) {
    const int id = __ldg(irow + k);
    float acc = 0.f;
    if (id >= 0 && id < V) {
      const uint16_t* wr = W + (long long)id * d;
      for (int i = lane * 8; i < d; i += 256) {
        const uint4 h = __ldg(reinterpret_cast<const uint4*>(Ht + i));
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(wr + i));
        acc = fmaf(bf16lo(h.x), bf16lo(w.x), acc);
        acc = fmaf(bf16hi(h.x), bf16hi(w.x), acc);
        acc = fmaf(bf16lo(h.y), bf16lo(w.y), acc);
        acc = fmaf(bf16hi(h.y), bf16hi(w.y), acc);
        acc = fmaf(bf16lo(h.z), bf16lo(w.z), acc);
        acc = fmaf(bf16hi(h.z), bf16hi(w.z), acc);
        acc = fmaf(bf16lo(h.w), bf16lo(w.w), acc);
        acc = fmaf(bf16hi(h.w), bf16hi(w.w), acc);
      }
    } else {
      ok = false;
    }
    acc = warp_sum_f(acc);
    if (lane == 0) zs[k] = acc;
  }
  if (!ok && lane == 0) record_error(status, DEV_ERR_INDEX_RANGE);
  __syncwarp();
  return ok;
}

// Restricted log-softmaxes and the token's reverse KL. On return, for each
// k handled by this lane (k = lane, lane + 32, ...): zs[k] = log qt_k and
// ls[k] = log p_k (-inf outside the support).
__device__ float rkl_token(const float* __restrict__ lrow, int K, float inv_tau, float* zs,
                           float* ls, int* status) {
  const int lane = threadIdx.x & 31;
  float am = -INFINITY, bm = -INFINITY;
  bool any = false;
  for (int k = lane; k < K; k += 32) {
    const float lg = __ldg(lrow + k);
    const bool keep = fabsf(lg) < INFINITY;  // -inf (and any non-finite) leaves the support
    ls[k] = keep ? lg * inv_tau : -INFINITY;
    zs[k] = keep ? zs[k] * inv_tau : -INFINITY;
    if (keep) {
      am = fmaxf(am, zs[k]);
      bm = fmaxf(bm, ls[k]);
      any = true;
    }
  }
  am = warp_max_f(am);
  bm = warp_max_f(bm);
  if (!__any_sync(0xffffffffu, any)) {
    if (lane == 0) record_error(status, DEV_ERR_INVALID_ARG);
    return 0.f;
  }
  float sa = 0.f, sb = 0.f;
  for (int k = lane; k < K; k += 32) {
    if (ls[k] > -INFINITY) {
      sa += expf(zs[k] - am);
      sb += expf(ls[k] - bm);
    }
  }
  const float lsa = am + logf(warp_sum_f(sa));
  const float lsb = bm + logf(warp_sum_f(sb));
  float r = 0.f;
  for (int k = lane; k < K; k += 32) {
    if (ls[k] > -INFINITY) {
      zs[k] -= lsa;  // log qt
      ls[k] -= lsb;  // log p
      r += expf(zs[k]) * (zs[k] - ls[k]);
    }
  }
  return warp_sum_f(r);
}

__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_forward_kernel(const uint16_t* __restrict__ H, const uint16_t* __restrict__ W,
                       const int32_t* __restrict__ idx, const float* __restrict__ logit,
                       const uint8_t* __restrict__ mask, int T, int d, int K, int V, float inv_tau,
                       float* __restrict__ token_rkl, double* __restrict__ block_sums,
                       int* n_count, int* status) {
  __shared__ float zs_all[RKL_WARPS][RKL_MAX_K];
  __shared__ float ls_all[RKL_WARPS][RKL_MAX_K];
  __shared__ double wsum[RKL_WARPS];
  __shared__ int wcount[RKL_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * RKL_WARPS + warp;
  double contrib = 0.0;
  int counted = 0;
  if (t < T) {
    float* zs = zs_all[warp];
    float* ls = ls_all[warp];
    rkl_gather_logits(H + (long long)t * d, W, idx + (long long)t * K, d, K, V, zs, status);
    const float r = rkl_token(logit + (long long)t * K, K, inv_tau, zs, ls, status);
    if (lane == 0) {
      if (token_rkl) token_rkl[t] = r;
      counted = (mask == nullptr || mask[t] != 0) ? 1 : 0;
      contrib = counted ? (double)r : 0.0;
    }
  }
  if (lane == 0) {
    wsum[warp] = contrib;
    wcount[warp] = counted;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    int c = 0;
    for (int w = 0; w < RKL_WARPS; ++w) {
      s += wsum[w];
      c += wcount[w];
    }
    block_sums[blockIdx.x] = s;
    if (c) atomicAdd(n_count, c);
  }
}

// Counts the tokens that contribute (the backward needs N before the gradient).
__global__ void rkl_count_kernel(const uint8_t* __restrict__ mask, int T, int* n_count) {
  int c = 0;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x)
    c += (mask == nullptr || mask[t] != 0) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(n_count, c);
}

__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_backward_kernel(const uint16_t* __restrict__ H, const uint16_t* __restrict__ W,
                        const int32_t* __restrict__ idx, const float* __restrict__ logit,
                        const uint8_t* __restrict__ mask, int T, int d, int K, int V,
                        float inv_tau, float grad_loss, const int* __restrict__ n_count,
                        uint16_t* __restrict__ dH, float* __restrict__ dW, int* status) {
  __shared__ float zs_all[RKL_WARPS][RKL_MAX_K];
  __shared__ float ls_all[RKL_WARPS][RKL_MAX_K];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * RKL_WARPS + warp;
  if (t >= T) return;  // no block-wide barrier below
  float* zs = zs_all[warp];
  float* ls = ls_all[warp];
  const uint16_t* Ht = H + (long long)t * d;
  const int32_t* irow = idx + (long long)t * K;
  const bool ids_ok = rkl_gather_logits(Ht, W, irow, d, K, V, zs, status);
  const float r = rkl_token(logit + (long long)t * K, K, inv_tau, zs, ls, status);
  const int n = *n_count;
  const bool counted = mask == nullptr || mask[t] != 0;
  const float scale = (counted && n > 0 && ids_ok) ? grad_loss * inv_tau / (float)n : 0.f;
  // g_k into zs (dropped entries: 0)
  for (int k = lane; k < K; k += 32)
    zs[k] = ls[k] > -INFINITY ? scale * expf(zs[k]) * (zs[k] - ls[k] - r) : 0.f;
  __syncwarp();
  // dH_t = sum_k g_k W[idx_k], 1024 columns at a time (32 per lane)
  for (int c0 = 0; c0 < d; c0 += 1024) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    for (int k = 0; k < K; ++k) {
      const float g = zs[k];
      const int id = __ldg(irow + k);
      if (g == 0.f || id < 0 || id >= V) continue;  // warp-uniform
      const uint16_t* wr = W + (long long)id * d;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = c0 + q * 256 + lane * 8;
        if (i < d) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(wr + i));
          acc[8 * q + 0] = fmaf(g, bf16lo(w.x), acc[8 * q + 0]);
          acc[8 * q + 1] = fmaf(g, bf16hi(w.x), acc[8 * q + 1]);
          acc[8 * q + 2] = fmaf(g, bf16lo(w.y), acc[8 * q + 2]);
          acc[8 * q + 3] = fmaf(g, bf16hi(w.y), acc[8 * q + 3]);
          acc[8 * q + 4] = fmaf(g, bf16lo(w.z), acc[8 * q + 4]);
          acc[8 * q + 5] = fmaf(g, bf16hi(w.z), acc[8 * q + 5]);
          acc[8 * q + 6] = fmaf(g, bf16lo(w.w), acc[8 * q + 6]);
          acc[8 * q + 7] = fmaf(g, bf16hi(w.w), acc[8 * q + 7]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = c0 + q * 256 + lane * 8;
      if (i < d) {
        uint4 o;
        o.x = pack_bf16x2(acc[8 * q + 0], acc[8 * q + 1]);
        o.y = pack_bf16x2(acc[8 * q + 2], acc[8 * q + 3]);
        o.z = pack_bf16x2(acc[8 * q + 4], acc[8 * q + 5]);
        o.w = pack_bf16x2(acc[8 * q + 6], acc[8 * q + 7]);
        *reinterpret_cast<uint4*>(dH + (long long)t * d + i) = o;
      }
    }
  }
  // dW[idx_k] += g_k H_t
  for (int k = 0; k < K; ++k) {
    const float g = zs[k];
    const int id = __ldg(irow + k);
    if (g == 0.f || id < 0 || id >= V) continue;  // warp-uniform
    float* wr = dW + (long long)id * d;
    for (int i = lane * 4; i < d; i += 128) {
      const uint2 h = __ldg(reinterpret_cast<const uint2*>(Ht + i));
      red_add_f32x4(wr + i, make_float4(g * bf16lo(h.x), g * bf16hi(h.x), g * bf16lo(h.y),
                                        g * bf16hi(h.y)));
    }
  }
}

cudaError_t launch_rkl_forward(const uint16_t* H, const uint16_t* W, const int32_t* idx,
                               const float* logit, const uint8_t* mask, int T, int d, int K, int V,
                               float inv_tau, float* token_rkl, double* block_sums, int* n_count,
                               int* status, cudaStream_t stream) {
  return launch_kernel("rkl_forward", rkl_forward_kernel, dim3((T + RKL_WARPS - 1) / RKL_WARPS),
                       dim3(RKL_WARPS * 32), 0, stream, H, W, idx, logit, mask, T, d, K, V, inv_tau,
                       token_rkl, block_sums, n_count, status);
}

int rkl_blocks(int T) { return (T + RKL_WARPS - 1) / RKL_WARPS; }

cudaError_t launch_rkl_backward(const uint16_t* H, const uint16_t* W, const int32_t* idx,
                                const float* logit, const uint8_t* mask, int T, int d, int K, int V,
                                float inv_tau, float grad_loss, int* n_count, uint16_t* dH,
                                float* dW, int* status, int num_sms, cudaStream_t stream) {
  cudaError_t e = launch_kernel("rkl_count", rkl_count_kernel, dim3(std::min(num_sms, 64)),
                                dim3(256), 0, stream, mask, T, n_count);
  if (e != cudaSuccess) return e;
  return launch_kernel("rkl_backward", rkl_backward_kernel, dim3(rkl_blocks(T)),
                       dim3(RKL_WARPS * 32), 0, stream, H, W, idx, logit, mask, T, d, K, V,
                       inv_tau, grad_loss, n_count, dH, dW, status);
}

}  // namespace kdkl
