// Bandwidth-light kernels around the tensor-core GEMMs:
//   teacher_prep   per token: validate ids, teacher softmax over the K cached
//                  logits, entropy term, sort (id, p) by id, count the mask.
//   lse_combine    per token: merge the vocabulary-split partials into lse and
//                  KL, plus a per-block sum of m_t KL_t (fp64).
//   loss_finalize  one block: ordered sum of the block sums / N.
//   f32_to_bf16    dH accumulator to bf16 (round to nearest even).
//
// Teacher distribution and KL from "Making knowledge distillation cheap
// enough to run at scale", section "Two system changes" (top-100 cache per
// position; the sparse teacher of the forward-chunked and fused variants).
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "kdkl_internal.h"
#include "tc_primitives.cuh"

namespace kdkl {

constexpr int PREP_WARPS = 8;

// One warp per token row. Dynamic shared memory: PREP_WARPS * p2 * 8 bytes.
__global__ void __launch_bounds__(PREP_WARPS * 32)
    teacher_prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ logit,
                        const uint8_t* __restrict__ mask, const int32_t* __restrict__ labels,
                        int T, int K, int p2, int V, float inv_tau, int32_t* __restrict__ sidx,
                        float* __restrict__ sp, float* __restrict__ ent, int* n_count,
                        int* status) {
  extern __shared__ uint8_t prep_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* keys = reinterpret_cast<int*>(prep_smem) + warp * p2;
  float* vals = reinterpret_cast<float*>(prep_smem + (size_t)PREP_WARPS * p2 * 4) + warp * p2;
  const int t = blockIdx.x * PREP_WARPS + warp;
  __shared__ int block_count;
  if (threadIdx.x == 0) block_count = 0;
  __syncthreads();

  if (t < T) {
    const int32_t* irow = idx + (long long)t * K;
    const float* lrow = logit + (long long)t * K;
    // max of a = logit / tau; validate ids and logits
    float amax = -INFINITY;
    bool bad_id = false, bad_logit = false;
    for (int k = lane; k < K; k += 32) {
      const int id = __ldg(irow + k);
      const float a = __ldg(lrow + k) * inv_tau;
      bad_id |= (id < 0 || id >= V);
      bad_logit |= (a != a) || (a == INFINITY);
      amax = fmaxf(amax, a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (__any_sync(0xffffffffu, bad_id) && lane == 0) record_error(status, DEV_ERR_INDEX_RANGE);
    const bool no_finite = !(amax > -INFINITY);
    if ((__any_sync(0xffffffffu, bad_logit) || no_finite) && lane == 0)
      record_error(status, DEV_ERR_INVALID_ARG);
    // sum of exp(a - max)
    float sum = 0.f;
    for (int k = lane; k < K; k += 32) sum += expf(__ldg(lrow + k) * inv_tau - amax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float log_sum = logf(sum);
    // p, entropy term sum p log p, and the (id, p) pairs to sort
    float h = 0.f;
    for (int k = lane; k < p2; k += 32) {
      if (k < K) {
        const float a = __ldg(lrow + k) * inv_tau - amax;  // <= 0 or -inf
        const float p = no_finite ? 0.f : expf(a) / sum;
        if (p > 0.f) h += p * (a - log_sum);
        keys[k] = __ldg(irow + k);
        vals[k] = p;
      } else {
        keys[k] = 0x7fffffff;
        vals[k] = 0.f;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    __syncwarp();
    // bitonic sort of p2 (power of two) pairs, ascending by id
    for (int size = 2; size <= p2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = lane; i < (p2 >> 1); i += 32) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool ascending = (lo & size) == 0;
          const int klo = keys[lo], khi = keys[hi];
          if ((klo > khi) == ascending) {
            keys[lo] = khi;
            keys[hi] = klo;
            const float vlo = vals[lo];
            vals[lo] = vals[hi];
            vals[hi] = vlo;
          }
        }
        __syncwarp();
      }
    }
    int32_t* so = sidx + (long long)t * K;
    float* po = sp + (long long)t * K;
    for (int k = lane; k < K; k += 32) {
      so[k] = keys[k];
      po[k] = vals[k];
    }
    if (lane == 0) {
      if (labels && (labels[t] < 0 || labels[t] >= V)) record_error(status, DEV_ERR_INDEX_RANGE);
      if (ent) ent[t] = h;
      if (mask == nullptr || mask[t] != 0) atomicAdd(&block_count, 1);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && block_count) atomicAdd(n_count, block_count);
}

constexpr int COMBINE_THREADS = 256;

__global__ void __launch_bounds__(COMBINE_THREADS)
    lse_combine_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                       const float* __restrict__ pd, int nsplit, int T,
                       const float* __restrict__ ent, const uint8_t* __restrict__ mask, float cl2,
                       float inv_tau, float* __restrict__ lse, float* __restrict__ token_kl,
                       double* __restrict__ block_sums) {
  const int t = blockIdx.x * COMBINE_THREADS + threadIdx.x;
  double contrib = 0.0;
  if (t < T) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pm[(long long)s * T + t]);
    float S = 0.f, D = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const long long o = (long long)s * T + t;
      S += ps[o] * exp2f((pm[o] - M) * cl2);
      D += pd[o];
    }
    const float l = M * inv_tau + logf(S);
    const float kl = ent[t] - D * inv_tau + l;
    lse[t] = l;
    if (token_kl) token_kl[t] = kl;
    if (mask == nullptr || mask[t] != 0) contrib = (double)kl;
  }
  // fixed-shape tree reduction: deterministic
  __shared__ double red[COMBINE_THREADS];
  red[threadIdx.x] = contrib;
  __syncthreads();
  for (int w = COMBINE_THREADS / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) block_sums[blockIdx.x] = red[0];
}

// Mixed loss: per token alpha c KL + (1 - alpha) CE with CE = lse_1 - z_label.
__global__ void __launch_bounds__(COMBINE_THREADS)
    lse_combine_mix_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                           const float* __restrict__ pd, const float* __restrict__ ps1,
                           const float* __restrict__ pzl, int nsplit, int T,
                           const float* __restrict__ ent, const uint8_t* __restrict__ mask,
                           float cl2, float inv_tau, float kl_w, float ce_w,
                           float* __restrict__ lse, float* __restrict__ lse1,
                           float* __restrict__ token_loss, double* __restrict__ block_sums) {
  const int t = blockIdx.x * COMBINE_THREADS + threadIdx.x;
  double contrib = 0.0;
  if (t < T) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pm[(long long)s * T + t]);
    float S = 0.f, S1 = 0.f, D = 0.f, Z = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const long long o = (long long)s * T + t;
      S += ps[o] * exp2f((pm[o] - M) * cl2);
      S1 += ps1[o] * exp2f((pm[o] - M) * 1.4426950408889634f);
      D += pd[o];
      Z += pzl[o];
    }
    const float l = M * inv_tau + logf(S);
    const float l1 = M + logf(S1);
    const float kl = ent[t] - D * inv_tau + l;
    const float tok = kl_w * kl + ce_w * (l1 - Z);
    lse[t] = l;
    lse1[t] = l1;
    if (token_loss) token_loss[t] = tok;
    if (mask == nullptr || mask[t] != 0) contrib = (double)tok;
  }
  __shared__ double red[COMBINE_THREADS];
  red[threadIdx.x] = contrib;
  __syncthreads();
  for (int w = COMBINE_THREADS / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) block_sums[blockIdx.x] = red[0];
}

__global__ void __launch_bounds__(1024)
    loss_finalize_kernel(const double* __restrict__ block_sums, int nblocks,
                         const int* __restrict__ n_count, float* __restrict__ loss) {
  __shared__ double red[1024];
  double a = 0.0;
  for (int i = threadIdx.x; i < nblocks; i += 1024) a += block_sums[i];
  red[threadIdx.x] = a;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int n = *n_count;
    loss[0] = n > 0 ? (float)(red[0] / (double)n) : 0.f;
  }
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out,
                                   long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = in[i];
    out[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// Merge each row's per-split top-K lists into the row's top-K, sorted by
// (logit descending, id ascending). One warp per row. Entries below the
// row's shared threshold key (the best K-th logit any split reached, which is
// at most the row's true K-th logit) cannot be in the top-K and are dropped;
// the survivors (at least K) are compacted in order and sorted as 64-bit keys
// (inverted order key of the logit, then the id) by a warp bitonic sort in
// shared memory.
__device__ __forceinline__ uint32_t merge_order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Number of keys among keys[0, m) at or below x, summed over the warp.
__device__ __forceinline__ int merge_count_le(const unsigned long long* keys, int m,
                                              unsigned long long x) {
  int c = 0;
  for (int i = threadIdx.x & 31; i < m; i += 32) c += keys[i] <= x ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Moves the K smallest of keys[0, m) (all distinct: the low half is the id)
// to keys[0, K), in their original order, and returns K. The K-th smallest key
// is found by bisection, first over the high 32 bits (the logit order), then,
// only when several entries share the K-th logit, over the low 32 bits (the
// id), so that ties keep the smaller ids.
__device__ int merge_select_k(unsigned long long* keys, int m, int K) {
  const int lane = threadIdx.x & 31;
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = lane; i < m; i += 32) {
    const uint32_t h = (uint32_t)(keys[i] >> 32);
    lo = min(lo, h);
    hi = max(hi, h);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  while (lo < hi) {  // smallest h with at least K keys whose high half is <= h
    const uint32_t mid = lo + ((hi - lo) >> 1);
    if (merge_count_le(keys, m, ((unsigned long long)mid << 32) | 0xffffffffull) >= K)
      hi = mid;
    else
      lo = mid + 1u;
  }
  unsigned long long cut = ((unsigned long long)lo << 32) | 0xffffffffull;
  if (merge_count_le(keys, m, cut) > K) {  // ties on the K-th logit: bisect the ids
    uint32_t a = 0u, b = 0xffffffffu;
    while (a < b) {
      const uint32_t mid = a + ((b - a) >> 1);
      if (merge_count_le(keys, m, ((unsigned long long)lo << 32) | mid) >= K)
        b = mid;
      else
        a = mid + 1u;
    }
    cut = ((unsigned long long)lo << 32) | a;
  }
  // stable in-place compaction of the keys <= cut (exactly K of them)
  const uint32_t below = (1u << lane) - 1u;
  int w = 0;
  for (int i0 = 0; i0 < m; i0 += 32) {
    const int i = i0 + lane;
    const unsigned long long k = i < m ? keys[i] : ~0ull;
    const bool keep = i < m && k <= cut;
    const uint32_t mask = __ballot_sync(0xffffffffu, keep);  // all reads of this round are done
    if (keep) keys[w + __popc(mask & below)] = k;
    w += __popc(mask);
  }
  __syncwarp();
  return w;
}

// One warp per row; `rows_per_block` warps share the block's shared memory,
// cap entries (a power of two >= nsplit * K) each.
__global__ void __launch_bounds__(256)
    topk_merge_kernel(const float* __restrict__ unit_val, const int32_t* __restrict__ unit_id,
                      const uint32_t* __restrict__ row_key, int nsplit, int T, int K, int cap,
                      int32_t* __restrict__ out_id, float* __restrict__ out_val) {
  extern __shared__ unsigned long long mkeys_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;  // whole warp leaves together; no block-wide barrier below
  unsigned long long* mkeys = mkeys_all + (size_t)warp * cap;
  const int n = nsplit * K;
  const uint32_t floor_key = row_key[t];
  const uint32_t below = (1u << lane) - 1u;
  int m = 0;
  constexpr int BATCH = 8;  // independent loads in flight per lane
  for (int e0 = 0; e0 < n; e0 += 32 * BATCH) {
    float vb[BATCH];
    int32_t ib[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int e = e0 + b * 32 + lane;
      if (e < n) {
        const int s = e / K, k = e - s * K;
        const long long o = ((long long)s * T + t) * K + k;
        vb[b] = unit_val[o];
        ib[b] = unit_id[o];
      } else {
        vb[b] = -INFINITY;
        ib[b] = -1;
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const uint32_t ok = merge_order_key(vb[b]);
      const bool keep = ib[b] >= 0 && ok >= floor_key;
      const uint32_t mask = __ballot_sync(0xffffffffu, keep);
      if (keep) mkeys[m + __popc(mask & below)] = ((unsigned long long)(~ok) << 32) | (uint32_t)ib[b];
      m += __popc(mask);
    }
  }
  __syncwarp();
  if (m > K) m = merge_select_k(mkeys, m, K);  // keep the K best, then sort only those
  int p2 = 2;
  while (p2 < m) p2 <<= 1;
  for (int e = m + lane; e < p2; e += 32) mkeys[e] = ~0ull;
  __syncwarp();
  for (int size = 2; size <= p2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < (p2 >> 1); i += 32) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool ascending = (lo & size) == 0;
        const unsigned long long a = mkeys[lo], b = mkeys[hi];
        if ((a > b) == ascending) {
          mkeys[lo] = b;
          mkeys[hi] = a;
        }
      }
      __syncwarp();
    }
  }
  for (int k = lane; k < K; k += 32) {
    const unsigned long long key = mkeys[k];
    const uint32_t ok = ~(uint32_t)(key >> 32);
    out_val[(long long)t * K + k] = __uint_as_float((ok & 0x80000000u) ? (ok & 0x7fffffffu) : ~ok);
    out_id[(long long)t * K + k] = (int32_t)(uint32_t)(key & 0xffffffffu);
  }
}

// ------------------------------------------------------------ host launchers

cudaError_t launch_teacher_prep(const int32_t* idx, const float* logit, const uint8_t* mask,
                                const int32_t* labels, int T, int K, int V, float inv_tau,
                                int32_t* sidx, float* sp, float* ent, int* n_count, int* status,
                                cudaStream_t stream) {
  int p2 = 1;
  while (p2 < K) p2 <<= 1;
  if (p2 < 2) p2 = 2;
  const size_t smem = (size_t)PREP_WARPS * p2 * 8;
  const int blocks = (T + PREP_WARPS - 1) / PREP_WARPS;
  return launch_kernel("teacher_prep", teacher_prep_kernel, dim3(blocks), dim3(PREP_WARPS * 32),
                       smem, stream, idx, logit, mask, labels, T, K, p2, V, inv_tau, sidx, sp,
                       ent, n_count, status);
}

int combine_blocks(int T) { return (T + COMBINE_THREADS - 1) / COMBINE_THREADS; }

cudaError_t launch_lse_combine(const float* pm, const float* ps, const float* pd, int nsplit, int T,
                               const float* ent, const uint8_t* mask, float cl2, float inv_tau,
                               float* lse, float* token_kl, double* block_sums,
                               cudaStream_t stream) {
  return launch_kernel("lse_combine", lse_combine_kernel, dim3(combine_blocks(T)),
                       dim3(COMBINE_THREADS), 0, stream, pm, ps, pd, nsplit, T, ent, mask, cl2,
                       inv_tau, lse, token_kl, block_sums);
}

cudaError_t launch_lse_combine_mix(const float* pm, const float* ps, const float* pd,
                                   const float* ps1, const float* pzl, int nsplit, int T,
                                   const float* ent, const uint8_t* mask, float cl2, float inv_tau,
                                   float kl_w, float ce_w, float* lse, float* lse1,
                                   float* token_loss, double* block_sums, cudaStream_t stream) {
  return launch_kernel("lse_combine_mix", lse_combine_mix_kernel, dim3(combine_blocks(T)),
                       dim3(COMBINE_THREADS), 0, stream, pm, ps, pd, ps1, pzl, nsplit, T, ent,
                       mask, cl2, inv_tau, kl_w, ce_w, lse, lse1, token_loss, block_sums);
}

cudaError_t launch_loss_finalize(const double* block_sums, int nblocks, const int* n_count,
                                 float* loss, cudaStream_t stream) {
  return launch_kernel("loss_finalize", loss_finalize_kernel, dim3(1), dim3(1024), 0, stream,
                       block_sums, nblocks, n_count, loss);
}

int topk_merge_p2(int nsplit, int K) {
  int p2 = 1;
  while (p2 < nsplit * K) p2 <<= 1;
  return p2 < 2 ? 2 : p2;
}

cudaError_t launch_topk_merge(const float* unit_val, const int32_t* unit_id, const uint32_t* row_key,
                              int nsplit, int T, int K, int32_t* out_id, float* out_val,
                              cudaStream_t stream) {
  const int cap = topk_merge_p2(nsplit, K);  // <= 4096 entries, 32 KB per warp
  const int warps = std::max(1, std::min(8, 6144 / cap));  // <= 48 KB of shared memory
  return launch_kernel("topk_merge", topk_merge_kernel, dim3((T + warps - 1) / warps),
                       dim3(32 * warps), (size_t)warps * cap * sizeof(unsigned long long), stream,
                       unit_val, unit_id, row_key, nsplit, T, K, cap, out_id, out_val);
}

cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, long long n, int num_sms,
                               cudaStream_t stream) {
  const long long n4 = n / 4;  // n is a multiple of 8 (d % 8 == 0)
  long long blocks = (n4 + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel("f32_to_bf16", f32_to_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0,
                       stream, reinterpret_cast<const float4*>(in), reinterpret_cast<uint2*>(out),
                       n4);
}

}  // namespace kdkl
