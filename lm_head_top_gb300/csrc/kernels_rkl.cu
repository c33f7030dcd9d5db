// Reverse KL restricted to the cached ids: a loss-choice variant whose
// gradient lives only on the K cached ids of each token, so it needs no
// vocabulary-wide GEMM. With z[t, idx_k] = H_t . W[idx_k] (fp32 sums of bf16
// products):
//   qt = softmax_k(z_idx / tau), p = softmax_k(topk_logit / tau)   (entries with
//   a non-finite teacher logit are outside the support and dropped from both)
//   RKL_t = sum_k qt_k (log qt_k - log p_k)
//   dRKL/dz_k = qt_k (log qt_k - log p_k - RKL_t) / tau.
//
// Kernels (all CUDA-core; the work is a sparse gather, not a contraction):
//   rkl_count      unmasked-token count N
//   rkl_z_segment  z for every (token, id) pair, vocabulary-major over the
//                  pairs sorted by id: each named row of W read once per
//                  segment, the tokens' rows of H streamed against it
//   rkl_forward    one warp per token: the restricted softmaxes of its K z,
//                  RKL_t, optionally G[t,k] = dL/dz at the ids (grad_loss = 1)
//   rkl_dH         one warp per token: dH_t = g * sum_k G[t,k] W[idx_k]
//   radix_hist / scan_* / radix_scatter / bucket_bounds
//                  stable LSD radix sort of the T*K (id, t*K+k) pairs by id, so
//                  that every vocabulary row's contributions are contiguous and
//                  in token order
//   rkl_dW_segment one warp per fixed segment of the sorted pairs: sums
//                  g G H_t per id in registers and writes each dW row once;
//                  ids that straddle a segment edge go to per-segment partials
//   rkl_dW_fixup   one warp per vocabulary row: adds the partials of
//                  straddling ids in segment order, zeroes untouched rows
// No atomics touch dW or dH and every sum runs in a fixed order, so the
// backward is bitwise reproducible.
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
constexpr int RADIX_TILE = 4096;
constexpr int RADIX_THREADS = 256;
constexpr int RADIX_ROUNDS = RADIX_TILE / RADIX_THREADS;
constexpr int RADIX_MAX_BITS = 10;
constexpr int RADIX_MAX_BINS = 1 << RADIX_MAX_BITS;
constexpr int SEG = 256;  // sorted pairs per dW segment (one warp)
constexpr int SCAN_THREADS = 1024;

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

__device__ __forceinline__ float dot8_bf16(uint4 h, uint4 w, float acc) {
  acc = fmaf(bf16lo(h.x), bf16lo(w.x), acc);
  acc = fmaf(bf16hi(h.x), bf16hi(w.x), acc);
  acc = fmaf(bf16lo(h.y), bf16lo(w.y), acc);
  acc = fmaf(bf16hi(h.y), bf16hi(w.y), acc);
  acc = fmaf(bf16lo(h.z), bf16lo(w.z), acc);
  acc = fmaf(bf16hi(h.z), bf16hi(w.z), acc);
  acc = fmaf(bf16lo(h.w), bf16lo(w.w), acc);
  return fmaf(bf16hi(h.w), bf16hi(w.w), acc);
}

__device__ __forceinline__ void axpy8_bf16(float* acc, float g, uint4 w) {
  acc[0] = fmaf(g, bf16lo(w.x), acc[0]);
  acc[1] = fmaf(g, bf16hi(w.x), acc[1]);
  acc[2] = fmaf(g, bf16lo(w.y), acc[2]);
  acc[3] = fmaf(g, bf16hi(w.y), acc[3]);
  acc[4] = fmaf(g, bf16lo(w.z), acc[4]);
  acc[5] = fmaf(g, bf16hi(w.z), acc[5]);
  acc[6] = fmaf(g, bf16lo(w.w), acc[6]);
  acc[7] = fmaf(g, bf16hi(w.w), acc[7]);
}

// The dW segments read rows of H RB at a time (2 measured best: 4 costs
// registers and occupancy, 1 a round trip per row), each as a 1024-column slice
// (4 x 16 bytes per lane): all RB * 4 loads are issued before any of them is
// used, so a warp waits on one memory round trip per RB rows instead of per
// row. Slots past the end of a run, and columns past d, read row 0 / column 0
// (always in bounds) and are discarded.
constexpr int RB = 2;

__device__ __forceinline__ void load_slices(uint4 (&w)[RB][4], const uint16_t* __restrict__ base,
                                            const int (&row)[RB], int c0, int d, int lane) {
#pragma unroll
  for (int u = 0; u < RB; ++u) {
    const uint16_t* r = base + (long long)row[u] * d;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = c0 + q * 256 + lane * 8;
      w[u][q] = __ldg(reinterpret_cast<const uint4*>(r + (i < d ? i : 0)));
    }
  }
}

// z[k] for the warp's token from a buffer the segment kernel filled (one
// float per (token, id) pair). Returns false (and flags the status) if an id is
// out of range; such entries hold 0.
__device__ bool rkl_load_logits(const int32_t* __restrict__ irow, const float* __restrict__ zrow,
                                int K, int V, float* zs, int* status) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  for (int k = lane; k < K; k += 32) {
    const int id = __ldg(irow + k);
    ok = ok && id >= 0 && id < V;
    zs[k] = __ldg(zrow + k);
  }
  ok = __all_sync(0xffffffffu, ok);
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

// Shared memory one warp of rkl_forward uses: z and log p for the K ids
// (K floats each, padded to 16 bytes).
__host__ __device__ __forceinline__ size_t rkl_forward_smem_per_warp(int K) {
  return (size_t)((K + 3) & ~3) * 8;
}

// Counts the tokens that contribute.
__global__ void rkl_count_kernel(const uint8_t* __restrict__ mask, int T, int* n_count) {
  int c = 0;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x)
    c += (mask == nullptr || mask[t] != 0) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(n_count, c);
}

// One warp per token, with z from zbuf (the segment kernel's output).
// token_rkl, G and block_sums may each be null.
//   G[t,k] = m_t / N * qt_k (log qt_k - log p_k - RKL_t) / tau   (0 off the support,
//            for masked tokens, and for a token with an out-of-range id)
//   block_sums[b] = sum over the block's unmasked tokens of RKL_t (fp64).
__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_forward_kernel(const int32_t* __restrict__ idx, const float* __restrict__ logit,
                       const uint8_t* __restrict__ mask, int T, int K, int V, float inv_tau,
                       const int* __restrict__ n_count, const float* __restrict__ zbuf,
                       float* __restrict__ token_rkl, float* __restrict__ G,
                       double* __restrict__ block_sums, int* status) {
  extern __shared__ __align__(16) unsigned char rkl_smem[];
  __shared__ double wsum[RKL_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * RKL_WARPS + warp;
  double contrib = 0.0;
  if (t < T) {
    const int kpad = (K + 3) & ~3;
    float* zs = reinterpret_cast<float*>(rkl_smem + (size_t)warp * rkl_forward_smem_per_warp(K));
    float* ls = zs + kpad;
    const int32_t* irow = idx + (long long)t * K;
    const bool ids_ok = rkl_load_logits(irow, zbuf + (long long)t * K, K, V, zs, status);
    const float r = rkl_token(logit + (long long)t * K, K, inv_tau, zs, ls, status);
  const bool counted = mask == nullptr || mask[t] != 0;
    if (lane == 0) {
      if (token_rkl) token_rkl[t] = r;
      contrib = counted ? (double)r : 0.0;
    }
    if (G) {
      const int n = *n_count;
      const float scale = (counted && n > 0 && ids_ok) ? inv_tau / (float)n : 0.f;
      float* grow = G + (long long)t * K;
      for (int k = lane; k < K; k += 32)
        grow[k] = ls[k] > -INFINITY ? scale * expf(zs[k]) * (zs[k] - ls[k] - r) : 0.f;
    }
  }
  if (block_sums == nullptr) return;  // uniform across the block
  if (lane == 0) wsum[warp] = contrib;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < RKL_WARPS; ++w) s += wsum[w];
    block_sums[blockIdx.x] = s;
  }
}

// One warp per token: dH_t = g * sum_k G[t,k] W[idx_k], in 1024-column passes
// (acc holds the lane's 32 columns of the slice).
__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_dH_kernel(const uint16_t* __restrict__ W, const int32_t* __restrict__ idx,
                  const float* __restrict__ G, float grad_loss, int T, int d, int K, int V,
                  uint16_t* __restrict__ dH, int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * RKL_WARPS + warp;
  if (t >= T) return;
  const int32_t* irow = idx + (long long)t * K;
  const float* grow = G + (long long)t * K;
  for (int c0 = 0; c0 < d; c0 += 1024) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 32) {
      const int kk = k0 + lane;
      const int my_id = kk < K ? __ldg(irow + kk) : 0;
      const float my_g = kk < K ? __ldg(grow + kk) * grad_loss : 0.f;
      const int n = min(32, K - k0);
      for (int j = 0; j < n; ++j) {
        const int id = __shfl_sync(0xffffffffu, my_id, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (id < 0 || id >= V) {  // warp-uniform; the entry reads nothing
          if (lane == 0 && c0 == 0) record_error(status, DEV_ERR_INDEX_RANGE);
          continue;
        }
        if (g == 0.f) continue;  // masked token or dropped entry
        const uint16_t* wr = W + (long long)id * d;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = c0 + q * 256 + lane * 8;
          if (i < d) axpy8_bf16(acc + 8 * q, g, __ldg(reinterpret_cast<const uint4*>(wr + i)));
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
}

// ----------------------------------------------------------- radix sort by id
// Keys are ids; an id outside [0, V) sorts as V (a bucket nothing reads).
// `first`: keys come straight from topk_idx and the values are the positions.

__device__ __forceinline__ int radix_key(const int32_t* __restrict__ keys, int i, int V, int first) {
  const int k = __ldg(keys + i);
  return first ? ((k < 0 || k >= V) ? V : k) : k;
}

__global__ void __launch_bounds__(RADIX_THREADS)
    radix_hist_kernel(const int32_t* __restrict__ keys, int n, int V, int first, int shift,
                      int nbins, int n_tiles, unsigned* __restrict__ hist) {
  __shared__ unsigned cnt[RADIX_MAX_BINS];
  for (int b = threadIdx.x; b < nbins; b += RADIX_THREADS) cnt[b] = 0;
  __syncthreads();
  const int base = blockIdx.x * RADIX_TILE;
  for (int r = 0; r < RADIX_ROUNDS; ++r) {
    const int i = base + r * RADIX_THREADS + threadIdx.x;
    if (i < n) atomicAdd(&cnt[(radix_key(keys, i, V, first) >> shift) & (nbins - 1)], 1u);
  }
  __syncthreads();
  // digit-major, so that one exclusive scan gives every (digit, tile) offset
  for (int b = threadIdx.x; b < nbins; b += RADIX_THREADS)
    hist[(long long)b * n_tiles + blockIdx.x] = cnt[b];
}

// Exclusive scan of a[0, m) in three launches: per-block sums of SCAN_CHUNK
// entries, a one-block scan of those sums, then each block scans its chunk
// from its offset. Threads own SCAN_ITEMS consecutive entries.
constexpr int SCAN_ITEMS = 4;
constexpr int SCAN_CHUNK = SCAN_THREADS * SCAN_ITEMS;

// Exclusive scan across the block; returns this thread's offset, *total the sum.
__device__ __forceinline__ unsigned block_exclusive_scan(unsigned x, unsigned* total) {
  __shared__ unsigned wsums[SCAN_THREADS / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) wsums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    unsigned w = lane < SCAN_THREADS / 32 ? wsums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < SCAN_THREADS / 32) wsums[lane] = w;  // inclusive
  }
  __syncthreads();
  *total = wsums[SCAN_THREADS / 32 - 1];
  const unsigned before = warp ? wsums[warp - 1] : 0u;
  __syncthreads();  // wsums is reused by the next call
  return before + inc - x;
}

__global__ void __launch_bounds__(SCAN_THREADS)
    scan_reduce_kernel(const unsigned* __restrict__ a, long long m, unsigned* __restrict__ bsum) {
  const long long base = (long long)blockIdx.x * SCAN_CHUNK;
  unsigned s = 0;
#pragma unroll
  for (int j = 0; j < SCAN_ITEMS; ++j) {
    const long long i = base + j * SCAN_THREADS + threadIdx.x;  // coalesced
    if (i < m) s += a[i];
  }
  unsigned total;
  block_exclusive_scan(s, &total);
  if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

// In-place exclusive scan of a small array with one block.
__global__ void __launch_bounds__(SCAN_THREADS)
    scan_small_kernel(unsigned* __restrict__ a, int m) {
  unsigned carry = 0;
  for (int b = 0; b < m; b += SCAN_THREADS) {
    const int i = b + threadIdx.x;
    const unsigned x = i < m ? a[i] : 0u;
    unsigned total;
    const unsigned off = block_exclusive_scan(x, &total);
    if (i < m) a[i] = carry + off;
    carry += total;
  }
}

__global__ void __launch_bounds__(SCAN_THREADS)
    scan_apply_kernel(unsigned* __restrict__ a, long long m, const unsigned* __restrict__ bsum) {
  const long long base = (long long)blockIdx.x * SCAN_CHUNK + (long long)threadIdx.x * SCAN_ITEMS;
  unsigned v[SCAN_ITEMS];
  unsigned s = 0;
#pragma unroll
  for (int j = 0; j < SCAN_ITEMS; ++j) {
    v[j] = base + j < m ? a[base + j] : 0u;
    s += v[j];
  }
  unsigned total;
  unsigned run = bsum[blockIdx.x] + block_exclusive_scan(s, &total);
#pragma unroll
  for (int j = 0; j < SCAN_ITEMS; ++j) {
    if (base + j < m) a[base + j] = run;
    run += v[j];
  }
}

// Stable scatter of one tile: entries are ranked in position order within
// their digit (warp ranks from __match_any_sync, earlier warps' counts from
// shared memory, earlier rounds' counts in `run`).
__global__ void __launch_bounds__(RADIX_THREADS)
    radix_scatter_kernel(const int32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
                         int n, int V, int first, int shift, int nbins, int n_tiles,
                         const unsigned* __restrict__ offs, int32_t* __restrict__ keys_out,
                         int32_t* __restrict__ vals_out) {
  constexpr int NW = RADIX_THREADS / 32;
  __shared__ unsigned run[RADIX_MAX_BINS];
  __shared__ unsigned char wcnt[NW][RADIX_MAX_BINS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = threadIdx.x; b < nbins; b += RADIX_THREADS) {
    run[b] = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) wcnt[w][b] = 0;
  }
  __syncthreads();
  const int base = blockIdx.x * RADIX_TILE;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < RADIX_ROUNDS; ++r) {
    const int i = base + r * RADIX_THREADS + threadIdx.x;
    const bool valid = i < n;
    int key = 0, val = 0;
    if (valid) {
      key = radix_key(keys_in, i, V, first);
      val = first ? i : __ldg(vals_in + i);
    }
    const int digit = valid ? (key >> shift) & (nbins - 1) : nbins;  // invalid lanes group apart
    const unsigned peers = __match_any_sync(0xffffffffu, digit);
    const unsigned below = peers & lt_mask;
    const bool leader = below == 0u;
    if (valid && leader) wcnt[warp][digit] = (unsigned char)__popc(peers);
    __syncthreads();
    unsigned rank = 0;
    if (valid) {
      rank = run[digit] + (unsigned)__popc(below);
      for (int w = 0; w < warp; ++w) rank += wcnt[w][digit];
    }
    __syncthreads();
    if (valid && leader) {
      atomicAdd(&run[digit], (unsigned)__popc(peers));
      wcnt[warp][digit] = 0;
    }
    __syncthreads();
    if (valid) {
      const unsigned pos = offs[(long long)digit * n_tiles + blockIdx.x] + rank;
      keys_out[pos] = key;
      vals_out[pos] = val;
    }
  }
}

// bstart/bend (zeroed, V + 1 entries): the sorted range [bstart[v], bend[v]) of id v.
__global__ void bucket_bounds_kernel(const int32_t* __restrict__ keys, int n,
                                     int* __restrict__ bstart, int* __restrict__ bend) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int k = keys[i];
    if (i == 0 || keys[i - 1] != k) bstart[k] = i;
    if (i == n - 1 || keys[i + 1] != k) bend[k] = i + 1;
  }
}

// ------------------------------------------------------------------- dW
// Writes the sum for id v accumulated over this segment's part of its bucket:
// straight into dW when the whole bucket lies in the segment, else into the
// segment's partial row (slot 0: the bucket began in an earlier segment;
// slot 1: it began here and continues).
__device__ __forceinline__ void dW_flush(const float (&acc)[32], int v, int s, int s0, int s1,
                                         const int* __restrict__ bstart,
                                         const int* __restrict__ bend, int c0, int d, int V,
                                         float* __restrict__ dW, float* __restrict__ part,
                                         int accumulate, int lane) {
  if (v >= V) return;
  const bool first = bstart[v] < s0;
  const bool last = bend[v] > s1;
  float* dst;
  bool add = false;
  if (!first && !last) {
    dst = dW + (long long)v * d;
    add = accumulate != 0;
  } else {
    dst = part + (2ll * s + (first ? 0 : 1)) * d;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = c0 + q * 256 + lane * 8;
    if (i < d) {
      float4* p = reinterpret_cast<float4*>(dst + i);
      float4 a = make_float4(acc[8 * q + 0], acc[8 * q + 1], acc[8 * q + 2], acc[8 * q + 3]);
      float4 b = make_float4(acc[8 * q + 4], acc[8 * q + 5], acc[8 * q + 6], acc[8 * q + 7]);
      if (add) {
        const float4 x = p[0], y = p[1];
        a = make_float4(x.x + a.x, x.y + a.y, x.z + a.z, x.w + a.w);
        b = make_float4(y.x + b.x, y.y + b.y, y.z + b.z, y.w + b.w);
      }
      p[0] = a;
      p[1] = b;
    }
  }
}

// z for every (token, id) pair, vocabulary-major: one warp per segment of SEG
// sorted pairs. For each run of equal id the warp holds that row of W (a
// 1024-column slice per pass, in registers) and reads the rows of H of the
// run's tokens, RB per memory round trip; each pair's dot product is summed
// over the warp into shared memory, pass after pass. So every named row of W
// is read once per segment it appears in, and the per-pair traffic is rows of
// H (far smaller than W, mostly L2-resident). Pairs with an out-of-range id
// (sorted to the bucket V) get z = 0.
__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_z_segment_kernel(const uint16_t* __restrict__ H, const uint16_t* __restrict__ W,
                         const int32_t* __restrict__ keys, const int32_t* __restrict__ vals,
                         int n, int d, int K, int V, float* __restrict__ zbuf) {
  __shared__ float zacc_all[RKL_WARPS][SEG];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x * RKL_WARPS + warp;
  const int s0 = s * SEG;
  if (s0 >= n) return;  // no block-wide barrier below
  const int s1 = min(n, s0 + SEG);
  float* zacc = zacc_all[warp];
  for (int i = lane; i < SEG; i += 32) zacc[i] = 0.f;
  __syncwarp();
  for (int c0 = 0; c0 < d; c0 += 1024) {
    bool col_ok[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) col_ok[q] = c0 + q * 256 + lane * 8 < d;
    for (int i0 = s0; i0 < s1; i0 += 32) {
      const int i = i0 + lane;
      const int cnt = min(32, s1 - i0);
      const int my_v = i < s1 ? __ldg(keys + i) : -1;
      const int my_t = i < s1 ? __ldg(vals + i) / K : 0;
      const int prev_v = __shfl_up_sync(0xffffffffu, my_v, 1);
      const unsigned starts = __ballot_sync(0xffffffffu, lane < cnt && (lane == 0 || my_v != prev_v));
      for (int j = 0; j < cnt;) {  // one run of equal id per iteration (warp-uniform)
        const int v = __shfl_sync(0xffffffffu, my_v, j);
        const unsigned later = j < 31 ? starts & ~((2u << j) - 1u) : 0u;
        const int jend = later ? __ffs(later) - 1 : cnt;
        if (v < V) {
          uint4 wv[4];
          const uint16_t* wr = W + (long long)v * d;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = c0 + q * 256 + lane * 8;
            wv[q] = __ldg(reinterpret_cast<const uint4*>(wr + (c < d ? c : 0)));
          }
          for (int jj = j; jj < jend; jj += RB) {
            int row[RB];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
              const int p = jj + u;
              const int t = __shfl_sync(0xffffffffu, my_t, p & 31);
              row[u] = p < jend ? t : 0;
            }
            uint4 h[RB][4];
            load_slices(h, H, row, c0, d, lane);
#pragma unroll
            for (int u = 0; u < RB; ++u) {
              float a = 0.f;
#pragma unroll
              for (int q = 0; q < 4; ++q) a = col_ok[q] ? dot8_bf16(h[u][q], wv[q], a) : a;
              a = warp_sum_f(a);
              if (lane == 0 && jj + u < jend) zacc[i0 - s0 + jj + u] += a;
            }
          }
        }
        j = jend;
      }
    }
  }
  __syncwarp();
  for (int i = s0 + lane; i < s1; i += 32) zbuf[__ldg(vals + i)] = zacc[i - s0];
}

// One warp per segment of SEG sorted pairs. Pairs are taken 32 at a time
// (one per lane), split into runs of equal id; each run is summed RB pairs per
// memory round trip, and the sum is flushed when the id changes.
__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_dW_segment_kernel(const uint16_t* __restrict__ H, const int32_t* __restrict__ keys,
                          const int32_t* __restrict__ vals, const float* __restrict__ G,
                          float grad_loss, const int* __restrict__ bstart,
                          const int* __restrict__ bend, int n, int d, int K, int V,
                          float* __restrict__ dW, float* __restrict__ part, int accumulate) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x * RKL_WARPS + warp;
  const int s0 = s * SEG;
  if (s0 >= n) return;
  const int s1 = min(n, s0 + SEG);
  for (int c0 = 0; c0 < d; c0 += 1024) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    int cur = -1;
    for (int i0 = s0; i0 < s1; i0 += 32) {
      const int i = i0 + lane;
      const int cnt = min(32, s1 - i0);
      int my_v = -1, my_t = 0;
      float my_g = 0.f;
      if (i < s1) {
        my_v = __ldg(keys + i);
        const int f = __ldg(vals + i);
        my_t = f / K;
        my_g = __ldg(G + f) * grad_loss;
      }
      const int prev_v = __shfl_up_sync(0xffffffffu, my_v, 1);
      const unsigned starts = __ballot_sync(0xffffffffu, lane < cnt && (lane == 0 || my_v != prev_v));
      for (int j = 0; j < cnt;) {  // one run of equal id per iteration (warp-uniform)
        const int v = __shfl_sync(0xffffffffu, my_v, j);
        const unsigned later = j < 31 ? starts & ~((2u << j) - 1u) : 0u;
        const int jend = later ? __ffs(later) - 1 : cnt;
        if (v != cur) {
          if (cur >= 0)
            dW_flush(acc, cur, s, s0, s1, bstart, bend, c0, d, V, dW, part, accumulate, lane);
#pragma unroll
          for (int q = 0; q < 32; ++q) acc[q] = 0.f;
          cur = v;
        }
        for (int jj = j; jj < jend; jj += RB) {
          int row[RB];
          float g[RB];
#pragma unroll
          for (int u = 0; u < RB; ++u) {
            const int p = jj + u;
            const int t = __shfl_sync(0xffffffffu, my_t, p & 31);
            const float gg = __shfl_sync(0xffffffffu, my_g, p & 31);
            const bool use = p < jend && gg != 0.f && v < V;
            row[u] = use ? t : 0;
            g[u] = use ? gg : 0.f;
          }
          uint4 w[RB][4];
          load_slices(w, H, row, c0, d, lane);
#pragma unroll
          for (int u = 0; u < RB; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q) axpy8_bf16(acc + 8 * q, g[u], w[u][q]);
        }
        j = jend;
      }
    }
    dW_flush(acc, cur, s, s0, s1, bstart, bend, c0, d, V, dW, part, accumulate, lane);
  }
}

// One warp per vocabulary row: rows no pair names are zeroed (unless
// accumulating); rows whose bucket straddles segments get their partials
// summed in segment order.
__global__ void __launch_bounds__(RKL_WARPS * 32)
    rkl_dW_fixup_kernel(const int* __restrict__ bstart, const int* __restrict__ bend,
                        const float* __restrict__ part, int V, int d, float* __restrict__ dW,
                        int accumulate) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = blockIdx.x * RKL_WARPS + warp;
  if (v >= V) return;
  const int bs = bstart[v], be = bend[v];
  float* row = dW + (long long)v * d;
  if (be == bs) {
    if (!accumulate)
      for (int c = lane * 4; c < d; c += 128)
        *reinterpret_cast<float4*>(row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int sa = bs / SEG, sb = (be - 1) / SEG;
  if (sa == sb) return;  // written by its segment
  for (int c = lane * 4; c < d; c += 128) {
    float4 a = *reinterpret_cast<const float4*>(part + (2ll * sa + 1) * d + c);
    for (int s = sa + 1; s <= sb; ++s) {
      const float4 x = *reinterpret_cast<const float4*>(part + (2ll * s) * d + c);
      a = make_float4(a.x + x.x, a.y + x.y, a.z + x.z, a.w + x.w);
    }
    if (accumulate) {
      const float4 y = *reinterpret_cast<const float4*>(row + c);
      a = make_float4(y.x + a.x, y.y + a.y, y.z + a.z, y.w + a.w);
    }
    *reinterpret_cast<float4*>(row + c) = a;
  }
}

// ------------------------------------------------------------------- host

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

RklLayout rkl_layout(long long T, long long d, int K, long long V, size_t header) {
  RklLayout L{};
  L.n = T * K;
  int nbits = 0;
  while ((1ll << nbits) <= V) ++nbits;  // keys run up to V
  L.passes = (nbits + RADIX_MAX_BITS - 1) / RADIX_MAX_BITS;
  L.bits = (nbits + L.passes - 1) / L.passes;
  L.nbins = 1 << L.bits;
  L.n_tiles = (L.n + RADIX_TILE - 1) / RADIX_TILE;
  L.n_seg = (L.n + SEG - 1) / SEG;
  size_t o = header;
  L.off_bsum = o;
  o += al256((size_t)((T + RKL_WARPS - 1) / RKL_WARPS) * sizeof(double));
  L.off_G = o;
  o += al256((size_t)L.n * 4);
  L.off_z = o;
  o += al256((size_t)L.n * 4);
  for (int b = 0; b < 2; ++b) {
    L.off_keys[b] = o;
    o += al256((size_t)L.n * 4);
    L.off_vals[b] = o;
    o += al256((size_t)L.n * 4);
  }
  L.off_hist = o;
  o += al256((size_t)L.nbins * L.n_tiles * 4);
  L.off_scan = o;
  o += al256((size_t)((L.nbins * L.n_tiles + SCAN_CHUNK - 1) / SCAN_CHUNK) * 4);
  L.off_bstart = o;
  o += al256((size_t)(V + 1) * 4);
  L.off_bend = o;
  o += al256((size_t)(V + 1) * 4);
  L.off_part = o;
  o += al256((size_t)2 * L.n_seg * d * 4);
  L.total = o;
  return L;
}

template <typename T>
static T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

static int blocks_for(long long items, int per_block) {
  return (int)((items + per_block - 1) / per_block);
}

static cudaError_t launch_forward_kernel(const char* name, const int32_t* idx, const float* logit,
                                         const uint8_t* mask, int T, int K, int V, float inv_tau,
                                         const int* n_count, const float* zbuf, float* token_rkl,
                                         float* G, double* bsum, int* status,
                                         cudaStream_t stream) {
  // at most 8 warps x 512 ids x 8 bytes = 32 KB: within the default limit
  const size_t smem = RKL_WARPS * rkl_forward_smem_per_warp(K);
  return launch_kernel(name, rkl_forward_kernel, dim3(blocks_for(T, RKL_WARPS)),
                       dim3(RKL_WARPS * 32), smem, stream, idx, logit, mask, T, K, V, inv_tau,
                       n_count, zbuf, token_rkl, G, bsum, status);
}

// Stable sort of the (id, position) pairs by id and each id's range in the
// sorted list. *keys / *vals receive the sorted arrays (in the workspace).
static cudaError_t rkl_sort(const RklLayout& L, const int32_t* idx, int V, void* ws, int num_sms,
                            cudaStream_t stream, const int32_t** keys, const int32_t** vals) {
  cudaError_t e;
  const int n = (int)L.n;
  unsigned* hist = ws_at<unsigned>(ws, L.off_hist);
  const int32_t* kin = idx;
  const int32_t* vin = nullptr;
  int buf = 0;
  for (int p = 0; p < L.passes; ++p) {
    const int first = p == 0 ? 1 : 0;
    const int shift = p * L.bits;
    int32_t* kout = ws_at<int32_t>(ws, L.off_keys[buf]);
    int32_t* vout = ws_at<int32_t>(ws, L.off_vals[buf]);
    e = launch_kernel("radix_hist", radix_hist_kernel, dim3((unsigned)L.n_tiles),
                      dim3(RADIX_THREADS), 0, stream, kin, n, V, first, shift, L.nbins,
                      (int)L.n_tiles, hist);
    if (e != cudaSuccess) return e;
    const long long m = (long long)L.nbins * L.n_tiles;
    const int nb = blocks_for(m, SCAN_CHUNK);
    unsigned* bsum = ws_at<unsigned>(ws, L.off_scan);
    e = launch_kernel("scan_reduce", scan_reduce_kernel, dim3(nb), dim3(SCAN_THREADS), 0, stream,
                      (const unsigned*)hist, m, bsum);
    if (e != cudaSuccess) return e;
    e = launch_kernel("scan_small", scan_small_kernel, dim3(1), dim3(SCAN_THREADS), 0, stream,
                      bsum, nb);
    if (e != cudaSuccess) return e;
    e = launch_kernel("scan_apply", scan_apply_kernel, dim3(nb), dim3(SCAN_THREADS), 0, stream,
                      hist, m, (const unsigned*)bsum);
    if (e != cudaSuccess) return e;
    e = launch_kernel("radix_scatter", radix_scatter_kernel, dim3((unsigned)L.n_tiles),
                      dim3(RADIX_THREADS), 0, stream, kin, vin, n, V, first, shift, L.nbins,
                      (int)L.n_tiles, (const unsigned*)hist, kout, vout);
    if (e != cudaSuccess) return e;
    kin = kout;
    vin = vout;
    buf ^= 1;
  }
  int* bstart = ws_at<int>(ws, L.off_bstart);
  int* bend = ws_at<int>(ws, L.off_bend);
  e = cudaMemsetAsync(bstart, 0, L.off_part - L.off_bstart, stream);  // bstart and bend
  if (e != cudaSuccess) return e;
  e = launch_kernel("bucket_bounds", bucket_bounds_kernel,
                    dim3(std::max(1, std::min(num_sms * 8, blocks_for(n, 256)))), dim3(256), 0,
                    stream, kin, n, bstart, bend);
  if (e != cudaSuccess) return e;
  *keys = kin;
  *vals = vin;
  return cudaSuccess;
}

// count -> sort -> z per pair (segments) -> per-token RKL / grad_z / block sums.
static cudaError_t rkl_token_pass(const RklLayout& L, const uint16_t* H, const uint16_t* W,
                                  const int32_t* idx, const float* logit, const uint8_t* mask,
                                  int T, int d, int K, int V, float inv_tau, float* token_rkl,
                                  float* G, double* bsum, void* ws, int* status, int* n_count,
                                  int num_sms, cudaStream_t stream, const int32_t** keys,
                                  const int32_t** vals) {
  cudaError_t e = launch_kernel("rkl_count", rkl_count_kernel, dim3(std::min(num_sms, 64)),
                                dim3(256), 0, stream, mask, T, n_count);
  if (e != cudaSuccess) return e;
  if ((e = rkl_sort(L, idx, V, ws, num_sms, stream, keys, vals)) != cudaSuccess) return e;
  float* zbuf = ws_at<float>(ws, L.off_z);
  e = launch_kernel("rkl_z_segment", rkl_z_segment_kernel, dim3(blocks_for(L.n_seg, RKL_WARPS)),
                    dim3(RKL_WARPS * 32), 0, stream, H, W, *keys, *vals, (int)L.n, d, K, V, zbuf);
  if (e != cudaSuccess) return e;
  return launch_forward_kernel("rkl_forward", idx, logit, mask, T, K, V, inv_tau, n_count, zbuf,
                               token_rkl, G, bsum, status, stream);
}

cudaError_t rkl_forward(const RklLayout& L, const uint16_t* H, const uint16_t* W,
                        const int32_t* idx, const float* logit, const uint8_t* mask, int T, int d,
                        int K, int V, float inv_tau, float* token_rkl, float* grad_z, float* loss,
                        void* ws, int* status, int* n_count, int num_sms, cudaStream_t stream) {
  double* bsum = ws_at<double>(ws, L.off_bsum);
  const int32_t* keys = nullptr;
  const int32_t* vals = nullptr;
  cudaError_t e = rkl_token_pass(L, H, W, idx, logit, mask, T, d, K, V, inv_tau, token_rkl, grad_z,
                                 bsum, ws, status, n_count, num_sms, stream, &keys, &vals);
  if (e != cudaSuccess) return e;
  return launch_loss_finalize(bsum, blocks_for(T, RKL_WARPS), n_count, loss, stream);
}

cudaError_t rkl_backward(const RklLayout& L, const uint16_t* H, const uint16_t* W,
                         const int32_t* idx, const float* logit, const uint8_t* mask, int T, int d,
                         int K, int V, float inv_tau, const float* grad_z, float grad_loss,
                         uint16_t* dH, float* dW, int accumulate, void* ws, int* status,
                         int* n_count, int num_sms, cudaStream_t stream) {
  cudaError_t e;
  const int32_t* keys = nullptr;
  const int32_t* vals = nullptr;
  const float* G = grad_z;
  if (G == nullptr) {  // recompute dL/dz at the ids (the sort is reused for dW)
    float* Gw = ws_at<float>(ws, L.off_G);
    e = rkl_token_pass(L, H, W, idx, logit, mask, T, d, K, V, inv_tau, nullptr, Gw, nullptr, ws,
                       status, n_count, num_sms, stream, &keys, &vals);
    if (e != cudaSuccess) return e;
    G = Gw;
  } else if ((e = rkl_sort(L, idx, V, ws, num_sms, stream, &keys, &vals)) != cudaSuccess) {
    return e;
  }
  e = launch_kernel("rkl_dH", rkl_dH_kernel, dim3(blocks_for(T, RKL_WARPS)), dim3(RKL_WARPS * 32),
                    0, stream, W, idx, G, grad_loss, T, d, K, V, dH, status);
  if (e != cudaSuccess) return e;
  const int* bstart = ws_at<int>(ws, L.off_bstart);
  const int* bend = ws_at<int>(ws, L.off_bend);
  float* part = ws_at<float>(ws, L.off_part);
  e = launch_kernel("rkl_dW_segment", rkl_dW_segment_kernel,
                    dim3(blocks_for(L.n_seg, RKL_WARPS)), dim3(RKL_WARPS * 32), 0, stream, H, keys,
                    vals, G, grad_loss, bstart, bend, (int)L.n, d, K, V, dW, part, accumulate);
  if (e != cudaSuccess) return e;
  return launch_kernel("rkl_dW_fixup", rkl_dW_fixup_kernel, dim3(blocks_for(V, RKL_WARPS)),
                       dim3(RKL_WARPS * 32), 0, stream, bstart, bend, (const float*)part, V, d, dW,
                       accumulate);
}

}  // namespace kdkl
