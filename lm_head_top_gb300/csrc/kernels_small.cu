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
#include <float.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <type_traits>

#include "kdkl_internal.h"
#include "tc_primitives.cuh"

namespace kdkl {

// teacher_prep: a row of K cached entries is handled by L lanes (16 or 32) of
// a warp, lane l holding elements l*E .. l*E+E-1 of the row padded to
// N = L*E (a power of two >= K). The row is read from global memory once, into
// registers; the teacher softmax, its entropy term and the validation run
// there. The (id, p) pairs are then ordered by id with a bitonic sorting
// network on packed keys (id, original position): exchanges between
// positions closer than E stay inside a lane, the rest exchange keys with
// __shfl_xor_sync, and p follows through a per-row shared-memory slot
// indexed by the original position. Packed keys are distinct, so the network
// needs no tie rule.
constexpr int PREP_THREADS = 256;

template <int N>
struct Log2 {
  static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

template <bool WIDE>
struct PrepKey;
template <>
struct PrepKey<false> {  // id << log2(N) | position: V * N <= 2^32
  using T = uint32_t;
  static constexpr T pad = 0xffffffffu;
};
template <>
struct PrepKey<true> {  // id << 32 | position
  using T = unsigned long long;
  static constexpr T pad = ~0ull;
};

__device__ __forceinline__ uint32_t shfl_key(uint32_t v, int o) {
  return __shfl_xor_sync(0xffffffffu, v, o);
}
__device__ __forceinline__ unsigned long long shfl_key(unsigned long long v, int o) {
  return __shfl_xor_sync(0xffffffffu, v, o);
}

__device__ __forceinline__ uint32_t kmin(uint32_t a, uint32_t b) { return min(a, b); }
__device__ __forceinline__ uint32_t kmax(uint32_t a, uint32_t b) { return max(a, b); }
__device__ __forceinline__ unsigned long long kmin(unsigned long long a, unsigned long long b) {
  return min(a, b);
}
__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b) {
  return max(a, b);
}

// Sum / max over the L lanes of one row (xor offsets below L stay in the row).
template <int L>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int L>
__device__ __forceinline__ float row_max(float v) {
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// rowmap == nullptr: output row t is token t, and the kernel counts the mask
// into *n_count. Otherwise output row r (r < *n_count, set by the mask scan)
// is token rowmap[r], and rows from *n_count on are left unwritten.
template <int L, int E, bool WIDE>
__global__ void __launch_bounds__(PREP_THREADS)
    teacher_prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ logit,
                        const uint8_t* __restrict__ mask, const int32_t* __restrict__ labels,
                        const int* __restrict__ rowmap, int T, int K, int V, float inv_tau,
                        int vec_io, int32_t* __restrict__ sidx, float* __restrict__ sp,
                        float* __restrict__ ent, int* n_count, int* status) {
  using Key = typename PrepKey<WIDE>::T;
  constexpr int N = L * E;
  constexpr int LOGN = Log2<N>::value;
  constexpr int ROWS = PREP_THREADS / L;  // rows per block
  __shared__ float p_slot[ROWS * N];
  __shared__ int block_count;
  const int lane = threadIdx.x & 31;
  const int row = threadIdx.x / L;  // row slot in the block
  const int l = threadIdx.x % L;    // lane within the row
  const int t = blockIdx.x * ROWS + row;  // output row
  const bool live = t < (rowmap ? *n_count : T);
  const int src = live ? (rowmap ? __ldg(rowmap + t) : t) : 0;  // token read
  if (threadIdx.x == 0) block_count = 0;
  __syncthreads();

  // ---- one read of the row into registers
  int id[E];
  float a[E];
  const long long base = (long long)src * K;
  const long long obase = (long long)t * K;
  // 16-byte loads and stores when rows and pointers allow (host-checked)
  const bool vec4 = (E % 4 == 0) && vec_io != 0;
  if (vec4) {
#pragma unroll
    for (int j = 0; j < E; j += 4) {
      const int k = l * E + j;
      const bool in = live && k < K;  // all four in or all out (K % 4 == 0)
      const int4 iv = in ? __ldg(reinterpret_cast<const int4*>(idx + base + k)) : make_int4(0, 0, 0, 0);
      const float4 lv = in ? __ldg(reinterpret_cast<const float4*>(logit + base + k))
                           : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      id[j] = iv.x, id[j + 1] = iv.y, id[j + 2] = iv.z, id[j + 3] = iv.w;
      a[j] = lv.x * inv_tau, a[j + 1] = lv.y * inv_tau, a[j + 2] = lv.z * inv_tau,
      a[j + 3] = lv.w * inv_tau;
    }
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int k = l * E + j;
      const bool in = live && k < K;
      id[j] = in ? __ldg(idx + base + k) : 0;
      a[j] = in ? __ldg(logit + base + k) * inv_tau : -INFINITY;
    }
  }

  // ---- validation, max of a = logit / tau. Padding and the slots of a row
  // past T hold (id 0, -inf), which pass both checks.
  bool bad_id = false, bad_logit = false;
  float amax = -INFINITY;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    bad_id |= (uint32_t)id[j] >= (uint32_t)V;  // negative ids wrap above V
    bad_logit |= !(a[j] < INFINITY);           // NaN or +inf
    amax = fmaxf(amax, a[j]);
  }
  amax = row_max<L>(amax);
  const bool no_finite = !(amax > -INFINITY);
  {
    // one report per warp is enough: the status keeps the first error
    const bool idx_err = __any_sync(0xffffffffu, bad_id);
    const bool arg_err = __any_sync(0xffffffffu, bad_logit || (live && no_finite));
    if (lane == 0 && idx_err) record_error(status, DEV_ERR_INDEX_RANGE);
    if (lane == 0 && arg_err) record_error(status, DEV_ERR_INVALID_ARG);
  }

  // ---- teacher softmax over the K entries and sum p log p (0 log 0 = 0).
  // With d = a - max and S = sum exp(d): p = exp(d) / S and
  // sum p log p = sum exp(d) d / S - log S. An entry at -inf has exp(d) = 0
  // and its d is clamped to -FLT_MAX, so it adds exactly 0. A row without a
  // finite entry (an error, reported above) gets p = 0 and 0.
  // __expf, __logf and a reciprocal (a few ulp; the loss tolerance is 1e-3
  // relative): the kernel is bound by its integer pipe (the sort), and every
  // instruction saved here counts.
  const float amax_s = no_finite ? 0.f : amax;
  float e[E];
  float sum = 0.f, ed = 0.f;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const float dj = a[j] - amax_s;
    e[j] = __expf(dj);  // 0 for -inf and padding
    sum += e[j];
    ed = fmaf(e[j], fmaxf(dj, -FLT_MAX), ed);
  }
  sum = row_sum<L>(sum);
  ed = row_sum<L>(ed);
  const float inv_sum = no_finite ? 0.f : 1.0f / sum;
  const float h = no_finite ? 0.f : fmaf(ed, inv_sum, -__logf(sum));
  float* ps = p_slot + row * N;
#pragma unroll
  for (int j = 0; j < E; ++j) ps[l * E + j] = e[j] * inv_sum;

  // ---- order the entries by id: bitonic network over packed keys
  Key key[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int k = l * E + j;
    const bool in = live && k < K;
    key[j] = !in ? PrepKey<WIDE>::pad
                 : (WIDE ? (((Key)(uint32_t)id[j]) << 32) | (Key)k
                         : (((Key)(uint32_t)id[j]) << LOGN) | (Key)k);
  }
  // Merge form of the bitonic network: each merge of two ascending runs of
  // size/2 first compares position i with its mirror i ^ (size - 1), then
  // half-cleans with strides size/4 .. 1. Every compare-exchange puts the
  // smaller key at the lower position, so no step depends on a direction
  // bit: an in-lane exchange is a min and a max, a cross-lane one a shuffle
  // and a min or a max.
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
    if (size <= E) {  // mirror inside the lane: slots j and j ^ (size - 1)
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int jm = j ^ (size - 1);
        if ((j & (size >> 1)) == 0) {
          const Key x = key[j], y = key[jm];
          key[j] = kmin(x, y);
          key[jm] = kmax(x, y);
        }
      }
    } else {  // mirror in lane l ^ (size / E - 1), slot E - 1 - j
      const bool lo = (l & (size / (2 * E))) == 0;
      Key o[E];
#pragma unroll
      for (int j = 0; j < E; ++j) o[j] = shfl_key(key[E - 1 - j], size / E - 1);
#pragma unroll
      for (int j = 0; j < E; ++j)
        key[j] = lo ? kmin(o[j], key[j]) : kmax(o[j], key[j]);
    }
#pragma unroll
    for (int stride = size >> 2; stride > 0; stride >>= 1) {
      if (stride >= E) {  // partner in lane l ^ (stride / E), same slot
        const bool lo = (l & (stride / E)) == 0;
#pragma unroll
        for (int j = 0; j < E; ++j) {
          const Key o = shfl_key(key[j], stride / E);
          key[j] = lo ? kmin(o, key[j]) : kmax(o, key[j]);
        }
      } else {  // partner in this lane, slot j ^ stride
#pragma unroll
        for (int j = 0; j < E; ++j) {
          if ((j & stride) == 0) {
            const Key x = key[j], y = key[j + stride];
            key[j] = kmin(x, y);
            key[j + stride] = kmax(x, y);
          }
        }
      }
    }
  }
  __syncwarp();

  // ---- write the sorted (id, p) row
  if (live) {
    int32_t* so = sidx + obase;
    float* po = sp + obase;
    int oid[E];
    float op[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int pos = (int)(key[j] & (Key)(WIDE ? 0xffffffffu : (uint32_t)(N - 1)));
      oid[j] = (int32_t)(uint32_t)(WIDE ? (key[j] >> 32) : (key[j] >> LOGN));
      op[j] = ps[pos & (N - 1)];
    }
    if (vec4) {
#pragma unroll
      for (int j = 0; j < E; j += 4) {
        const int k = l * E + j;
        if (k < K) {
          *reinterpret_cast<int4*>(so + k) = make_int4(oid[j], oid[j + 1], oid[j + 2], oid[j + 3]);
          *reinterpret_cast<float4*>(po + k) = make_float4(op[j], op[j + 1], op[j + 2], op[j + 3]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int k = l * E + j;
        if (k < K) {
          so[k] = oid[j];
          po[k] = op[j];
        }
      }
    }
    if (l == 0) {
      if (labels && (labels[src] < 0 || labels[src] >= V)) record_error(status, DEV_ERR_INDEX_RANGE);
      if (ent) ent[t] = h;
    }
  }
  if (rowmap) return;  // N came from the mask scan
  const bool counted = live && l == 0 && (mask == nullptr || mask[t] != 0);
  const uint32_t cnt = __popc(__ballot_sync(0xffffffffu, counted));
  if (lane == 0 && cnt) atomicAdd(&block_count, (int)cnt);
  __syncthreads();
  if (threadIdx.x == 0 && block_count) atomicAdd(n_count, block_count);
}

constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_WARPS = COMBINE_THREADS / 32;
constexpr int COMBINE_TOK = 32;  // tokens per block: one per lane

// exp2((x - m) * c) for x <= m, exactly 1 when x == m (both -inf included)
__device__ __forceinline__ float rescale2(float x, float m, float c) {
  return x == m ? 1.f : exp2f((x - m) * c);
}

// lse_combine: per token, merge the vocabulary splits' partials (max m_s,
// sum_s exp((z - m_s) / tau) over the split, and the teacher-weighted logit
// sum d_s) into lse and KL, plus one fp64 sum of m_t KL_t per block. A block
// takes 32 tokens (one per lane); its 8 warps take every 8th split each,
// with a running max, and warp 0 merges the 8 partials in warp order: the
// order of every sum is fixed, so results are deterministic. invmap: token
// t's row among the partials (-1: masked, never computed: lse and KL read 0),
// or nullptr (row t).
// MIX adds the temperature-1 sums and the label logit: the per-token loss is
// kl_w KL + ce_w (lse_1 - z_label).
template <bool MIX>
__global__ void __launch_bounds__(COMBINE_THREADS)
    lse_combine_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                       const float* __restrict__ pd, const float* __restrict__ ps1,
                       const float* __restrict__ pzl, int nsplit, int T,
                       const float* __restrict__ ent, const uint8_t* __restrict__ mask,
                       const int* __restrict__ invmap, float cl2, float inv_tau, float kl_w,
                       float ce_w, float* __restrict__ lse, float* __restrict__ lse1,
                       float* __restrict__ token_loss, double* __restrict__ block_sums) {
  constexpr float L2E = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int t = blockIdx.x * COMBINE_TOK + lane;
  const int r = t < T ? (invmap ? invmap[t] : t) : -1;
  float M = -INFINITY, S = 0.f, D = 0.f, S1 = 0.f, Z = 0.f;
  if (r >= 0) {
#pragma unroll 4
    for (int s = w; s < nsplit; s += COMBINE_WARPS) {
      const long long o = (long long)s * T + r;
      const float m = pm[o];
      const float nm = fmaxf(M, m);
      S = S * rescale2(M, nm, cl2) + ps[o] * rescale2(m, nm, cl2);
      D += pd[o];
      if (MIX) {
        S1 = S1 * rescale2(M, nm, L2E) + ps1[o] * rescale2(m, nm, L2E);
        Z += pzl[o];
      }
      M = nm;
    }
  }
  __shared__ float part[MIX ? 5 : 3][COMBINE_WARPS][COMBINE_TOK];
  part[0][w][lane] = M;
  part[1][w][lane] = S;
  part[2][w][lane] = D;
  if (MIX) {
    part[3][w][lane] = S1;
    part[4][w][lane] = Z;
  }
  __syncthreads();
  if (w != 0) return;
  double contrib = 0.0;
  if (t < T) {
    float l = 0.f, l1 = 0.f, tok = 0.f;
    if (r >= 0) {
      M = -INFINITY;
#pragma unroll
      for (int i = 0; i < COMBINE_WARPS; ++i) M = fmaxf(M, part[0][i][lane]);
      S = D = S1 = Z = 0.f;
#pragma unroll
      for (int i = 0; i < COMBINE_WARPS; ++i) {
        const float mi = part[0][i][lane];
        S += part[1][i][lane] * rescale2(mi, M, cl2);
        D += part[2][i][lane];
        if (MIX) {
          S1 += part[3][i][lane] * rescale2(mi, M, L2E);
          Z += part[4][i][lane];
        }
      }
      l = M * inv_tau + logf(S);
      const float kl = ent[r] - D * inv_tau + l;
      if (MIX) {
        l1 = M + logf(S1);
        tok = kl_w * kl + ce_w * (l1 - Z);
      } else {
        tok = kl;
      }
    }
    lse[t] = l;
    if (MIX) lse1[t] = l1;
    if (token_loss) token_loss[t] = tok;
    if (invmap ? r >= 0 : (mask == nullptr || mask[t] != 0)) contrib = (double)tok;
  }
  // fixed-shape butterfly over the warp: deterministic
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) contrib += __shfl_xor_sync(0xffffffffu, contrib, o);
  if (lane == 0) block_sums[blockIdx.x] = contrib;
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

// out row t = bf16(in row invmap[t]), or zeros when invmap[t] < 0; invmap
// nullptr: row t. One block per row at a time, d4 = d / 4 float4 per row.
__global__ void f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out, int T,
                                   int d4, const int* __restrict__ invmap) {
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const int r = invmap ? __ldg(invmap + t) : t;
    uint2* o = out + (long long)t * d4;
    if (r < 0) {
      for (int c = threadIdx.x; c < d4; c += blockDim.x) o[c] = make_uint2(0u, 0u);
      continue;
    }
    const float4* src = in + (long long)r * d4;
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 v = src[c];
      o[c] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
  }
}

// Compaction of the counted tokens, one block: rowmap[r] = the r-th token
// with mask != 0 (in order), invmap[t] = its r or -1, *n_count = N. The mask
// is taken in tiles of 32 x 1024 tokens: warp w owns 32 consecutive 32-token
// chunks of a tile, counts them with ballots (lane j keeps chunk j's count),
// a block scan gives each chunk its first row, and a second pass writes the
// maps. Loads and invmap stores are coalesced 32-token pieces.
constexpr int SCAN_THREADS = 1024;
__global__ void __launch_bounds__(SCAN_THREADS)
    mask_scan_kernel(const uint8_t* __restrict__ mask, int T, int* __restrict__ rowmap,
                     int* __restrict__ invmap, int* __restrict__ n_count) {
  __shared__ int warp_base[SCAN_THREADS / 32];
  __shared__ int tile_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  constexpr long long TILE = 32LL * SCAN_THREADS;  // tokens per tile
  int base = 0;                                     // rows before this tile
  for (long long t0 = 0; t0 < T; t0 += TILE) {
    const long long w0 = t0 + (long long)warp * 32 * 32;  // this warp's first token
    int my_count = 0;                                     // chunk `lane` of this warp
    for (int j = 0; j < 32; ++j) {
      const long long t = w0 + (long long)j * 32 + lane;
      const bool on = t < T && mask[t] != 0;
      const int c = __popc(__ballot_sync(0xffffffffu, on));
      if (lane == j) my_count = c;
    }
    int incl = my_count;  // chunks of this warp, in order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_base[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int wt = warp_base[lane];
      int wi = wt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      warp_base[lane] = wi - wt;
      if (lane == 31) tile_total = wi;
    }
    __syncthreads();
    const int chunk_first = base + warp_base[warp] + incl - my_count;  // chunk `lane`'s first row
    for (int j = 0; j < 32; ++j) {
      const long long t = w0 + (long long)j * 32 + lane;
      const bool on = t < T && mask[t] != 0;
      const uint32_t b = __ballot_sync(0xffffffffu, on);
      const int first = __shfl_sync(0xffffffffu, chunk_first, j);
      if (t < T) {
        const int r = first + __popc(b & below);
        if (on) rowmap[r] = (int)t;
        invmap[t] = on ? r : -1;
      }
    }
    base += tile_total;
    __syncthreads();  // warp_base and tile_total are rewritten by the next tile
  }
  if (threadIdx.x == 0) *n_count = base;
}

// Hc row r = H row rowmap[r] for r < N; rows N .. (N rounded up to `round`)
// are zeroed (the partial last tile the GEMMs read). One block per row at a
// time, 16-byte pieces.
__global__ void gather_rows_kernel(const uint4* __restrict__ H, int row16,
                                   const int* __restrict__ rowmap, const int* __restrict__ n_count,
                                   long long rows_cap, int round, uint4* __restrict__ Hc) {
  const long long N = *n_count;
  long long end = (N + round - 1) / round * round;
  if (end > rows_cap) end = rows_cap;
  for (long long r = blockIdx.x; r < end; r += gridDim.x) {
    uint4* o = Hc + r * row16;
    if (r >= N) {
      for (int c = threadIdx.x; c < row16; c += blockDim.x) o[c] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* src = H + (long long)__ldg(rowmap + r) * row16;
    for (int c = threadIdx.x; c < row16; c += blockDim.x) o[c] = src[c];
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
    const uint32_t mask = __ballot_sync(0xffffffffu, keep);  // this pass of 32 has read its keys
    if (keep) keys[w + __popc(mask & below)] = k;
    w += __popc(mask);
  }
  __syncwarp();
  return w;
}

// One warp per row; `rows_per_block` warps share the block's shared memory,
// cap entries each (a power of two, at least K + 32). Split s of row t kept
// unit_cnt[s, t] entries (at most K) at the start of its [s, t] slot.
__global__ void __launch_bounds__(256)
    topk_merge_kernel(const float* __restrict__ unit_val, const int32_t* __restrict__ unit_id,
                      const int* __restrict__ unit_cnt, const uint32_t* __restrict__ row_key,
                      int nsplit, int T, int K, int cap, int32_t* __restrict__ out_id,
                      float* __restrict__ out_val) {
  extern __shared__ unsigned long long mkeys_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;  // whole warp leaves together; no block-wide barrier below
  unsigned long long* mkeys = mkeys_all + (size_t)warp * cap;
  const uint32_t floor_key = row_key[t];
  const uint32_t below = (1u << lane) - 1u;
  int m = 0;
  unsigned long long cut = ~0ull;  // every kept key is below it
  constexpr int BATCH = 8;  // splits whose entries are loaded together
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int c_lane = s0 + lane < nsplit ? min(unit_cnt[(long long)(s0 + lane) * T + t], K) : 0;
    const int nb = min(32, nsplit - s0);
    for (int j0 = 0; j0 < nb; j0 += BATCH) {
      // the first 32 entries of BATCH splits in flight at once; longer lists
      // (up to K) are finished split by split below
      float vb[BATCH];
      int32_t ib[BATCH];
      int cb[BATCH];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        cb[b] = __shfl_sync(0xffffffffu, c_lane, (j0 + b) & 31);
        if (j0 + b >= nb) cb[b] = 0;
        const long long o = ((long long)(s0 + j0 + b) * T + t) * K + lane;
        vb[b] = lane < cb[b] ? unit_val[o] : -INFINITY;
        ib[b] = lane < cb[b] ? unit_id[o] : -1;
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        for (int k0 = 0; k0 < cb[b]; k0 += 32) {
          float v = vb[b];
          int32_t id = ib[b];
          if (k0 > 0) {
            const long long o = ((long long)(s0 + j0 + b) * T + t) * K + k0 + lane;
            v = k0 + lane < cb[b] ? unit_val[o] : -INFINITY;
            id = k0 + lane < cb[b] ? unit_id[o] : -1;
          }
          const uint32_t ok = merge_order_key(v);
          const unsigned long long key = ((unsigned long long)(~ok) << 32) | (uint32_t)id;
          const bool keep = id >= 0 && ok >= floor_key && key < cut;
          // A full buffer keeps only its K best before taking more (ids are
          // distinct within a row, as merge_select_k needs); the largest of
          // those K keys then bounds every later entry: one with a larger key
          // (a smaller logit, or the same logit and a larger id) cannot enter.
          if (m + 32 > cap) {
            __syncwarp();
            m = merge_select_k(mkeys, m, K);
            unsigned long long mx = 0ull;
            for (int e = lane; e < m; e += 32) mx = mkeys[e] > mx ? mkeys[e] : mx;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const unsigned long long y = __shfl_xor_sync(0xffffffffu, mx, o);
              mx = y > mx ? y : mx;
            }
            cut = mx;
          }
          const bool take = keep && key < cut;
          const uint32_t mask = __ballot_sync(0xffffffffu, take);
          if (take) mkeys[m + __popc(mask & below)] = key;
          m += __popc(mask);
        }
      }
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

namespace {

template <int L, int E>
cudaError_t launch_prep(bool wide, const int32_t* idx, const float* logit, const uint8_t* mask,
                        const int32_t* labels, const int* rowmap, int T, int K, int V,
                        float inv_tau, int vec_io, int32_t* sidx,
                        float* sp, float* ent, int* n_count, int* status, cudaStream_t stream) {
  constexpr int rows = PREP_THREADS / L;
  const dim3 grid((T + rows - 1) / rows);
  if (wide)
    return launch_kernel("teacher_prep", teacher_prep_kernel<L, E, true>, grid, dim3(PREP_THREADS),
                         0, stream, idx, logit, mask, labels, rowmap, T, K, V, inv_tau, vec_io,
                         sidx, sp, ent, n_count, status);
  return launch_kernel("teacher_prep", teacher_prep_kernel<L, E, false>, grid, dim3(PREP_THREADS),
                       0, stream, idx, logit, mask, labels, rowmap, T, K, V, inv_tau, vec_io,
                       sidx, sp, ent, n_count, status);
}

}  // namespace

cudaError_t launch_teacher_prep(const int32_t* idx, const float* logit, const uint8_t* mask,
                                const int32_t* labels, const int* rowmap, int T, int K, int V,
                                float inv_tau, int32_t* sidx, float* sp, float* ent, int* n_count,
                                int* status, cudaStream_t stream) {
  // Rows of up to 128 entries take 16 lanes (two rows per warp), longer rows
  // a whole warp. Packed 32-bit keys when every id fits beside the position.
  int n = 16;
  while (n < K) n <<= 1;
  // KDKL_PREP_WIDE=1 (test hook, read per call) takes the 64-bit keys anyway.
  const char* force_wide = getenv("KDKL_PREP_WIDE");
  const bool wide = (unsigned long long)V * (unsigned long long)n >= (1ull << 32) ||
                    (force_wide && force_wide[0] == '1');
  auto a16 = [](const void* q) { return ((uintptr_t)q & 15u) == 0; };
  const int vec_io = (K % 4 == 0 && a16(idx) && a16(logit) && a16(sidx) && a16(sp)) ? 1 : 0;
#define KDKL_PREP(L, E)                                                                     \
  launch_prep<L, E>(wide, idx, logit, mask, labels, rowmap, T, K, V, inv_tau, vec_io, sidx,   \
                    sp, ent, n_count, status, stream)
  if (K <= 16) return KDKL_PREP(16, 1);
  if (K <= 32) return KDKL_PREP(16, 2);
  if (K <= 64) return KDKL_PREP(16, 4);
  if (K <= 128) return KDKL_PREP(16, 8);
  if (K <= 256) return KDKL_PREP(32, 8);
  return KDKL_PREP(32, 16);
#undef KDKL_PREP
}

int combine_blocks(int T) { return (T + COMBINE_TOK - 1) / COMBINE_TOK; }

cudaError_t launch_lse_combine(const float* pm, const float* ps, const float* pd, int nsplit, int T,
                               const float* ent, const uint8_t* mask, const int* invmap,
                               float cl2, float inv_tau, float* lse, float* token_kl,
                               double* block_sums, cudaStream_t stream) {
  return launch_kernel("lse_combine", lse_combine_kernel<false>, dim3(combine_blocks(T)),
                       dim3(COMBINE_THREADS), 0, stream, pm, ps, pd, nullptr, nullptr, nsplit, T,
                       ent, mask, invmap, cl2, inv_tau, 1.f, 0.f, lse, nullptr, token_kl,
                       block_sums);
}

cudaError_t launch_lse_combine_mix(const float* pm, const float* ps, const float* pd,
                                   const float* ps1, const float* pzl, int nsplit, int T,
                                   const float* ent, const uint8_t* mask, const int* invmap,
                                   float cl2, float inv_tau, float kl_w, float ce_w, float* lse,
                                   float* lse1, float* token_loss, double* block_sums,
                                   cudaStream_t stream) {
  return launch_kernel("lse_combine_mix", lse_combine_kernel<true>, dim3(combine_blocks(T)),
                       dim3(COMBINE_THREADS), 0, stream, pm, ps, pd, ps1, pzl, nsplit, T, ent,
                       mask, invmap, cl2, inv_tau, kl_w, ce_w, lse, lse1, token_loss, block_sums);
}

cudaError_t launch_loss_finalize(const double* block_sums, int nblocks, const int* n_count,
                                 float* loss, cudaStream_t stream) {
  return launch_kernel("loss_finalize", loss_finalize_kernel, dim3(1), dim3(1024), 0, stream,
                       block_sums, nblocks, n_count, loss);
}

// Merge buffer entries per row: room for every split's list when that is at
// most 2048 entries, else 2048 (the buffer is cut back to the K best when full).
int topk_merge_p2(int nsplit, int K) {
  int p2 = 64;
  while (p2 < nsplit * K && p2 < 2048) p2 <<= 1;
  while (p2 < K + 32) p2 <<= 1;
  return p2;
}

cudaError_t launch_topk_merge(const float* unit_val, const int32_t* unit_id, const int* unit_cnt,
                              const uint32_t* row_key, int nsplit, int T, int K, int32_t* out_id,
                              float* out_val, cudaStream_t stream) {
  const int cap = topk_merge_p2(nsplit, K);  // <= 2048 entries, 16 KB per warp
  const int warps = std::max(1, std::min(8, 6144 / cap));  // <= 48 KB of shared memory
  return launch_kernel("topk_merge", topk_merge_kernel, dim3((T + warps - 1) / warps),
                       dim3(32 * warps), (size_t)warps * cap * sizeof(unsigned long long), stream,
                       unit_val, unit_id, unit_cnt, row_key, nsplit, T, K, cap, out_id, out_val);
}

cudaError_t launch_mask_scan(const uint8_t* mask, int T, int* rowmap, int* invmap, int* n_count,
                             cudaStream_t stream) {
  return launch_kernel("mask_scan", mask_scan_kernel, dim3(1), dim3(SCAN_THREADS), 0, stream, mask,
                       T, rowmap, invmap, n_count);
}

cudaError_t launch_gather_rows(const uint16_t* H, int d, const int* rowmap, const int* n_count,
                               long long rows_cap, int round, uint16_t* Hc, int num_sms,
                               cudaStream_t stream) {
  const int row16 = d / 8;  // 16-byte pieces per bf16 row (d % 8 == 0)
  return launch_kernel("gather_rows", gather_rows_kernel, dim3((unsigned)num_sms * 8), dim3(256), 0,
                       stream, reinterpret_cast<const uint4*>(H), row16, rowmap, n_count, rows_cap,
                       round, reinterpret_cast<uint4*>(Hc));
}

cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, long long n, int d,
                               const int* invmap, int num_sms, cudaStream_t stream) {
  const int T = (int)(n / d);  // n = T * d, d a multiple of 8
  const int blocks = std::max(1, std::min(T, num_sms * 8));
  return launch_kernel("f32_to_bf16", f32_to_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0,
                       stream, reinterpret_cast<const float4*>(in), reinterpret_cast<uint2*>(out),
                       T, d / 4, invmap);
}

}  // namespace kdkl
