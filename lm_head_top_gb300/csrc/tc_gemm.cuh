// Persistent, warp-specialised tcgen05 GEMM for the fused KL loss, with the
// three epilogues the method needs:
//
//   EPI_LSE   forward: logits tile S = H_tile . W_tile^T lives only in TMEM;
//             each epilogue thread owns one token row and folds the tile into
//             a running max / sum of exp2 (the logsumexp) and into
//             sum_k p_k z[idx_k] for the teacher ids that fall in the tile.
//             Writes one (max, sum, dot) partial per (row, vocab split).
//   EPI_GRAD  backward: recompute S, form (softmax - P) * m / (tau N) * g in
//             the epilogue and store it as bf16 into the chunk buffer.
//   EPI_STORE plain fp32 output (dH and dW GEMMs), store or add.
//   EPI_TOPK  teacher cache producer: per-row candidate lists above a running
//             admission threshold, compacted to the row's top-K per split.
//   EPI_LSE_MIX / EPI_GRAD_MIX  the soft KL mixed with a hard-label CE.
//
// Roles per CTA (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and
// TMEM owner, warps 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
// By default two CTAs of a cluster share a 256 x 256 tile (tcgen05
// cta_group::2; PAIR); otherwise tiles are 128 x BN. The K step is 64 deep,
// with as many shared-memory stages as fit in ~200 KB (6 for pairs), and two
// fp32 accumulators in TMEM so the epilogue of one tile overlaps the MMAs of
// the next.
//
// Source of the method: "Making knowledge distillation cheap enough to run at
// scale", section "Two system changes" (the fused, chunked KL: each chunk's
// projection is folded into the running loss and discarded, then computed
// again in backward); the same in "Efficient knowledge distillation for LLMs:
// offline top-K logits and a fused chunked KL loss", section "Two systemic
// changes for scalable distillation".
#pragma once

#include <cuda_bf16.h>

#include "tc_primitives.cuh"

namespace kdkl {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int GEMM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;  // two accumulators of up to 256 fp32 columns
// MN-major operands arrive as 64-element-wide atoms of BK rows each.
constexpr uint32_t MN_ATOM_BYTES = BK * 128;
// N tile of the logit GEMMs (vocabulary direction).
constexpr int LOGIT_BN = 256;

// Shared-memory plan for an MMA tile of TILE_M x BN. With PAIR, two CTAs of a
// cluster share one 256 x BN tile: each holds 128 rows of A and BN/2 rows of B
// (so half the B bytes per CTA) and its own 128 x BN accumulator. As many
// 64-deep stages as fit in ~200 KB, then the barriers.
template <int BN, bool PAIR>
struct TileCfg {
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64..256 in steps of 64");
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows held by one CTA
  static constexpr int B_STAGE_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE_BYTES > 8 ? 8 : (200 * 1024) / STAGE_BYTES;
  // full, empty, tmem full x2, tmem empty x2, drain, unit-slot full / empty
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * 4;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*alignment slack*/ + 512;
};

enum { EPI_LSE = 0, EPI_GRAD = 1, EPI_STORE = 2, EPI_TOPK = 3, EPI_LSE_MIX = 4, EPI_GRAD_MIX = 5 };

// Work decomposition: `units` = m_tiles * nsplit. A unit is one m-tile and one
// split (a contiguous range of n-tiles). Units are numbered group by group:
// the m-tiles form groups of `group_m`; inside a group the m-tile runs
// fastest, then the split. Units are handed out in that order while the
// kernel runs (an atomic counter; see `counter`), so the units in flight at
// any moment are a window of consecutive numbers: a few splits of one group's
// m-tiles. Their B tiles are read from DRAM about once per group and their
// A rows (group_m m-tiles) stay in L2 for the group's duration, however the
// CTAs' speeds differ. group_m == 1 gives m-major order (every split of an
// m-tile, then the next m-tile).
struct GemmShape {
  int m_tiles, n_tiles, nsplit, group_m, units;
  int k_blocks;
  int a_m0, a_k0;  // A coordinate offsets (rows M / reduction K)
  int b_n0, b_k0;  // B coordinate offsets (rows N / reduction K)
  // Failure-detection test only: the producer issues nothing, so the MMA
  // warp's first wait runs out (after kInjectedWaitLimitNs) and the block
  // unwinds through its error path. Never set in normal calls.
  int inject_stall;
  // Nonzero: split 0 of every m-tile runs first (units 0 .. m_tiles-1), then
  // the groups over splits 1.. . The top-K producer uses it so that a row's
  // other splits start from the threshold its first split published.
  int first_group;
  // When > 0 (with first_group): split 0 covers n-tiles [0, first_ntiles)
  // and splits 1.. share the rest evenly; 0: every split gets an even share.
  int first_ntiles;
  // Unit counter for this launch (zero before it starts): the leader CTA's
  // producer takes the next unit with atomicAdd. nullptr: static round-robin
  // (CTA group g takes units g, g + groups, ...), kept to compare schedules.
  int* counter;
  // Token rows counted on the device (masked tokens compacted away): when
  // non-null, this launch's live extent along dyn_dim (0: the M rows of A,
  // 1: the K reduction) is clamp(*dyn_rows - dyn_base, 0, dyn_cap), and
  // m_tiles / units or k_blocks shrink to it before any role starts.
  const int* dyn_rows;
  int dyn_base, dyn_cap, dyn_dim;
  // Nonzero (B MN-major only): the last n-tile holds at most BN/2 columns of
  // B (d = 2880 is 11 tiles of 256 and 64 columns), so its MMAs run N = BN/2
  // and each CTA copies half of its B rows: half the padded work and B bytes.
  int narrow_last;
};

// n-tile range [nb, ne) of split s.
__device__ __forceinline__ void split_range(const GemmShape& sh, int s, int& nb, int& ne) {
  if (sh.first_ntiles > 0 && sh.nsplit > 1) {
    if (s == 0) {
      nb = 0;
      ne = sh.first_ntiles;
      return;
    }
    const long long rest = sh.n_tiles - sh.first_ntiles;
    nb = sh.first_ntiles + (int)(((long long)(s - 1) * rest) / (sh.nsplit - 1));
    ne = sh.first_ntiles + (int)(((long long)s * rest) / (sh.nsplit - 1));
    return;
  }
  nb = (int)(((long long)s * sh.n_tiles) / sh.nsplit);
  ne = (int)(((long long)(s + 1) * sh.n_tiles) / sh.nsplit);
}

struct EpiParams {
  // EPI_LSE and EPI_GRAD
  const int* rowmap;    // compacted row -> caller's token (lse, mask, labels), or nullptr
  const int32_t* sidx;  // [T, K] teacher ids sorted ascending per row
  const float* sp;      // [T, K] teacher probabilities in the same order
  int K;
  int T;
  int row0;     // first token row of this launch (EPI_GRAD)
  int rows;     // token rows in this launch
  int col0;     // first vocabulary id of this launch
  int cols;     // vocabulary columns in this launch
  float cl2;    // log2(e) / tau
  // EPI_LSE
  float* pm;  // [nsplit, T] running max of z
  float* ps;  // [nsplit, T] sum of exp2((z - max) * cl2)
  float* pd;  // [nsplit, T] sum_k p_k z[idx_k]
  // EPI_GRAD
  const float* lse;
  const uint8_t* mask;  // may be null (all tokens count)
  const int* n_count;   // number of counted tokens N
  float g_over_tau;
  uint16_t* G;   // bf16 bits, [rows_pad, ldg]
  int64_t ldg;
  // EPI_STORE
  float* out;
  int64_t ldo;
  int out_rows, out_cols;
  int accumulate;
  // EPI_LSE_MIX / EPI_GRAD_MIX: soft KL mixed with a hard-label cross-entropy
  const int32_t* labels;  // [T] hard label per token
  int same_tau;           // tau == 1: the temperature-1 sums equal the tau sums
  float* ps1;             // [nsplit, T] sum of exp2((z - max) * log2(e))   (LSE_MIX)
  float* pzl;             // [nsplit, T] z at the label if in this split, else 0 (LSE_MIX)
  const float* lse1;      // [T] logsumexp of z at temperature 1        (GRAD_MIX)
  float kl_weight;        // alpha * c / tau (times g / N per counted row) (GRAD_MIX)
  float ce_weight;        // (1 - alpha)     (times g / N per counted row) (GRAD_MIX)
  // EPI_TOPK (K is the field above)
  int topk_cap;      // capacity of a row's candidate list (K + slack, at most 1024)
  float2* cand;      // [gridDim.x * BM, topk_cap] (logit, id bits), one list per (CTA, row)
  uint32_t* row_key; // [T] order key of the best K-th logit any split has seen (0 = none)
  float* unit_val;   // [nsplit, T, K] each split's kept top-K entries per row (id order)
  int32_t* unit_id;
  int* unit_cnt;     // [nsplit, T] entries kept per (split, row)
};

// Order-preserving map of an fp32 value to uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t f32_order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The whole warp reduces one row's candidate list (n entries, n >= K, at most
// 32 * MAXE, appended in increasing id order) to its K best by (logit
// descending, id ascending), in place and in the same id order. Returns the K-th best logit,
// the row's new admission threshold: a later candidate of the same row has a
// larger id, so only a strictly larger logit can displace a kept entry.
// The K-th largest key is found by bisection over the 32-bit order keys,
// starting from the list's min/max keys and stopping early once a midpoint
// separates exactly K keys.
template <int MAXE>
static __device__ __noinline__ float topk_compact_row_n(float2* list, int n, int K) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  uint32_t key[MAXE];
  float idv[MAXE];  // id bits carried as a float
#pragma unroll
  for (int i = 0; i < MAXE; ++i) {
    const int e = i * 32 + lane;
    const float2 c = e < n ? list[e] : make_float2(0.f, 0.f);
    key[i] = e < n ? f32_order_key(c.x) : 0u;
    idv[i] = c.y;
  }
  // Search range: the list's own smallest and largest keys.
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int i = 0; i < MAXE; ++i) {
    if (i * 32 + lane < n) {
      lo = min(lo, key[i]);
      hi = max(hi, key[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  // Invariant: at least K keys are >= lo. Stop early when a midpoint has
  // exactly K keys at or above it (then those K are the top K and the
  // threshold is the smallest of them); otherwise lo ends at the K-th key.
  bool exact = false;
  while (lo < hi) {
    const uint32_t mid = lo + ((hi - lo) >> 1) + 1u;
    int c = 0;
#pragma unroll
    for (int i = 0; i < MAXE; ++i) c += (i * 32 + lane < n && key[i] >= mid) ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (c == K) {
      lo = mid;
      exact = true;
      break;
    }
    if (c > K) lo = mid; else hi = mid - 1u;
  }
  if (exact) {
    // the K kept keys are those >= lo; the threshold is the smallest of them
    uint32_t kmin = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < MAXE; ++i)
      if (i * 32 + lane < n && key[i] >= lo) kmin = min(kmin, key[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    lo = kmin;  // exactly K keys are >= kmin (no key lies in [kmin, mid) beyond those)
  }
  int gt = 0;
#pragma unroll
  for (int i = 0; i < MAXE; ++i) gt += (i * 32 + lane < n && key[i] > lo) ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) gt += __shfl_xor_sync(0xffffffffu, gt, o);
  const int need_eq = K - gt;
  __syncwarp();
  int written = 0, eq_seen = 0;
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < MAXE; ++i) {
    const bool valid = i * 32 + lane < n;
    const bool is_gt = valid && key[i] > lo;
    const bool is_eq = valid && key[i] == lo;
    const uint32_t eq_mask = __ballot_sync(0xffffffffu, is_eq);
    const int eq_rank = eq_seen + __popc(eq_mask & below);
    const bool keep = is_gt || (is_eq && eq_rank < need_eq);
    const uint32_t keep_mask = __ballot_sync(0xffffffffu, keep);
    if (keep) list[written + __popc(keep_mask & below)] = make_float2(f32_from_order_key(key[i]), idv[i]);
    written += __popc(keep_mask);
    eq_seen += __popc(eq_mask);
  }
  __syncwarp();
  return f32_from_order_key(lo);
}

// Lists of up to 512 entries (K <= 256 with the default slack) take the
// 16-slot form; longer ones (K up to 512) the 32-slot form.
__device__ __forceinline__ float topk_compact_row(float2* list, int n, int K, int cap) {
  return cap <= 512 ? topk_compact_row_n<16>(list, n, K) : topk_compact_row_n<32>(list, n, K);
}

// Admission threshold from the best K-th logit published by any split of the
// row: values equal to it are still admitted (an equal logit with a smaller
// id may belong to the row's top-K), values below cannot be in the top-K.
__device__ __forceinline__ float topk_shared_threshold(const uint32_t* row_key) {
  const uint32_t k = *reinterpret_cast<const volatile uint32_t*>(row_key);
  return k == 0u ? -INFINITY : nextafterf(f32_from_order_key(k), -INFINITY);
}

__device__ __forceinline__ void unit_coords(const GemmShape& sh, int u, int& m, int& s, int& nb,
                                            int& ne) {
  int s0 = 0;
  if (sh.first_group) {
    if (u < sh.m_tiles) {
      m = u;
      s = 0;
      split_range(sh, 0, nb, ne);
      return;
    }
    u -= sh.m_tiles;
    s0 = 1;
  }
  const int ns = sh.nsplit - s0;
  const int per_group = sh.group_m * ns;
  const int g = u / per_group;
  const int r = u - g * per_group;
  const int gm = min(sh.group_m, sh.m_tiles - g * sh.group_m);  // the last group may be short
  const int si = r / gm;
  s = s0 + si;
  m = g * sh.group_m + (r - si * gm);
  split_range(sh, s, nb, ne);
}

// First position in the sorted id row whose id is >= v (K when none).
__device__ __forceinline__ int lower_bound_row(const int32_t* row, int K, int v) {
  int lo = 0, hi = K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(row + mid) < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Shrinks a shape to the rows counted on the device (see GemmShape::dyn_rows);
// returns the live extent along M (or -1 when M is not shrunk).
template <int TILE_M>
__device__ __forceinline__ int shrink_shape(GemmShape& sh) {
  if (!sh.dyn_rows) return -1;
  const int a = max(0, min(*sh.dyn_rows - sh.dyn_base, sh.dyn_cap));
  if (sh.dyn_dim == 0) {
    sh.m_tiles = min(sh.m_tiles, (a + TILE_M - 1) / TILE_M);
    sh.units = sh.m_tiles * sh.nsplit;
    return a;
  }
  sh.k_blocks = min(sh.k_blocks, (a + BK - 1) / BK);
  return -1;
}

// DUAL: two store GEMMs in one persistent launch, their units in one
// sequence: job 0 (maps tmA/tmB, shape sh, output ep; A as A_MN) and then job
// 1 (tmA1/tmB1, sh1, ep1; A the other way round, B as B_MN). The backward runs
// dW and dH of a block this way (the tail of the first job's units is filled
// by the second job's).
template <int EPI, bool A_MN, bool B_MN, int BN, bool PAIR, bool DUAL>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB1, const GemmShape sh_in,
                   const GemmShape sh1_in, const EpiParams ep, const EpiParams ep1, int* status) {
  static_assert(!DUAL || EPI == EPI_STORE, "two jobs per launch only for store epilogues");
  using Cfg = TileCfg<BN, PAIR>;
  constexpr bool IS_LSE = EPI == EPI_LSE || EPI == EPI_LSE_MIX;
  constexpr bool IS_GRAD = EPI == EPI_GRAD || EPI == EPI_GRAD_MIX;
  constexpr bool MIX = EPI == EPI_LSE_MIX || EPI == EPI_GRAD_MIX;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int B_STAGE_BYTES = Cfg::B_STAGE_BYTES;
  constexpr int STAGE_BYTES = Cfg::STAGE_BYTES;
  constexpr int NUM_BARS = Cfg::NUM_BARS;
  constexpr int TILE_M = Cfg::TILE_M;
  constexpr int B_ROWS = Cfg::B_ROWS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Ring of units handed from the scheduler (the leader CTA's producer) to
  // every other role of both CTAs: slot i holds a unit number (-1: no more).
  constexpr int NSLOT = 4;
  volatile int* unit_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto ufull_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 5 + i); };
  auto uempty_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 5 + NSLOT + i); };

  // Every role shrinks the shapes to the live rows the same way, so they all
  // see the same units and K steps.
  GemmShape sh = sh_in;
  GemmShape sh1 = sh1_in;
  int live_rows = IS_LSE || IS_GRAD ? ep.rows : 0;  // rows whose token counts
  {
    const int a = shrink_shape<TILE_M>(sh);
    if (a >= 0) live_rows = min(live_rows, a);
    if (DUAL) shrink_shape<TILE_M>(sh1);
  }
  const int units0 = sh.units;
  const int units_all = units0 + (DUAL ? sh1.units : 0);
  // Per unit: its job's shape, the unit within that job, and A's layout.
  auto job_of = [&](int u, const GemmShape*& js, int& uu, bool& a_mn) {
    const bool j1 = DUAL && u >= units0;
    js = j1 ? &sh1 : &sh;
    uu = j1 ? u - units0 : u;
    a_mn = j1 ? !A_MN : A_MN;
    return j1;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = sh.inject_stall ? kInjectedWaitLimitNs : kWaitLimitNs;
  // PAIR: CTAs 2c and 2c+1 form cluster c; rank 0 (the leader) issues the MMAs.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int group0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int groups = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), PAIR ? 8 : 4);
    }
    mbar_init(drain_bar, 1);
    // A slot is released by every role that reads it: the MMA thread and the
    // 4 epilogue warps here, and with a pair the peer's producer and its 4
    // epilogue warps (remote arrives on the leader's barrier).
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(ufull_bar(i), 1);
      mbar_init(uempty_bar(i), PAIR ? 10 : 5);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (DUAL) {
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
    }
  }
  if (warp == 1) {
    __syncwarp();
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Consumer side of the unit ring: wait for slot q's unit (cluster-scope
  // acquire with a pair: the leader wrote the peer's slot remotely), then
  // release the slot on the leader's barrier once the value is read.
  const uint32_t uempty_leader0 = PAIR ? mapa_shared(uempty_bar(0), 0) : uempty_bar(0);
  auto take_unit = [&](int q, int& u) -> bool {
    const int slot = q & (NSLOT - 1);
    const uint32_t ph = (uint32_t)(q / NSLOT) & 1u;
    const bool got = PAIR ? mbar_wait_cluster_bounded(ufull_bar(slot), ph, abort_flag, status, limit)
                          : mbar_wait_bounded(ufull_bar(slot), ph, abort_flag, status, limit);
    if (got) u = unit_slot[slot];
    return got;
  };
  auto release_unit = [&](int q) {
    const int slot = q & (NSLOT - 1);
    if (PAIR)
      mbar_arrive_cluster(uempty_leader0 + 8u * slot);
    else
      mbar_arrive(uempty_bar(slot));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      // Loads this CTA's A rows and B rows of every stage into its own shared
      // memory. Single CTA: signals its own full barrier. Pair: both CTAs
      // signal the LEADER's full barrier (pair form of the copy), which the
      // leader arms with the bytes of both halves, so the leader's MMA thread
      // waits on one barrier for the whole 256-row stage.
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = sh.inject_stall == 0;
      const uint32_t full_leader0 = PAIR ? mapa_shared(full_bar(0), 0) : full_bar(0);
      // The leader's producer is also the scheduler: it takes units from the
      // launch's counter (the next one fetched a unit ahead, so the atomic's
      // latency hides behind a unit of copies) and publishes each in the ring.
      const bool dyn = sh.counter != nullptr;
      int next = (ok && leader) ? (dyn ? atomicAdd(sh.counter, 1) : group0) : -1;
      const uint32_t peer_slot0 = PAIR ? mapa_shared(smem_u32((const void*)unit_slot), 1) : 0u;
      const uint32_t peer_ufull0 = PAIR ? mapa_shared(ufull_bar(0), 1) : 0u;
      for (int uq = 0; ok; ++uq) {
        int u = -1;
        if (leader) {
          const int slot = uq & (NSLOT - 1);
          const uint32_t ph = ((uint32_t)(uq / NSLOT) & 1u) ^ 1u;
          const bool freed =
              PAIR ? mbar_wait_cluster_bounded(uempty_bar(slot), ph, abort_flag, status, limit)
                   : mbar_wait_bounded(uempty_bar(slot), ph, abort_flag, status, limit);
          if (!freed) {
            ok = false;
            break;
          }
          u = next < units_all ? next : -1;
          if (u >= 0) next = dyn ? atomicAdd(sh.counter, 1) : next + groups;
          unit_slot[slot] = u;
          if (PAIR) {
            st_shared_cluster_u32(peer_slot0 + 4u * slot, (uint32_t)u);
            mbar_arrive_cluster(peer_ufull0 + 8u * slot);
          }
          mbar_arrive(ufull_bar(slot));
        } else {
          if (!take_unit(uq, u)) {
            ok = false;
            break;
          }
          release_unit(uq);
        }
        if (u < 0) break;
        const GemmShape* js;
        int uu;
        bool a_mn;
        const bool j1 = job_of(u, js, uu, a_mn);
        const CUtensorMap* ta = j1 ? &tmA1 : &tmA;
        const CUtensorMap* tb = j1 ? &tmB1 : &tmB;
        int m, s, nb, ne;
        unit_coords(*js, uu, m, s, nb, ne);
        const int a_row = js->a_m0 + m * TILE_M + (int)rank * BM;
        for (int n = nb; ok && n < ne; ++n) {
          const bool narrow = B_MN && js->narrow_last && n == js->n_tiles - 1;
          const int b_rows = narrow ? B_ROWS / 2 : B_ROWS;  // B rows this CTA copies
          const int b_row = js->b_n0 + n * BN + (int)rank * b_rows;
          const uint32_t stage_bytes = (uint32_t)(A_STAGE_BYTES + b_rows * BK * 2);
          for (int kb = 0; kb < js->k_blocks; ++kb) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status, limit)) {
              ok = false;
              break;
            }
            const uint32_t fb = full_leader0 + 8u * stage;
            if (leader) mbar_arrive_expect_tx(full_bar(stage), (PAIR ? 2u : 1u) * stage_bytes);
            const uint32_t a_dst = smem_u32(sA + stage * A_STAGE_BYTES);
            const uint32_t b_dst = smem_u32(sB + stage * B_STAGE_BYTES);
            const int kc = kb * BK;
            auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y) {
              if (PAIR)
                tma_load_2d_pair(dst, tm, fb, x, y);
              else
                tma_load_2d(dst, tm, fb, x, y);
            };
            if (!a_mn) {
              load(a_dst, ta, js->a_k0 + kc, a_row);
            } else {
#pragma unroll
              for (int a = 0; a < BM / 64; ++a)
                load(a_dst + a * MN_ATOM_BYTES, ta, a_row + 64 * a, js->a_k0 + kc);
            }
            if (!B_MN) {
              load(b_dst, tb, js->b_k0 + kc, b_row);
            } else {
              for (int a = 0; a < b_rows / 64; ++a)
                load(b_dst + a * MN_ATOM_BYTES, tb, b_row + 64 * a, js->b_k0 + kc);
            }
            ++fills;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Teardown: every copy issued must have landed before the CTA exits. The
      // full barriers live in the leader and count both halves of the pair,
      // so the leader drains for both; the peer's copies are also covered by
      // the closing cluster barrier, which the leader reaches only after its
      // MMAs consumed every stage.
      if (leader)
        for (long long f = fills - 1; f >= 0 && f >= fills - STAGES; --f)
          mbar_drain_bounded(full_bar((int)(f % STAGES)), (uint32_t)((f / STAGES) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc0 = idesc_bf16_f32(TILE_M, BN, A_MN, B_MN);
      constexpr uint32_t idesc1 = idesc_bf16_f32(TILE_M, BN, !A_MN, B_MN);  // DUAL job 1
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int uq = 0; ok; ++uq) {
        int u = -1;
        if (!take_unit(uq, u)) break;
        release_unit(uq);
        if (u < 0) break;
        const GemmShape* js;
        int uu;
        bool a_mn;
        const bool j1 = job_of(u, js, uu, a_mn);
        // No K steps (no counted token in a dW launch): nothing to multiply;
        // the epilogue writes zeros without touching TMEM.
        if (js->k_blocks == 0) continue;
        const uint32_t idesc = j1 ? idesc1 : idesc0;
        int m, s, nb, ne;
        unit_coords(*js, uu, m, s, nb, ne);
        for (int n = nb; ok && n < ne; ++n) {
          // the narrow last tile (see GemmShape::narrow_last) multiplies N = BN/2
          const bool narrow = B_MN && js->narrow_last && n == js->n_tiles - 1;
          const uint32_t idesc_n =
              narrow ? idesc_bf16_f32(TILE_M, BN / 2, a_mn, B_MN) : idesc;
          const bool freed = PAIR ? mbar_wait_cluster_bounded(tempty_bar(acc), acc_phase ^ 1u,
                                                              abort_flag, status, limit)
                                  : mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u,
                                                      abort_flag, status, limit);
          if (!freed) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          for (int kb = 0; kb < js->k_blocks; ++kb) {
            if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, status, limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
            const uint32_t b_base = smem_u32(sB + stage * B_STAGE_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t ad = a_mn ? sdesc_sw128(a_base + k * 2048, MN_ATOM_BYTES, 1024)
                                       : sdesc_sw128(a_base + k * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(b_base + k * 2048, MN_ATOM_BYTES, 1024)
                                       : sdesc_sw128(b_base + k * 32, 16, 1024);
              if (PAIR)
                tc_mma_bf16_pair(d_tmem, ad, bd, idesc_n, (kb | k) != 0 ? 1u : 0u);
              else
                tc_mma_bf16(d_tmem, ad, bd, idesc_n, (kb | k) != 0 ? 1u : 0u);
            }
            if (PAIR)
              tc_commit_pair_multicast(empty_bar(stage), 0x3);
            else
              tc_commit(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (PAIR)
            tc_commit_pair_multicast(tfull_bar(acc), 0x3);
          else
            tc_commit(tfull_bar(acc));
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      // Teardown: all MMAs issued by this thread complete before TMEM is freed.
      if (PAIR)
        tc_commit_pair_local(drain_bar);
      else
        tc_commit(drain_bar);
      mbar_drain_bounded(drain_bar, 0);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint32_t tempty_remote0 = PAIR ? mapa_shared(tempty_bar(0), 0) : 0u;
    // EPI_TOPK: each (CTA, row) has two list banks. When a unit ends, the warp
    // switches bank and finishes the old unit's rows later (compaction to K
    // and write-out, one row at a time), in the waits for the next unit's
    // accumulators, instead of in one burst at the unit boundary.
    int bank = 0;
    uint32_t pend = 0u;  // rows of the finished unit still to write (warp-uniform)
    int pend_cnt = 0;    // this lane's list length in that unit
    int pend_bank = 0, pend_s = 0, pend_r0 = 0;
    auto list_of = [&](int row_in_warp, int b) {
      return ep.cand + (((long long)blockIdx.x * BM + q * 32 + row_in_warp) * 2 + b) * ep.topk_cap;
    };
    auto finalize_row = [&](int i) {  // warp-collective
      const int ni = __shfl_sync(0xffffffffu, pend_cnt, i);
      float2* li = list_of(i, pend_bank);
      if (ni > ep.K) {
        const float thi = topk_compact_row(li, ni, ep.K, ep.topk_cap);
        if (lane == 0) atomicMax(ep.row_key + ep.row0 + pend_r0 + i, f32_order_key(thi));
      }
      __syncwarp();
      // Only entries at or above the row's best published K-th logit can be
      // in its top-K: the rest are dropped here, the kept ones written in
      // order with their count, so the merge reads only what survives.
      const long long row = (long long)ep.row0 + pend_r0 + i;
      const float th_now = topk_shared_threshold(ep.row_key + row);
      const int nk = min(ni, ep.K);
      const long long o = ((long long)pend_s * ep.T + row) * ep.K;
      const uint32_t below = (1u << lane) - 1u;
      int w = 0;
      for (int k0 = 0; k0 < nk; k0 += 32) {
        const int k = k0 + lane;
        const float2 c = k < nk ? li[k] : make_float2(-INFINITY, 0.f);
        const bool keep = k < nk && c.x > th_now;
        const uint32_t km = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          ep.unit_val[o + w + __popc(km & below)] = c.x;
          ep.unit_id[o + w + __popc(km & below)] = __float_as_int(c.y);
        }
        w += __popc(km);
      }
      if (lane == 0) ep.unit_cnt[(long long)pend_s * ep.T + row] = w;
    };
    for (int uq = 0; ok; ++uq) {  // uq: position in the unit ring (q is the lane quarter)
      int u = -1;
      const bool got_unit = __all_sync(0xffffffffu, take_unit(uq, u));
      if (!got_unit) {
        ok = false;
        break;
      }
      __syncwarp();  // every lane has read the slot before it is released
      if (lane == 0) release_unit(uq);
      if (u < 0) break;
      const GemmShape* js;
      int uu;
      bool a_mn_unused;
      const bool j1 = job_of(u, js, uu, a_mn_unused);
      const EpiParams& eo = j1 ? ep1 : ep;  // the unit's output (store epilogues)
      const bool no_k = js->k_blocks == 0;  // zeros, no TMEM (see the MMA role)
      int m, s, nb, ne;
      unit_coords(*js, uu, m, s, nb, ne);
      const int r = m * TILE_M + (int)rank * BM + r_in_tile;  // row within this launch
      // per-unit row state
      float run_max = -INFINITY, run_sum = 0.f, dot = 0.f;
      float lse2 = 0.f, scale = 0.f;
      int cursor = ep.K, cur_id = 0x7fffffff;
      const int32_t* id_row = nullptr;
      const float* p_row = nullptr;
      bool row_ok = false;    // the row exists in this launch
      bool row_live = false;  // ... and holds a token (a counted one when compacted)
      // EPI_TOPK row state: admission threshold and candidate count
      float th = INFINITY;
      int cnt = 0;
      float2* c_list = nullptr;
      uint32_t* rkey = nullptr;
      if (EPI == EPI_TOPK) {
        row_ok = r < ep.rows;
        c_list = list_of(lane, bank);
        if (row_ok) {
          rkey = ep.row_key + ep.row0 + r;
          th = topk_shared_threshold(rkey);
        }
      }
      // MIX row state: temperature-1 sum, label logit, label id
      float run_s1 = 0.f, zl = 0.f, lse12 = 0.f, w_kl = 0.f, w_ce = 0.f;
      int lab = -1;
      if (IS_LSE || IS_GRAD) {
        row_ok = r < ep.rows;
        row_live = r < live_rows;
        if (row_live) {
          // trow: the row of the teacher cache, partials and G; tok: the
          // caller's token (lse, mask, labels), the same unless compacted
          const long long trow = (long long)ep.row0 + r;
          const long long tok = ep.rowmap ? (long long)__ldg(ep.rowmap + trow) : trow;
          id_row = ep.sidx + trow * ep.K;
          p_row = ep.sp + trow * ep.K;
          cursor = lower_bound_row(id_row, ep.K, ep.col0 + nb * BN);
          cur_id = cursor < ep.K ? __ldg(id_row + cursor) : 0x7fffffff;
          if (IS_GRAD) {
            lse2 = __ldg(ep.lse + tok) * 1.4426950408889634f;
            const int n = *ep.n_count;
            const bool counted =
                ep.rowmap || ep.mask == nullptr || __ldg(ep.mask + tok) != 0;
            scale = (counted && n > 0) ? ep.g_over_tau / (float)n : 0.f;
            if (MIX) {
              lse12 = __ldg(ep.lse1 + tok) * 1.4426950408889634f;
              const float per_row = (counted && n > 0) ? 1.f / (float)n : 0.f;
              w_kl = ep.kl_weight * per_row;  // kl_weight carries g * alpha * c / tau
              w_ce = ep.ce_weight * per_row;  // ce_weight carries g * (1 - alpha)
            }
          }
          if (MIX) lab = ep.labels ? __ldg(ep.labels + tok) : -1;
        }
      }
      for (int n = nb; n < ne; ++n) {
        if (EPI == EPI_TOPK) {
          // While the next accumulator is not ready, compact rows whose lists
          // are past half their slack: work moved out of the bursts in which
          // many rows must compact before the next 32 appends (and the MMA
          // waits on this warp). At most 32 rows per wait.
          const int watermark = (ep.topk_cap + ep.K) / 2;
          for (int spins = 0; spins < 32; ++spins) {
            if (__any_sync(0xffffffffu, mbar_test_wait(tfull_bar(acc), acc_phase))) break;
            if (pend) {  // the finished unit's rows come first
              const int i = __ffs(pend) - 1;
              pend &= pend - 1u;
              finalize_row(i);
              continue;
            }
            const uint32_t want = __ballot_sync(0xffffffffu, cnt > watermark);
            if (!want) break;
            const int i = __ffs(want) - 1;
            const int ni = __shfl_sync(0xffffffffu, cnt, i);
            const float thi = topk_compact_row(list_of(i, bank), ni, ep.K, ep.topk_cap);
            if (lane == i) {
              th = fmaxf(th, thi);
              cnt = ep.K;
              atomicMax(rkey, f32_order_key(thi));
            }
          }
        }
        bool got = no_k || mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, status, limit);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + lane_off + (uint32_t)(acc * BN);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int cl = n * BN + c * 32;  // column within this launch
          if (IS_LSE || IS_GRAD || EPI == EPI_TOPK) {
            if (cl >= ep.cols) break;  // warp-uniform
          } else {
            if (cl >= eo.out_cols) break;
          }
          if (EPI == EPI_TOPK) {
            // room for this piece's 32 possible appends in every row of the warp
            uint32_t need = __ballot_sync(0xffffffffu, cnt > ep.topk_cap - 32);
            while (need) {
              const int i = __ffs(need) - 1;
              need &= need - 1u;
              const int ni = __shfl_sync(0xffffffffu, cnt, i);
              const float thi = topk_compact_row(list_of(i, bank), ni, ep.K, ep.topk_cap);
              if (lane == i) {
                th = fmaxf(th, thi);
                cnt = ep.K;
                atomicMax(rkey, f32_order_key(thi));  // share with the row's other splits
              }
            }
            if (c == 0 && row_ok) th = fmaxf(th, topk_shared_threshold(rkey));
          }
          float v[32];
          __syncwarp();
          if (no_k) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          } else {
            tmem_ld32(tbase + (uint32_t)(c * 32), v);
          }
          if (IS_LSE) {
            const int vid0 = ep.col0 + cl;
            if (cl + 32 > ep.cols) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (cl + j >= ep.cols) v[j] = -INFINITY;
            }
            float mx = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) mx = fmaxf(mx, v[j]);
            const float nm = fmaxf(run_max, mx);
            const float nmc = nm * ep.cl2;
            float acc_s = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) acc_s += ex2_approx(fmaf(v[j], ep.cl2, -nmc));
            run_sum = fmaf(run_sum, ex2_approx((run_max - nm) * ep.cl2), acc_s);
            if (MIX && !ep.same_tau) {
              constexpr float L2E = 1.4426950408889634f;
              const float nm1 = nm * L2E;
              float acc1 = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) acc1 += ex2_approx(fmaf(v[j], L2E, -nm1));
              run_s1 = fmaf(run_s1, ex2_approx((run_max - nm) * L2E), acc1);
            }
            run_max = nm;
            if (MIX && row_live && lab >= vid0 && lab < vid0 + 32 && lab < ep.col0 + ep.cols)
              zl = select32(v, lab - vid0);
            if (row_live) {
              const int vend = ep.col0 + min(cl + 32, ep.cols);
              while (cur_id < vend) {
                if (cur_id >= vid0) dot = fmaf(__ldg(p_row + cursor), select32(v, cur_id - vid0), dot);
                ++cursor;
                cur_id = cursor < ep.K ? __ldg(id_row + cursor) : 0x7fffffff;
              }
            }
          } else if (IS_GRAD) {
            const int vid0 = ep.col0 + cl;
            float g[32];
            if (MIX) {
              // w_kl (q_tau - P) + w_ce (q_1 - onehot(label)); the weights hold m g / N
              constexpr float L2E = 1.4426950408889634f;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float qt = ex2_approx(fmaf(v[j], ep.cl2, -lse2));
                const float q1 = ep.same_tau ? qt : ex2_approx(fmaf(v[j], L2E, -lse12));
                g[j] = fmaf(qt, w_kl, q1 * w_ce);
              }
              if (row_live && lab >= vid0 && lab < vid0 + 32) {
                const int jl = lab - vid0;
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = (j == jl) ? g[j] - w_ce : g[j];
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) g[j] = ex2_approx(fmaf(v[j], ep.cl2, -lse2));
            }
            if (row_ok) {
              // rows past the live ones (compacted tokens end mid-tile) get
              // zeros: their teacher rows are never read (cursor stays at K)
              const int vend = ep.col0 + min(cl + 32, ep.cols);
              while (cur_id < vend) {
                if (cur_id >= vid0) {
                  const float pk = MIX ? __ldg(p_row + cursor) * w_kl : __ldg(p_row + cursor);
                  const int jj = cur_id - vid0;
#pragma unroll
                  for (int j = 0; j < 32; ++j) g[j] = (j == jj) ? g[j] - pk : g[j];
                }
                ++cursor;
                cur_id = cursor < ep.K ? __ldg(id_row + cursor) : 0x7fffffff;
              }
              if (MIX) scale = row_live ? 1.f : 0.f;  // weights already applied
              if (!row_live) {
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = 0.f;
              }
              uint4* dst = reinterpret_cast<uint4*>(ep.G + (long long)r * ep.ldg + cl);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint4 w;
                w.x = pack_bf16x2(g[8 * j + 0] * scale, g[8 * j + 1] * scale);
                w.y = pack_bf16x2(g[8 * j + 2] * scale, g[8 * j + 3] * scale);
                w.z = pack_bf16x2(g[8 * j + 4] * scale, g[8 * j + 5] * scale);
                w.w = pack_bf16x2(g[8 * j + 6] * scale, g[8 * j + 7] * scale);
                dst[j] = w;
              }
            }
          } else if (EPI == EPI_TOPK) {
            const int vid0 = ep.col0 + cl;
            const int nv = min(32, ep.cols - cl);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < nv && v[j] > th) {
                c_list[cnt] = make_float2(v[j], __int_as_float(vid0 + j));
                ++cnt;
              }
            }
          } else {  // EPI_STORE
            if (r < eo.out_rows) {
              float* dst = eo.out + (long long)r * eo.ldo + cl;
              const int nvalid = min(32, eo.out_cols - cl);  // multiple of 4
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                if (4 * j < nvalid) {
                  const float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                  // Accumulate with a vector reduction: every element gets
                  // exactly one add per launch and launches are stream-ordered,
                  // so the sum order is fixed (deterministic).
                  if (eo.accumulate)
                    red_add_f32x4(dst + 4 * j, o);
                  else
                    *reinterpret_cast<float4*>(dst + 4 * j) = o;
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (no_k) continue;  // no accumulator was used
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster(tempty_remote0 + 8u * acc);  // the leader's barrier
          else
            mbar_arrive(tempty_bar(acc));
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) break;
      if (EPI == EPI_TOPK) {
        // Hand this unit's lists over to the deferred final step. Rows still
        // pending from the unit before (only when units are a few tiles long)
        // are finished first, since their bank is about to be reused.
        while (pend) {
          const int i = __ffs(pend) - 1;
          pend &= pend - 1u;
          finalize_row(i);
        }
        pend = __ballot_sync(0xffffffffu, row_ok);
        pend_cnt = cnt;
        pend_bank = bank;
        pend_s = s;
        pend_r0 = m * TILE_M + (int)rank * BM + q * 32;
        bank ^= 1;
      }
      if (IS_LSE && row_live) {
        const long long o = (long long)s * ep.T + ep.row0 + r;
        ep.pm[o] = run_max;
        ep.ps[o] = run_sum;
        ep.pd[o] = dot;
        if (MIX) {
          ep.ps1[o] = ep.same_tau ? run_sum : run_s1;
          ep.pzl[o] = zl;
        }
      }
    }
    if (EPI == EPI_TOPK && ok) {
      while (pend) {
        const int i = __ffs(pend) - 1;
        pend &= pend - 1u;
        finalize_row(i);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the leader's MMAs into the peer's TMEM are done
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace kdkl
