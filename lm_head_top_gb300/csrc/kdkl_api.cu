// C ABI of the fused chunked KL distillation loss: argument checks, the
// workspace plan, the chunk scheduler and the launch sequence.
//
// Forward  (one pass over all tokens; no logits leave the SMs):
//   teacher_prep -> fwd_lse_gemm -> lse_combine -> loss_finalize
// Backward (recompute per block of the tokens x vocabulary plane):
//   teacher_prep -> for each block: bwd_grad_gemm -> dH_gemm -> dW_gemm
//                -> f32_to_bf16 (dH)
//
// The pages ("Making knowledge distillation cheap enough to run at scale",
// section "Two system changes"; "Efficient knowledge distillation for LLMs:
// offline top-K logits and a fused chunked KL loss", section "Two systemic
// changes for scalable distillation") process one chunk of sequence positions
// at a time so memory grows linearly with the sequence, and compute each
// chunk again in backward. Here `chunk` bounds the one buffer that
// holds gradients of logits (chunk x V bf16). The forward needs no such
// buffer at all: its epilogue keeps only three floats per token and split.
// In backward the scheduler tiles the same budget either as `chunk` tokens by
// the whole vocabulary, or (when T <= V) all tokens by a vocabulary slab, so
// that the fp32 read-modify-write lands on the smaller of dW [V,d] and
// dH [T,d]. Both tilings give the same sums.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "kdkl.h"
#include "kdkl_internal.h"
#include "tc_gemm.cuh"

namespace kdkl {

// ------------------------------------------------------------ bookkeeping

namespace {

std::atomic<int64_t> g_launches{0};
std::atomic<bool> g_timing{false};
std::mutex g_timing_mu;

struct PendingTiming {
  const char* name;
  cudaEvent_t start, stop;
};
std::vector<PendingTiming> g_pending;

}  // namespace

void note_launch_begin(const char* name, cudaStream_t stream, void** token) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  *token = nullptr;
  if (!g_timing.load(std::memory_order_acquire)) return;
  auto* p = new PendingTiming{name, nullptr, nullptr};
  if (cudaEventCreate(&p->start) != cudaSuccess || cudaEventCreate(&p->stop) != cudaSuccess) {
    delete p;
    return;
  }
  cudaEventRecord(p->start, stream);
  *token = p;
}

void note_launch_end(void* token, cudaStream_t stream) {
  if (!token) return;
  auto* p = static_cast<PendingTiming*>(token);
  cudaEventRecord(p->stop, stream);
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_pending.push_back(*p);
  delete p;
}

// ------------------------------------------------------------- device info

namespace {

constexpr size_t kHeaderBytes = 256;  // int status; int n_count; padding
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  bool supported = false;
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

kd_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KD_ERR_CUDA;
    di.supported = (major == 10 && minor == 3);
    di.num_sms = sms;
    di.init = true;
  }
  *out = di;
  return di.supported ? KD_OK : KD_ERR_UNSUPPORTED;
}

kd_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode ? KD_OK : KD_ERR_CUDA;
}

// bf16 row-major matrix [outer, inner] with the given row stride (elements),
// 128-byte swizzle, box of box_inner x box_outer elements. Out-of-range
// elements of a box read as zero.
bool encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// -------------------------------------------------------------- planning

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Unit plan of the logit GEMMs (forward, backward recompute, top-K). A unit is
// one m-tile and one split of about `split_tiles` vocabulary tiles; units are
// handed out while the kernel runs, in groups of group_m m-tiles with the
// m-tile fastest (tc_gemm.cuh). The group's A rows (tile_m x d bf16 per
// m-tile) stay in L2 while its splits stream past, so group_m is set by an
// L2 budget for them. Short units keep the units in flight on a narrow window
// of vocabulary tiles, which are then read from DRAM about once per group.
struct LogitPlan {
  int m_tiles, n_tiles, nsplit, group_m, units;
};
constexpr double kL2RowBudgetDefault = 32.0 * 1024 * 1024;

// KDKL_L2_ROWS_MB overrides the L2 budget for the A rows of one group (tuning).
double l2_row_budget() {
  const char* v = getenv("KDKL_L2_ROWS_MB");
  const double mb = v ? atof(v) : 0.0;
  return mb > 0 ? mb * 1024 * 1024 : kL2RowBudgetDefault;
}

// KDKL_SPLIT_TILES overrides the vocabulary tiles per unit of the forward
// logit GEMM (tuning).
int fwd_split_tiles() {
  const char* v = getenv("KDKL_SPLIT_TILES");
  const int n = v ? atoi(v) : 0;
  return n > 0 ? n : 8;
}

LogitPlan plan_logit(int64_t rows, int64_t cols, int64_t d, int tile_m, int split_tiles) {
  LogitPlan lp{};
  lp.m_tiles = (int)std::max<int64_t>(ceil_div(rows, tile_m), 1);
  lp.n_tiles = (int)ceil_div(cols, LOGIT_BN);
  lp.nsplit = (int)std::max<int64_t>(1, ceil_div(lp.n_tiles, std::max(1, split_tiles)));
  const double a_tile_bytes = (double)tile_m * (double)d * 2.0;
  const int gm = (int)std::max(1.0, std::floor(l2_row_budget() / a_tile_bytes));
  lp.group_m = std::min(gm, lp.m_tiles);
  lp.units = lp.m_tiles * lp.nsplit;
  return lp;
}

// KDKL_STATIC_SCHED=1: units are taken round-robin by CTA group instead of
// from the launch counter (same order; kept to compare the two schedules).
bool static_schedule() {
  const char* v = getenv("KDKL_STATIC_SCHED");
  return v && v[0] == '1';
}

// The prepared teacher side of a call, at the same place in the forward and
// the backward workspaces (from `base` on), so that a backward can read the
// forward's: sorted ids and p [T, K]; when a mask is given, the compaction of
// the counted tokens: rowmap [T] (row -> token), invmap [T] (token -> row or
// -1) and Hc, H's counted rows [T_pad, d] bf16 (T_pad = T rounded up to 256).
struct TeacherLayout {
  size_t off_sidx, off_sp, off_rowmap, off_invmap, off_Hc, end;
};

TeacherLayout teacher_layout(size_t base, const kd_kl_problem& p) {
  TeacherLayout L{};
  const size_t TK = (size_t)p.T * p.K;
  size_t o = base;
  L.off_sidx = o; o = align256(o + TK * 4);
  L.off_sp = o; o = align256(o + TK * 4);
  L.off_rowmap = o; o = align256(o + (size_t)p.T * 4);
  L.off_invmap = o; o = align256(o + (size_t)p.T * 4);
  L.off_Hc = o; o = align256(o + (size_t)round_up(p.T, 2 * BM) * p.d * 2);
  L.end = o;
  return L;
}

struct FwdPlan {
  bool pair;
  int m_tiles, n_tiles, nsplit, group_m, grid;
  TeacherLayout tl;
  size_t off_ent, off_pm, off_ps, off_pd, off_ps1, off_pzl, off_bsum, total;
};

// Per-launch unit counters live in the workspace header (ints from this
// index on), zeroed with it at the start of every call.
constexpr int kHeaderCounter0 = 16;
constexpr int kHeaderCounters = 48;

struct BwdPlan {
  int64_t Tb, Vb;    // block extent (tokens, vocabulary)
  int64_t Tb_pad, Vb_pad;
  int64_t n_tblocks, n_vblocks;
  // off_ctr: one unit counter per GEMM launch (3 per block), right after the
  // header, zeroed with it at the start of every call; tl: the teacher side
  // (none when the backward reads the forward's)
  size_t off_ctr;
  TeacherLayout tl;
  size_t off_G, off_dH, total;
};

bool problem_ok(const kd_kl_problem* p) {
  if (!p) return false;
  if (p->T < 0 || p->d < 8 || p->V < 1 || p->K < 1) return false;
  if (p->K > KDKL_MAX_K || (int64_t)p->K > p->V) return false;
  if (p->T >= (1ll << 31) || p->V >= (1ll << 31) || p->d >= (1ll << 31)) return false;
  if (p->d % 8 != 0) return false;
  if (!(p->temperature > 0.f) || !isfinite(p->temperature)) return false;
  if (p->chunk < 1) return false;
  return true;
}

FwdPlan plan_forward(const kd_kl_problem& p, int num_sms, bool pair, int procs, bool mix = false) {
  (void)num_sms;
  FwdPlan f{};
  const int tile_m = pair ? 2 * BM : BM;
  f.pair = pair;
  const LogitPlan lp = plan_logit(p.T, p.V, p.d, tile_m, fwd_split_tiles());
  f.m_tiles = lp.m_tiles;
  f.n_tiles = lp.n_tiles;
  f.nsplit = p.T > 0 ? lp.nsplit : 1;
  f.group_m = lp.group_m;
  f.grid = (pair ? 2 : 1) * (int)std::min<int64_t>((int64_t)f.m_tiles * f.nsplit, procs);
  f.tl = teacher_layout(kHeaderBytes, p);
  size_t o = f.tl.end;
  f.off_ent = o; o = align256(o + (size_t)p.T * 4);
  f.off_pm = o; o = align256(o + (size_t)f.nsplit * p.T * 4);
  f.off_ps = o; o = align256(o + (size_t)f.nsplit * p.T * 4);
  f.off_pd = o; o = align256(o + (size_t)f.nsplit * p.T * 4);
  f.off_ps1 = o; o = align256(o + (mix ? (size_t)f.nsplit * p.T * 4 : 0));
  f.off_pzl = o; o = align256(o + (mix ? (size_t)f.nsplit * p.T * 4 : 0));
  f.off_bsum = o; o = align256(o + (size_t)combine_blocks((int)std::max<int64_t>(p.T, 1)) * 8);
  f.total = o;
  return f;
}

// Block plans of the backward over the tokens x vocabulary plane, each block
// within the chunk x V budget of the bf16 gradient-of-logits buffer (up to
// 255 columns over it: vocabulary blocks are whole 256-wide tiles, so that
// only the last block has a partial tile in the logits and dW GEMMs).
//   slabs:  all tokens x a vocabulary slab (T <= V), or chunk tokens x all
//           vocabulary (T > V);
//   2D:     about sqrt(budget) tokens x the vocabulary that fits.
// Every block adds its partial dH into the fp32 dH accumulator (one
// read-modify-write of T x d per vocabulary block after the first) and its
// partial dW into dW (one of V x d per token block after the first); the plan
// with the fewer such bytes is taken, 2D only when it saves a quarter.
struct BlockPlan {
  int64_t Tb, Vb, n_tblocks, n_vblocks;
};

BlockPlan slab_plan(const kd_kl_problem& p, int64_t T, double budget) {
  BlockPlan b{};
  if (T <= p.V) {
    b.Tb = T;
    int64_t vb_max = (int64_t)std::min<double>((double)p.V, std::floor(budget / (double)T));
    vb_max = std::max<int64_t>(vb_max, 256);
    b.n_vblocks = ceil_div(p.V, vb_max);
    b.Vb = std::min<int64_t>(round_up(ceil_div(p.V, b.n_vblocks), LOGIT_BN), p.V);
    b.n_vblocks = ceil_div(p.V, b.Vb);
    b.n_tblocks = 1;
  } else {
    b.Vb = p.V;
    b.Tb = std::min<int64_t>(round_up(std::min<int64_t>(p.chunk, T), BM), T);
    b.n_tblocks = ceil_div(T, b.Tb);
    b.n_vblocks = 1;
  }
  return b;
}

BlockPlan square_plan(const kd_kl_problem& p, int64_t T, double budget) {
  BlockPlan b{};
  const int64_t tb = std::min<int64_t>(T, round_up((int64_t)std::sqrt(budget), 256));
  b.n_tblocks = ceil_div(T, tb);
  b.Tb = std::min<int64_t>(round_up(ceil_div(T, b.n_tblocks), 256), T);
  b.n_tblocks = ceil_div(T, b.Tb);
  int64_t vb_max = (int64_t)std::min<double>((double)p.V, std::floor(budget / (double)b.Tb));
  vb_max = std::max<int64_t>(vb_max, 256);
  b.n_vblocks = ceil_div(p.V, vb_max);
  b.Vb = std::min<int64_t>(round_up(ceil_div(p.V, b.n_vblocks), LOGIT_BN), p.V);
  b.n_vblocks = ceil_div(p.V, b.Vb);
  return b;
}

double rmw_bytes(const BlockPlan& b, int64_t T, const kd_kl_problem& p) {
  return 8.0 * (double)p.d *
         ((double)(b.n_vblocks - 1) * (double)T + (double)(b.n_tblocks - 1) * (double)p.V);
}

// own_teacher: the backward prepares the sorted teacher cache itself (sidx,
// sp in its workspace); otherwise it reads the forward's.
BwdPlan plan_backward(const kd_kl_problem& p, bool own_teacher = true) {
  BwdPlan b{};
  const int64_t T = std::max<int64_t>(p.T, 1);
  const double budget = (double)p.chunk * (double)p.V;  // gradient-of-logits elements
  const BlockPlan slab = slab_plan(p, T, budget);
  const BlockPlan sq = square_plan(p, T, budget);
  const char* e2d = getenv("KDKL_BWD_2D");  // tuning: 1 / 0 forces the 2D / slab plan
  const bool two_d = e2d ? (e2d[0] == '1')
                         : (rmw_bytes(sq, T, p) <= 0.75 * rmw_bytes(slab, T, p));
  const BlockPlan& bp = two_d ? sq : slab;
  b.Tb = bp.Tb;
  b.Vb = bp.Vb;
  b.n_tblocks = bp.n_tblocks;
  b.n_vblocks = bp.n_vblocks;
  b.Tb_pad = round_up(b.Tb, BM);
  b.Vb_pad = round_up(b.Vb, LOGIT_BN);
  size_t o = kHeaderBytes;
  b.off_ctr = o; o = align256(o + (size_t)3 * b.n_tblocks * b.n_vblocks * 4);
  b.tl = teacher_layout(o, p);
  if (own_teacher) o = b.tl.end;
  b.off_G = o; o = align256(o + (size_t)b.Tb_pad * b.Vb_pad * 2);
  b.off_dH = o; o = align256(o + (size_t)p.T * p.d * 4);
  b.total = o;
  return b;
}

// ---- offline top-K producer


// nsplit * K at most: bounds the per-split lists in the workspace (8 bytes per
// entry per row: 128 KB per token at this size)
constexpr int kTopkMergeMax = 4096;
// 256: measured faster than 512 (24.86/24.89 vs 25.38/25.23 ms at 32K tokens,
// alternating) and than 128 (26.2) once the first split sets the thresholds;
// smaller lists also leave more of L2 to the operand tiles.
constexpr int kTopkSlackDefault = 256;

// Candidate-list room above K before a row's list is compacted (64 to 512;
// the list holds at most 1024). Smaller slack compacts more often and raises
// the shared thresholds sooner, larger slack compacts less often. Above
// K = 256 the compactions cost more than the thresholds gain and the slack
// doubles: K = 512 took 32.0-32.6 ms per 32K tokens with 512 against
// 34.2-35.1 with 256 (K = 256: 28.2 with 256 against 29.5 with 512).
// KDKL_TOPK_SLACK overrides the default (tuning).
int topk_slack(int K) {
  const char* v = getenv("KDKL_TOPK_SLACK");
  int s = v ? atoi(v) : 0;
  if (s <= 0) s = K > 256 ? 2 * kTopkSlackDefault : kTopkSlackDefault;
  return std::max(64, std::min(512, s));
}

struct TopkPlan {
  bool pair;
  int m_tiles, n_tiles, nsplit, group_m, grid, cap;
  size_t off_cand, off_row_key, off_unit_val, off_unit_id, off_unit_cnt, total;
};

bool topk_problem_ok(const kd_topk_problem* p) {
  return p && p->T >= 0 && p->T < (1ll << 31) && p->d >= 8 && p->d < (1ll << 31) &&
         p->d % 8 == 0 && p->V >= 1 && p->V < (1ll << 31) && p->K >= 1 &&
         p->K <= KDKL_TOPK_MAX_K && (int64_t)p->K <= p->V;
}

TopkPlan plan_topk(const kd_topk_problem& p, int num_sms, bool pair, int procs) {
  (void)num_sms;
  TopkPlan f{};
  const int tile_m = pair ? 2 * BM : BM;
  f.pair = pair;
  const int n_tiles = (int)ceil_div(p.V, LOGIT_BN);
  // Units of about 48 vocabulary tiles (KDKL_TOPK_SPLIT_TILES overrides; a
  // split's K-th logit, the threshold it publishes for its rows, is the
  // sharper the wider the split, and the fewer entries reach the merge:
  // measured at 32K tokens, merge 2.08 / 1.71 / 1.03 / 0.47 ms for 16 / 32 /
  // 48 / 80 tiles with the GEMM within noise, 48 and 80 best in total), but
  // never more than kTopkMergeMax list entries per row (nsplit * K).
  const char* stv = getenv("KDKL_TOPK_SPLIT_TILES");
  const int st0 = stv && atoi(stv) > 0 ? atoi(stv) : 48;
  int st = std::max<int>(st0, (int)ceil_div((int64_t)n_tiles * p.K, kTopkMergeMax));
  while (ceil_div(n_tiles, st) * p.K > kTopkMergeMax && st < n_tiles) ++st;
  const LogitPlan lp = plan_logit(p.T, p.V, p.d, tile_m, st);
  f.m_tiles = lp.m_tiles;
  f.n_tiles = lp.n_tiles;
  f.nsplit = lp.nsplit;
  f.group_m = lp.group_m;
  f.grid = (pair ? 2 : 1) * (int)std::min<int64_t>((int64_t)f.m_tiles * f.nsplit, procs);
  f.cap = std::max(p.K + 64, std::min(1024, p.K + topk_slack(p.K)));
  // two list banks per (CTA, row), any grid <= SMs
  const size_t cand = (size_t)num_sms * BM * 2 * f.cap;
  const size_t unit = (size_t)f.nsplit * p.T * p.K;
  size_t o = kHeaderBytes;
  f.off_cand = o; o = align256(o + cand * 8);
  f.off_row_key = o; o = align256(o + (size_t)p.T * 4);
  f.off_unit_val = o; o = align256(o + unit * 4);
  f.off_unit_id = o; o = align256(o + unit * 4);
  f.off_unit_cnt = o; o = align256(o + (size_t)f.nsplit * p.T * 4);
  f.total = o;
  return f;
}

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// GEMM tiling mode: 2-CTA pairs (cta_group::2, 256-row tiles, half the B
// bytes per CTA) unless KDKL_CTA_PAIR=0 selects single-CTA 128-row tiles.
// Both compute the same sums; the switch exists to compare them.
bool use_pair() {
  const char* v = getenv("KDKL_CTA_PAIR");
  return !(v && v[0] == '0');
}

// KDKL_LOG_PLAN=1 prints each GEMM launch plan to stderr (tuning aid).
bool log_plan() {
  const char* v = getenv("KDKL_LOG_PLAN");
  return v && v[0] == '1';
}

void print_plan(const char* what, bool pair, int procs, const GemmShape& sh, int grid) {
  fprintf(stderr,
          "[kdkl] %s pair=%d procs=%d max_clusters=%d m_tiles=%d n_tiles=%d nsplit=%d "
          "group_m=%d units=%d k_blocks=%d grid=%d dynamic=%d\n",
          what, pair ? 1 : 0, procs, pair ? pair_max_active_clusters() : 0, sh.m_tiles,
          sh.n_tiles, sh.nsplit, sh.group_m, sh.units, sh.k_blocks, grid, sh.counter ? 1 : 0);
}

// Unit processors of the persistent GEMM grid: CTAs, or co-resident CTA pairs.
int gemm_procs(int num_sms, bool pair) {
  if (!pair) return num_sms;
  const int fit = pair_max_active_clusters();
  const int half = num_sms / 2;
  return std::max(1, fit > 0 ? std::min(half, fit) : half);
}

// Failure-detection test hook: with KDKL_INJECT_STALL=1 in the environment the
// GEMM kernels stall on purpose, their bounded waits run out after 2 ms and
// the call reports KD_ERR_TIMEOUT through kd_kl_check_status. Read per call.
int inject_stall_from_env() {
  const char* v = getenv("KDKL_INJECT_STALL");
  return (v && v[0] == '1') ? 1 : 0;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Forward workspaces whose prepared teacher cache a backward may reuse: the
// problem each one was last filled for by a forward call that queued all its
// work. A forward call drops its workspace's entry when it starts and adds it
// back when it has queued everything, so a failed call leaves none.
struct FwdRecord {
  const void* ws;
  int64_t T, d, V;
  int32_t K;
  float temperature;
  size_t bytes;
  const void* mask;  // the forward's mask pointer (its compaction is reused)
};
constexpr size_t kMaxFwdRecords = 64;
std::mutex g_fwd_mu;
std::vector<FwdRecord> g_fwd_records;

void forget_forward(const void* ws) {
  std::lock_guard<std::mutex> lk(g_fwd_mu);
  for (size_t i = 0; i < g_fwd_records.size(); ++i)
    if (g_fwd_records[i].ws == ws) {
      g_fwd_records.erase(g_fwd_records.begin() + (long)i);
      return;
    }
}

void remember_forward(const void* ws, const kd_kl_problem& p, size_t bytes, const void* mask) {
  std::lock_guard<std::mutex> lk(g_fwd_mu);
  for (size_t i = 0; i < g_fwd_records.size(); ++i)
    if (g_fwd_records[i].ws == ws) {
      g_fwd_records.erase(g_fwd_records.begin() + (long)i);
      break;
    }
  if (g_fwd_records.size() >= kMaxFwdRecords) g_fwd_records.erase(g_fwd_records.begin());
  g_fwd_records.push_back(FwdRecord{ws, p.T, p.d, p.V, p.K, p.temperature, bytes, mask});
}

// True when `ws` was last filled by a forward call on the same problem (chunk
// aside: it does not change the teacher cache) with the same mask pointer,
// and the caller says it is at least as long as that call needed.
bool forward_matches(const void* ws, size_t ws_bytes, const kd_kl_problem& p, const void* mask) {
  std::lock_guard<std::mutex> lk(g_fwd_mu);
  for (const FwdRecord& r : g_fwd_records)
    if (r.ws == ws)
      return r.T == p.T && r.d == p.d && r.V == p.V && r.K == p.K &&
             r.temperature == p.temperature && ws_bytes >= r.bytes && r.mask == mask;
  return false;
}

#define KD_CUDA(x)                              \
  do {                                          \
    if ((x) != cudaSuccess) return KD_ERR_CUDA; \
  } while (0)

}  // namespace
}  // namespace kdkl

using namespace kdkl;

// ------------------------------------------------------------------- C ABI

extern "C" {

const char* kd_status_string(kd_status s) {
  switch (s) {
    case KD_OK: return "KD_OK";
    case KD_ERR_INVALID_ARG: return "KD_ERR_INVALID_ARG";
    case KD_ERR_SHAPE: return "KD_ERR_SHAPE";
    case KD_ERR_ALIGNMENT: return "KD_ERR_ALIGNMENT";
    case KD_ERR_INDEX_RANGE: return "KD_ERR_INDEX_RANGE";
    case KD_ERR_WORKSPACE: return "KD_ERR_WORKSPACE";
    case KD_ERR_CUDA: return "KD_ERR_CUDA";
    case KD_ERR_TIMEOUT: return "KD_ERR_TIMEOUT";
    case KD_ERR_UNSUPPORTED: return "KD_ERR_UNSUPPORTED";
  }
  return "KD_ERR_UNKNOWN";
}

int64_t kd_launch_count(void) { return g_launches.load(); }

size_t kd_kl_workspace_size(const kd_kl_problem* prob, int which) {
  if (!problem_ok(prob)) return 0;
  if (which == 0 || which == 2) {
    const bool mix = which == 2;
    DeviceInfo di;
    const int sms = (device_info(&di) == KD_OK) ? di.num_sms : 148;
    // The split count depends on the SM count and the tiling mode; size for
    // the larger of the two modes so the answer holds for either.
    // Pair plans are sized for any number of co-resident clusters up to sms/2.
    size_t total = plan_forward(*prob, sms, false, sms, mix).total;
    for (int procs = 1; procs <= sms / 2; ++procs)
      total = std::max(total, plan_forward(*prob, sms, true, procs, mix).total);
    return total;
  }
  if (which == 1 || which == 3) return plan_backward(*prob).total;
  if (which == 4) return plan_backward(*prob, false).total;
  return 0;
}

struct MixWeights {
  float kl, ce;  // per-token loss = kl * KL + ce * CE
};

static MixWeights mix_weights(const kd_kl_problem& p, const kd_kl_options& o) {
  const float c = o.scale_tau_sq ? p.temperature * p.temperature : 1.0f;
  return MixWeights{o.alpha * c, 1.0f - o.alpha};
}

static kd_status validate_options(const kd_kl_problem* prob, const kd_kl_options* o) {
  if (!(o->alpha >= 0.0f && o->alpha <= 1.0f)) return KD_ERR_INVALID_ARG;
  if (o->alpha < 1.0f && prob->T > 0 && !o->labels) return KD_ERR_INVALID_ARG;
  if (!aligned(o->labels, 4)) return KD_ERR_ALIGNMENT;
  return KD_OK;
}

static kd_status validate_common(const kd_kl_problem* prob, const void* H, const void* W,
                                 const void* idx, const void* logit, const void* workspace) {
  if (!prob) return KD_ERR_INVALID_ARG;
  if (prob->T < 0 || prob->d < 8 || prob->V < 1 || prob->K < 1 || prob->K > KDKL_MAX_K ||
      (int64_t)prob->K > prob->V || prob->T >= (1ll << 31) || prob->V >= (1ll << 31) ||
      prob->d >= (1ll << 31))
    return KD_ERR_SHAPE;
  if (!(prob->temperature > 0.f) || !isfinite(prob->temperature) || prob->chunk < 1)
    return KD_ERR_INVALID_ARG;
  if (prob->d % 8 != 0) return KD_ERR_ALIGNMENT;
  if (!workspace) return KD_ERR_WORKSPACE;
  if (prob->T > 0 && (!H || !idx || !logit)) return KD_ERR_INVALID_ARG;
  if (!W) return KD_ERR_INVALID_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(workspace, 16)) return KD_ERR_ALIGNMENT;
  if (!aligned(idx, 4) || !aligned(logit, 4)) return KD_ERR_ALIGNMENT;
  return KD_OK;
}

static kd_status forward_impl(const kd_kl_problem* prob, const kd_kl_options* opts,
                              const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                              const float* topk_logit, const uint8_t* mask, float* loss, float* lse,
                              float* lse1, float* token_kl, void* workspace,
                              size_t workspace_bytes, void* stream_ptr) {
  kd_status st = validate_common(prob, H, W, topk_idx, topk_logit, workspace);
  if (st != KD_OK) return st;
  if (!loss || (prob->T > 0 && !lse)) return KD_ERR_INVALID_ARG;
  if (!aligned(loss, 4) || !aligned(lse, 4) || !aligned(token_kl, 4)) return KD_ERR_ALIGNMENT;
  const bool mix = opts != nullptr;
  if (mix && ((st = validate_options(prob, opts)) != KD_OK)) return st;
  if (mix && prob->T > 0 && !lse1) return KD_ERR_INVALID_ARG;
  if (!aligned(lse1, 4)) return KD_ERR_ALIGNMENT;
  DeviceInfo di;
  if ((st = device_info(&di)) != KD_OK) return st;
  if ((st = get_encoder()) != KD_OK) return st;
  const kd_kl_problem& p = *prob;
  const bool pair = use_pair();
  const FwdPlan f = plan_forward(p, di.num_sms, pair, gemm_procs(di.num_sms, pair), mix);
  if (workspace_bytes < f.total) return KD_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  forget_forward(workspace);

  int* status = at<int>(workspace, 0);
  int* n_count = status + 1;
  KD_CUDA(cudaMemsetAsync(workspace, 0, kHeaderBytes, stream));
  if (p.T == 0) {
    KD_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), stream));
    remember_forward(workspace, p, f.tl.end, mask);
    return KD_OK;
  }
  const int T = (int)p.T, K = p.K, V = (int)p.V, d = (int)p.d;
  const float inv_tau = 1.0f / p.temperature;
  const float cl2 = 1.4426950408889634f * inv_tau;
  int32_t* sidx = at<int32_t>(workspace, f.tl.off_sidx);
  float* sp = at<float>(workspace, f.tl.off_sp);
  float* ent = at<float>(workspace, f.off_ent);
  // With a mask, the counted tokens are compacted first and every step
  // after that runs on them only: masked tokens cost no tensor-core work.
  const bool compact = mask != nullptr;
  int* rowmap = compact ? at<int>(workspace, f.tl.off_rowmap) : nullptr;
  int* invmap = compact ? at<int>(workspace, f.tl.off_invmap) : nullptr;
  uint16_t* Hc = at<uint16_t>(workspace, f.tl.off_Hc);
  const int64_t T_pad = round_up(T, 2 * BM);
  if (compact) {
    KD_CUDA(launch_mask_scan(mask, T, rowmap, invmap, n_count, stream));
    KD_CUDA(launch_gather_rows(H, d, rowmap, n_count, T_pad, 2 * BM, Hc, di.num_sms, stream));
  }
  KD_CUDA(launch_teacher_prep(topk_idx, topk_logit, mask, mix ? opts->labels : nullptr, rowmap, T,
                              K, V, inv_tau, sidx, sp, ent, n_count, status, stream));

  CUtensorMap tmH, tmW;
  const int b_rows = f.pair ? LOGIT_BN / 2 : LOGIT_BN;  // W rows one CTA loads per tile
  if (!encode_bf16_2d(&tmH, compact ? Hc : H, d, compact ? T_pad : T, d, BK, BM) ||
      !encode_bf16_2d(&tmW, W, d, V, d, BK, b_rows))
    return KD_ERR_CUDA;
  GemmShape sh{};
  sh.inject_stall = inject_stall_from_env();
  sh.m_tiles = f.m_tiles;
  sh.n_tiles = f.n_tiles;
  sh.nsplit = f.nsplit;
  sh.group_m = f.group_m;
  sh.units = f.m_tiles * f.nsplit;
  sh.k_blocks = (int)ceil_div(d, BK);
  sh.counter = static_schedule() ? nullptr : status + kHeaderCounter0;
  if (compact) {
    sh.dyn_rows = n_count;
    sh.dyn_base = 0;
    sh.dyn_cap = T;
    sh.dyn_dim = 0;
  }
  EpiParams ep{};
  ep.rowmap = rowmap;
  ep.sidx = sidx;
  ep.sp = sp;
  ep.K = K;
  ep.T = T;
  ep.row0 = 0;
  ep.rows = T;
  ep.col0 = 0;
  ep.cols = V;
  ep.cl2 = cl2;
  ep.pm = at<float>(workspace, f.off_pm);
  ep.ps = at<float>(workspace, f.off_ps);
  ep.pd = at<float>(workspace, f.off_pd);
  if (mix) {
    ep.labels = opts->labels;
    ep.same_tau = p.temperature == 1.0f ? 1 : 0;
    ep.ps1 = at<float>(workspace, f.off_ps1);
    ep.pzl = at<float>(workspace, f.off_pzl);
  }
  if (log_plan()) print_plan("fwd_lse", f.pair, gemm_procs(di.num_sms, f.pair), sh, f.grid);
  KD_CUDA(launch_gemm(mix ? GEMM_FWD_LSE_MIX : GEMM_FWD_LSE, LOGIT_BN, f.pair, tmH, tmW, sh, ep,
                      status, f.grid, stream));

  double* bsum = at<double>(workspace, f.off_bsum);
  if (mix) {
    const MixWeights mw = mix_weights(p, *opts);
    KD_CUDA(launch_lse_combine_mix(ep.pm, ep.ps, ep.pd, ep.ps1, ep.pzl, f.nsplit, T, ent, mask,
                                   invmap, cl2, inv_tau, mw.kl, mw.ce, lse, lse1, token_kl, bsum,
                                   stream));
  } else {
    KD_CUDA(launch_lse_combine(ep.pm, ep.ps, ep.pd, f.nsplit, T, ent, mask, invmap, cl2, inv_tau,
                               lse, token_kl, bsum, stream));
  }
  KD_CUDA(launch_loss_finalize(bsum, combine_blocks(T), n_count, loss, stream));
  // the teacher side (header with N, sorted ids and p, the compaction) is
  // what a backward reuses
  remember_forward(workspace, p, f.tl.end, mask);
  return KD_OK;
}

kd_status kd_kl_forward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                        const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                        float* loss, float* lse, float* token_kl, void* workspace,
                        size_t workspace_bytes, void* stream_ptr) {
  return forward_impl(prob, nullptr, H, W, topk_idx, topk_logit, mask, loss, lse, nullptr,
                      token_kl, workspace, workspace_bytes, stream_ptr);
}

kd_status kd_kl_forward_ex(const kd_kl_problem* prob, const kd_kl_options* opts,
                           const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                           const float* topk_logit, const uint8_t* mask, float* loss, float* lse,
                           float* lse1, float* token_loss, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!opts) return KD_ERR_INVALID_ARG;
  return forward_impl(prob, opts, H, W, topk_idx, topk_logit, mask, loss, lse, lse1, token_loss,
                      workspace, workspace_bytes, stream);
}

static kd_status backward_impl(const kd_kl_problem* prob, const kd_kl_options* opts,
                               const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                               const float* topk_logit, const uint8_t* mask, const float* lse,
                               const float* lse1, float grad_loss, uint16_t* dH, float* dW,
                               int accumulate_dW, void* workspace, size_t workspace_bytes,
                               void* stream_ptr, const void* fwd_ws = nullptr,
                               size_t fwd_ws_bytes = 0) {
  const bool reuse = fwd_ws != nullptr;
  // With a reused forward workspace the teacher cache is not read: stand-in
  // non-null pointers pass the common checks.
  kd_status st = validate_common(prob, H, W, reuse ? fwd_ws : topk_idx,
                                 reuse ? fwd_ws : topk_logit, workspace);
  if (st != KD_OK) return st;
  if (reuse && !forward_matches(fwd_ws, fwd_ws_bytes, *prob, mask)) return KD_ERR_INVALID_ARG;
  const bool mix = opts != nullptr;
  if (mix && ((st = validate_options(prob, opts)) != KD_OK)) return st;
  // temperature-1 logsumexp: needed when the CE term is on and tau != 1
  if (mix && prob->T > 0 && !lse1 && opts->alpha < 1.0f && prob->temperature != 1.0f)
    return KD_ERR_INVALID_ARG;
  if (!aligned(lse1, 4)) return KD_ERR_ALIGNMENT;
  if (!dW || (prob->T > 0 && (!lse || !dH))) return KD_ERR_INVALID_ARG;
  if (!isfinite(grad_loss)) return KD_ERR_INVALID_ARG;
  if (!aligned(dH, 16) || !aligned(dW, 16) || !aligned(lse, 4)) return KD_ERR_ALIGNMENT;
  DeviceInfo di;
  if ((st = device_info(&di)) != KD_OK) return st;
  if ((st = get_encoder()) != KD_OK) return st;
  const kd_kl_problem& p = *prob;
  const BwdPlan b = plan_backward(p, !reuse);
  if (workspace_bytes < b.total) return KD_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  int* status = at<int>(workspace, 0);
  // the counted-token total N: this call's own, or the forward's
  int* n_count = reuse ? const_cast<int*>(static_cast<const int*>(fwd_ws)) + 1 : status + 1;
  KD_CUDA(cudaMemsetAsync(workspace, 0, b.tl.off_sidx, stream));  // header and unit counters
  int* counters = static_schedule() ? nullptr : at<int>(workspace, b.off_ctr);
  int launch_no = 0;  // index of the next GEMM launch's counter
  auto next_counter = [&]() { return counters ? counters + launch_no++ : nullptr; };
  if (p.T == 0) {
    if (!accumulate_dW) KD_CUDA(cudaMemsetAsync(dW, 0, (size_t)p.V * p.d * 4, stream));
    return KD_OK;
  }
  const int T = (int)p.T, K = p.K, V = (int)p.V, d = (int)p.d;
  const float inv_tau = 1.0f / p.temperature;
  const float cl2 = 1.4426950408889634f * inv_tau;
  // The teacher side (sorted ids and p; with a mask, the compaction of the
  // counted tokens): the forward workspace's, at the same offsets, or
  // prepared here.
  char* tws = reuse ? static_cast<char*>(const_cast<void*>(fwd_ws)) : static_cast<char*>(workspace);
  const TeacherLayout tl = reuse ? teacher_layout(kHeaderBytes, p) : b.tl;
  int32_t* sidx = at<int32_t>(tws, tl.off_sidx);
  float* sp = at<float>(tws, tl.off_sp);
  const bool compact = mask != nullptr;
  int* rowmap = compact ? at<int>(tws, tl.off_rowmap) : nullptr;
  int* invmap = compact ? at<int>(tws, tl.off_invmap) : nullptr;
  uint16_t* Hc = at<uint16_t>(tws, tl.off_Hc);
  const int64_t T_pad = round_up(T, 2 * BM);
  uint16_t* Gbuf = at<uint16_t>(workspace, b.off_G);
  float* dH_acc = at<float>(workspace, b.off_dH);

  if (!reuse) {
    if (compact) {
      KD_CUDA(launch_mask_scan(mask, T, rowmap, invmap, n_count, stream));
      KD_CUDA(launch_gather_rows(H, d, rowmap, n_count, T_pad, 2 * BM, Hc, di.num_sms, stream));
    }
    KD_CUDA(launch_teacher_prep(topk_idx, topk_logit, mask, mix ? opts->labels : nullptr, rowmap,
                                T, K, V, inv_tau, sidx, sp, nullptr, n_count, status, stream));
  }

  const bool pair = use_pair();
  const int tile_m = pair ? 2 * BM : BM;
  const int procs = gemm_procs(di.num_sms, pair);
  const int cta_per_proc = pair ? 2 : 1;
  // Rows of the token operand: the compacted counted tokens, or H itself.
  const uint16_t* Hop = compact ? Hc : H;
  const int64_t H_rows = compact ? T_pad : T;
  CUtensorMap tmH_K, tmW_K, tmW_MN, tmH_MN;
  if (!encode_bf16_2d(&tmH_K, Hop, d, H_rows, d, BK, BM) ||
      !encode_bf16_2d(&tmW_K, W, d, V, d, BK, pair ? LOGIT_BN / 2 : LOGIT_BN) ||
      !encode_bf16_2d(&tmW_MN, W, d, V, d, 64, BK) ||
      !encode_bf16_2d(&tmH_MN, Hop, d, H_rows, d, 64, BK))
    return KD_ERR_CUDA;

  // N tile of the dH / dW GEMMs (hidden dimension). 192-wide tiles avoid the
  // zero-padded columns when d % 256 != 0 but measured slower on d = 2880
  // (more operand bytes per MAC), so 256 is used throughout.
  const int out_bn = 256;
  const int dn_tiles = (int)ceil_div(d, out_bn);
  // When the last column tile of d holds at most half a tile (d = 2880:
  // 11 x 256 + 64), it runs as a 128-wide tile (KDKL_NARROW_LAST=0 keeps the
  // full width, to compare).
  const char* nl_env = getenv("KDKL_NARROW_LAST");
  const int narrow_last =
      (d % out_bn != 0 && d % out_bn <= out_bn / 2 && !(nl_env && nl_env[0] == '0')) ? 1 : 0;
  const int stall = inject_stall_from_env();
  for (int64_t tb = 0; tb < b.n_tblocks; ++tb) {
    const int row0 = (int)(tb * b.Tb);
    const int rows = (int)std::min<int64_t>(b.Tb, p.T - row0);
    for (int64_t vb = 0; vb < b.n_vblocks; ++vb) {
      const int col0 = (int)(vb * b.Vb);
      const int cols = (int)std::min<int64_t>(b.Vb, p.V - col0);
      if (cols <= 0 || rows <= 0) continue;

      // 1) recompute the logits of the block and store (softmax - P) * m g / (tau N)
      {
        // Units of 2 vocabulary tiles: nothing runs across tiles but each
        // row's cursor into its teacher ids, and short units keep the tail
        // of these short launches small.
        const LogitPlan lp = plan_logit(rows, cols, d, tile_m, 2);
        GemmShape sh{};
        sh.inject_stall = stall;
        sh.m_tiles = lp.m_tiles;
        sh.n_tiles = lp.n_tiles;
        sh.nsplit = lp.nsplit;
        sh.group_m = lp.group_m;
        sh.units = lp.units;
        sh.k_blocks = (int)ceil_div(d, BK);
        sh.a_m0 = row0;
        sh.b_n0 = col0;
        sh.counter = next_counter();
        if (compact) {  // only the block's counted tokens
          sh.dyn_rows = n_count;
          sh.dyn_base = row0;
          sh.dyn_cap = rows;
          sh.dyn_dim = 0;
        }
        EpiParams ep{};
        ep.rowmap = rowmap;
        ep.sidx = sidx;
        ep.sp = sp;
        ep.K = K;
        ep.T = T;
        ep.row0 = row0;
        ep.rows = rows;
        ep.col0 = col0;
        ep.cols = cols;
        ep.cl2 = cl2;
        ep.lse = lse;
        ep.mask = compact ? nullptr : mask;
        ep.n_count = n_count;
        ep.g_over_tau = grad_loss * inv_tau;
        ep.G = Gbuf;
        ep.ldg = b.Vb_pad;
        if (mix) {
          const MixWeights mw = mix_weights(p, *opts);
          ep.labels = opts->labels;
          ep.same_tau = p.temperature == 1.0f ? 1 : 0;
          ep.lse1 = lse1 ? lse1 : lse;
          ep.kl_weight = grad_loss * mw.kl * inv_tau;
          ep.ce_weight = grad_loss * mw.ce;
        }
        const int grid = cta_per_proc * (int)std::min<int64_t>(sh.units, procs);
        if (log_plan() && vb == 0 && tb == 0) print_plan("bwd_grad", pair, procs, sh, grid);
        KD_CUDA(launch_gemm(mix ? GEMM_BWD_GRAD_MIX : GEMM_BWD_GRAD, LOGIT_BN, pair, tmH_K, tmW_K,
                            sh, ep, status, grid, stream));
      }
      // 2) dH[rows] (+)= G . W[cols] and 3) dW[cols] (+)= G^T . H[rows]: two
      // launches, or for small blocks one whose units run the job with the
      // longer units first, so the short ones fill its tail. Each output
      // element still gets one store or one add per launch, in stream order:
      // deterministic.
      CUtensorMap tmG_K, tmG_MN;
      if (!encode_bf16_2d(&tmG_K, Gbuf, cols, rows, b.Vb_pad, BK, BM) ||
          !encode_bf16_2d(&tmG_MN, Gbuf, cols, rows, b.Vb_pad, 64, BK))
        return KD_ERR_CUDA;
      GemmShape sh_dh{};
      sh_dh.inject_stall = stall;
      sh_dh.m_tiles = (int)ceil_div(rows, tile_m);
      sh_dh.n_tiles = dn_tiles;
      sh_dh.nsplit = dn_tiles;
      sh_dh.group_m = 1;  // m-major: an m-tile's output tiles run side by side
      sh_dh.units = sh_dh.m_tiles * sh_dh.nsplit;
      sh_dh.k_blocks = (int)ceil_div(cols, BK);
      sh_dh.b_k0 = col0;
      sh_dh.narrow_last = narrow_last;
      if (compact) {
        sh_dh.dyn_rows = n_count;
        sh_dh.dyn_base = row0;
        sh_dh.dyn_cap = rows;
        sh_dh.dyn_dim = 0;  // M: the block's counted tokens
      }
      EpiParams ep_dh{};
      ep_dh.out = dH_acc + (int64_t)row0 * d;
      ep_dh.ldo = d;
      ep_dh.out_rows = rows;
      ep_dh.out_cols = d;
      ep_dh.accumulate = vb > 0 ? 1 : 0;
      GemmShape sh_dw{};
      sh_dw.inject_stall = stall;
      sh_dw.m_tiles = (int)ceil_div(cols, tile_m);
      sh_dw.n_tiles = dn_tiles;
      sh_dw.nsplit = dn_tiles;
      sh_dw.group_m = 1;
      sh_dw.units = sh_dw.m_tiles * sh_dw.nsplit;
      sh_dw.k_blocks = (int)ceil_div(rows, BK);
      sh_dw.b_k0 = row0;
      sh_dw.narrow_last = narrow_last;
      if (compact) {
        sh_dw.dyn_rows = n_count;
        sh_dw.dyn_base = row0;
        sh_dw.dyn_cap = rows;
        sh_dw.dyn_dim = 1;  // K: the block's counted tokens
      }
      EpiParams ep_dw{};
      ep_dw.out = dW + (int64_t)col0 * d;
      ep_dw.ldo = d;
      ep_dw.out_rows = cols;
      ep_dw.out_cols = d;
      ep_dw.accumulate = (accumulate_dW || tb > 0) ? 1 : 0;
      // One launch pays only when both jobs are small (together at most two
      // waves of units): it saves a launch and a tail where each is a large
      // share of the work; the job with the longer units goes first. Otherwise
      // two launches, which measured faster even with a partial last wave
      // (their units start together and share operand tiles in L2): 15.6-15.8
      // vs 16.1-16.5 ms per step for 8K tokens of the Llama-3B-like head, whose
      // dH has 5.05 waves; 54.1-54.4 vs 54.7-55.0 ms for the padded 4 x 8K
      // batch at chunk 512; 45.7 vs 47.4 ms at 16K tokens of the GPT-OSS-like
      // head. At 256 tokens one launch is faster (0.283 vs 0.335 ms per step).
      const char* dual_env = getenv("KDKL_DUAL_DHDW");  // 1: always one launch, 0: never
      const bool dual = dual_env ? dual_env[0] == '1'
                                 : ((int64_t)sh_dw.units + sh_dh.units <= 2 * (int64_t)procs);
      if (!dual) {
        sh_dh.counter = next_counter();
        int grid = cta_per_proc * (int)std::min<int64_t>(sh_dh.units, procs);
        if (log_plan() && vb == 0 && tb == 0) print_plan("dH", pair, procs, sh_dh, grid);
        KD_CUDA(launch_gemm(GEMM_DH, out_bn, pair, tmG_K, tmW_MN, sh_dh, ep_dh, status, grid,
                            stream));
        sh_dw.counter = next_counter();
        grid = cta_per_proc * (int)std::min<int64_t>(sh_dw.units, procs);
        if (log_plan() && vb == 0 && tb == 0) print_plan("dW", pair, procs, sh_dw, grid);
        KD_CUDA(launch_gemm(GEMM_DW, out_bn, pair, tmG_MN, tmH_MN, sh_dw, ep_dw, status, grid,
                            stream));
      } else {
        // the launch's one counter, read from job 0's shape
        sh_dw.counter = sh_dh.counter = next_counter();
        const int grid =
            cta_per_proc * (int)std::min<int64_t>((int64_t)sh_dw.units + sh_dh.units, procs);
        if (log_plan() && vb == 0 && tb == 0) {
          print_plan("dW (job 0)", pair, procs, sh_dw, grid);
          print_plan("dH (job 1)", pair, procs, sh_dh, grid);
        }
        const bool dh_first = sh_dh.k_blocks > sh_dw.k_blocks;  // longer units first
        KD_CUDA(launch_gemm_dw_dh(pair, dh_first, tmG_MN, tmH_MN, sh_dw, ep_dw, tmG_K, tmW_MN,
                                  sh_dh, ep_dh, status, grid, stream));
      }
    }
  }
  // dH rows back to the callers' tokens; masked rows are exact zeros
  KD_CUDA(launch_f32_to_bf16(dH_acc, dH, (long long)p.T * p.d, d, invmap, di.num_sms, stream));
  return KD_OK;
}

kd_status kd_kl_backward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                         const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                         const float* lse, float grad_loss, uint16_t* dH, float* dW,
                         int accumulate_dW, void* workspace, size_t workspace_bytes,
                         void* stream_ptr) {
  return backward_impl(prob, nullptr, H, W, topk_idx, topk_logit, mask, lse, nullptr, grad_loss, dH,
                       dW, accumulate_dW, workspace, workspace_bytes, stream_ptr);
}

kd_status kd_kl_backward_ex(const kd_kl_problem* prob, const kd_kl_options* opts,
                            const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                            const float* topk_logit, const uint8_t* mask, const float* lse,
                            const float* lse1, float grad_loss, uint16_t* dH, float* dW,
                            int accumulate_dW, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!opts) return KD_ERR_INVALID_ARG;
  return backward_impl(prob, opts, H, W, topk_idx, topk_logit, mask, lse, lse1, grad_loss, dH, dW,
                       accumulate_dW, workspace, workspace_bytes, stream);
}

kd_status kd_kl_backward_reuse(const kd_kl_problem* prob, const kd_kl_options* opts,
                               const uint16_t* H, const uint16_t* W, const uint8_t* mask,
                               const float* lse, const float* lse1, const void* fwd_workspace,
                               size_t fwd_workspace_bytes, float grad_loss, uint16_t* dH,
                               float* dW, int accumulate_dW, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!fwd_workspace) return KD_ERR_INVALID_ARG;
  return backward_impl(prob, opts, H, W, nullptr, nullptr, mask, lse, lse1, grad_loss, dH, dW,
                       accumulate_dW, workspace, workspace_bytes, stream, fwd_workspace,
                       fwd_workspace_bytes);
}

static bool rkl_problem_ok(const kd_kl_problem* p) {
  return problem_ok(p) && p->T * (int64_t)p->K < (1ll << 31);
}

size_t kd_rkl_workspace_size(const kd_kl_problem* prob) {
  if (!rkl_problem_ok(prob)) return 0;
  return rkl_layout(prob->T, prob->d, prob->K, prob->V, kHeaderBytes).total;
}

static kd_status rkl_validate(const kd_kl_problem* prob, const void* H, const void* W,
                              const void* idx, const void* logit, const void* workspace,
                              size_t workspace_bytes, const void* grad_z) {
  kd_status st = validate_common(prob, H, W, idx, logit, workspace);
  if (st != KD_OK) return st;
  if (prob->T * (int64_t)prob->K >= (1ll << 31)) return KD_ERR_SHAPE;
  if (!aligned(grad_z, 4)) return KD_ERR_ALIGNMENT;
  if (workspace_bytes < kd_rkl_workspace_size(prob)) return KD_ERR_WORKSPACE;
  return KD_OK;
}

kd_status kd_rkl_forward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                         const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                         float* loss, float* token_rkl, float* grad_z, void* workspace,
                         size_t workspace_bytes, void* stream_ptr) {
  kd_status st =
      rkl_validate(prob, H, W, topk_idx, topk_logit, workspace, workspace_bytes, grad_z);
  if (st != KD_OK) return st;
  if (!loss) return KD_ERR_INVALID_ARG;
  if (!aligned(loss, 4) || !aligned(token_rkl, 4)) return KD_ERR_ALIGNMENT;
  DeviceInfo di;
  if ((st = device_info(&di)) != KD_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int* status = at<int>(workspace, 0);
  KD_CUDA(cudaMemsetAsync(workspace, 0, kHeaderBytes, stream));
  if (prob->T == 0) {
    KD_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), stream));
    return KD_OK;
  }
  const RklLayout L = rkl_layout(prob->T, prob->d, prob->K, prob->V, kHeaderBytes);
  KD_CUDA(rkl_forward(L, H, W, topk_idx, topk_logit, mask, (int)prob->T, (int)prob->d, prob->K,
                      (int)prob->V, 1.0f / prob->temperature, token_rkl, grad_z, loss, workspace,
                      status, status + 1, di.num_sms, stream));
  return KD_OK;
}

kd_status kd_rkl_backward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                          const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                          const float* grad_z, float grad_loss, uint16_t* dH, float* dW,
                          int accumulate_dW, void* workspace, size_t workspace_bytes,
                          void* stream_ptr) {
  kd_status st =
      rkl_validate(prob, H, W, topk_idx, topk_logit, workspace, workspace_bytes, grad_z);
  if (st != KD_OK) return st;
  if (!dW || (prob->T > 0 && !dH)) return KD_ERR_INVALID_ARG;
  if (!isfinite(grad_loss)) return KD_ERR_INVALID_ARG;
  if (!aligned(dH, 16) || !aligned(dW, 16)) return KD_ERR_ALIGNMENT;
  DeviceInfo di;
  if ((st = device_info(&di)) != KD_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int* status = at<int>(workspace, 0);
  KD_CUDA(cudaMemsetAsync(workspace, 0, kHeaderBytes, stream));
  if (prob->T == 0) {
    if (!accumulate_dW) KD_CUDA(cudaMemsetAsync(dW, 0, (size_t)prob->V * prob->d * 4, stream));
    return KD_OK;
  }
  const RklLayout L = rkl_layout(prob->T, prob->d, prob->K, prob->V, kHeaderBytes);
  KD_CUDA(rkl_backward(L, H, W, topk_idx, topk_logit, mask, (int)prob->T, (int)prob->d, prob->K,
                       (int)prob->V, 1.0f / prob->temperature, grad_z, grad_loss, dH, dW,
                       accumulate_dW ? 1 : 0, workspace, status, status + 1, di.num_sms, stream));
  return KD_OK;
}

size_t kd_lmhead_topk_workspace_size(const kd_topk_problem* prob) {
  if (!topk_problem_ok(prob)) return 0;
  DeviceInfo di;
  const int sms = (device_info(&di) == KD_OK) ? di.num_sms : 160;
  size_t total = plan_topk(*prob, sms, false, sms).total;
  for (int procs = 1; procs <= sms / 2; ++procs)
    total = std::max(total, plan_topk(*prob, sms, true, procs).total);
  return total;
}

kd_status kd_lmhead_topk(const kd_topk_problem* prob, const uint16_t* H, const uint16_t* W,
                         int32_t* topk_idx, float* topk_logit, void* workspace,
                         size_t workspace_bytes, void* stream_ptr) {
  if (!prob) return KD_ERR_INVALID_ARG;
  if (!topk_problem_ok(prob)) return (prob->d % 8 != 0 && prob->d >= 8) ? KD_ERR_ALIGNMENT
                                                                        : KD_ERR_SHAPE;
  if (!workspace) return KD_ERR_WORKSPACE;
  if (!W || (prob->T > 0 && (!H || !topk_idx || !topk_logit))) return KD_ERR_INVALID_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(workspace, 16) || !aligned(topk_idx, 4) ||
      !aligned(topk_logit, 4))
    return KD_ERR_ALIGNMENT;
  DeviceInfo di;
  kd_status st;
  if ((st = device_info(&di)) != KD_OK) return st;
  if ((st = get_encoder()) != KD_OK) return st;
  const kd_topk_problem& p = *prob;
  const bool pair = use_pair();
  const int procs = gemm_procs(di.num_sms, pair);
  const TopkPlan f = plan_topk(p, di.num_sms, pair, procs);
  if (workspace_bytes < f.total) return KD_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int* status = at<int>(workspace, 0);
  KD_CUDA(cudaMemsetAsync(workspace, 0, kHeaderBytes, stream));
  if (p.T == 0) return KD_OK;
  const int T = (int)p.T, d = (int)p.d, V = (int)p.V, K = p.K;

  CUtensorMap tmH, tmW;
  if (!encode_bf16_2d(&tmH, H, d, T, d, BK, BM) ||
      !encode_bf16_2d(&tmW, W, d, V, d, BK, pair ? LOGIT_BN / 2 : LOGIT_BN))
    return KD_ERR_CUDA;
  GemmShape sh{};
  sh.inject_stall = inject_stall_from_env();
  sh.m_tiles = f.m_tiles;
  sh.n_tiles = f.n_tiles;
  sh.nsplit = f.nsplit;
  sh.group_m = f.group_m;
  sh.units = f.m_tiles * f.nsplit;
  sh.k_blocks = (int)ceil_div(d, BK);
  sh.counter = static_schedule() ? nullptr : status + kHeaderCounter0;
  EpiParams ep{};
  ep.K = K;
  ep.T = T;
  ep.row0 = 0;
  ep.rows = T;
  ep.col0 = 0;
  ep.cols = V;
  ep.topk_cap = f.cap;
  // One split of every row runs first, alone: the row's other splits then
  // start from the threshold it published instead of compacting from -inf
  // (measured: the MMA's wait on the epilogue halves, 4 % fewer cycles).
  // Only when there are at least as many m-tiles as unit processors: with
  // fewer, that phase does not fill the GPU and the rows' other splits run
  // beside it anyway (8K tokens: 6.13 ms without it, 6.19-6.51 with it).
  sh.first_group = (f.nsplit > 1 && f.m_tiles >= procs) ? 1 : 0;
  // That first split is half as wide as the others' even share: enough
  // vocabulary for a useful threshold, and half as long in the phase where
  // ~all m-tiles are in flight at once and their A rows do not fit in L2.
  // Measured at 32K tokens, alternating on one box: 26.04-26.45 ms, against
  // 26.82-26.86 with no first split and 27.26-27.28 with a full-width one.
  if (sh.first_group) sh.first_ntiles = std::max(1, sh.n_tiles / (2 * sh.nsplit));
  ep.cand = at<float2>(workspace, f.off_cand);
  ep.row_key = at<uint32_t>(workspace, f.off_row_key);
  KD_CUDA(cudaMemsetAsync(ep.row_key, 0, (size_t)T * 4, stream));
  ep.unit_val = at<float>(workspace, f.off_unit_val);
  ep.unit_id = at<int32_t>(workspace, f.off_unit_id);
  ep.unit_cnt = at<int>(workspace, f.off_unit_cnt);
  if (log_plan()) print_plan("topk", pair, procs, sh, f.grid);
  KD_CUDA(launch_gemm(GEMM_TOPK, LOGIT_BN, pair, tmH, tmW, sh, ep, status, f.grid, stream));
  KD_CUDA(launch_topk_merge(ep.unit_val, ep.unit_id, ep.unit_cnt, ep.row_key, f.nsplit, T, K,
                            topk_idx,
                            topk_logit, stream));
  return KD_OK;
}

kd_status kd_kl_check_status(void* workspace, void* stream_ptr) {
  if (!workspace) return KD_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int code = 0;
  if (cudaMemcpyAsync(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return KD_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KD_ERR_CUDA;
  switch (code) {
    case 0: return KD_OK;
    case DEV_ERR_INVALID_ARG: return KD_ERR_INVALID_ARG;
    case DEV_ERR_INDEX_RANGE: return KD_ERR_INDEX_RANGE;
    case DEV_ERR_TIMEOUT: return KD_ERR_TIMEOUT;
    default: return KD_ERR_CUDA;
  }
}

kd_status kd_timing_begin(void) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing.store(true, std::memory_order_release);
  return KD_OK;
}

kd_status kd_timing_end(kd_kernel_time* out, int max_entries, int* n_entries) {
  g_timing.store(false, std::memory_order_release);
  std::vector<PendingTiming> pend;
  {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    pend.swap(g_pending);
  }
  std::vector<kd_kernel_time> rows;
  kd_status st = KD_OK;
  for (auto& p : pend) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess)
      st = KD_ERR_CUDA;
    cudaEventDestroy(p.start);
    cudaEventDestroy(p.stop);
    auto it = std::find_if(rows.begin(), rows.end(),
                           [&](const kd_kernel_time& r) { return strcmp(r.name, p.name) == 0; });
    if (it == rows.end()) {
      kd_kernel_time r{};
      snprintf(r.name, sizeof(r.name), "%s", p.name);
      rows.push_back(r);
      it = rows.end() - 1;
    }
    it->launches += 1;
    it->total_ms += ms;
  }
  const int n = (int)std::min<size_t>(rows.size(), (size_t)std::max(max_entries, 0));
  for (int i = 0; i < n && out; ++i) out[i] = rows[i];
  if (n_entries) *n_entries = (int)rows.size();
  return st;
}

}  // extern "C"
