/*
 * kdkl.h — C ABI of the fused chunked KL distillation loss for GB300 (sm_103a).
 *
 * The operation is the one the pages state ("Making knowledge distillation
 * cheap enough to run at scale", section "Two system changes"): a student's
 * output projection z = H W^T over the full vocabulary, compared by a KL
 * divergence with an offline cache of the teacher's top-K (id, logit) pairs
 * per token, without ever storing the tokens x vocabulary logit grid. The
 * backward computes each chunk's projection a second time instead of keeping
 * it (same section, the fused-chunked bullet; "Efficient knowledge
 * distillation for LLMs: offline top-K logits and a fused chunked KL loss",
 * section "Two systemic changes for scalable distillation", item 2).
 *
 * Definitions (the pages name a closed-form gradient but do not print it):
 *   p[t,k]   = softmax_k(topk_logit[t,k] / tau)        teacher, renormalised over K
 *   lse[t]   = log sum_v exp(z[t,v] / tau)             full vocabulary
 *   KL[t]    = sum_k p[t,k] (log p[t,k] - z[t,idx[t,k]]/tau + lse[t])
 *   loss     = sum_t m[t] KL[t] / N,  N = sum_t m[t]   (0 when N = 0)
 *   dL/dz    = m[t] (softmax(z[t]/tau) - P[t]) / (tau N), P = p scattered at idx
 *   dH = g dL/dz . W,  dW = g (dL/dz)^T . H            (g = upstream gradient)
 *
 * Conventions for every call:
 *   - All arrays are DEVICE pointers, row-major and contiguous, owned by the
 *     caller. The library never allocates device memory: scratch lives in a
 *     caller-provided workspace of kd_kl_workspace_size() bytes.
 *   - bf16 arrays are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *     asynchronous on it and never synchronise the device, except
 *     kd_kl_check_status() and kd_timing_end(), which say so.
 *   - Argument errors are returned synchronously and launch nothing.
 *     Errors found on the device (a topk index outside [0, V), a teacher row
 *     with no finite logit, a pipeline wait that ran out) are recorded in the
 *     workspace and read with kd_kl_check_status().
 *   - Calls sharing one workspace must be ordered on one stream.
 */
#ifndef KDKL_H
#define KDKL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDKL_MAX_K 512 /* largest K the teacher-prep sort handles */

typedef enum {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,  /* null pointer, tau <= 0 or not finite, chunk < 1,
                              or (device) a teacher row without a finite logit */
  KD_ERR_SHAPE = 2,        /* T < 0, d < 8, V < 1, K < 1, K > V, K > KDKL_MAX_K,
                              or a size >= 2^31 */
  KD_ERR_ALIGNMENT = 3,    /* d % 8 != 0, or H/W/dH/dW/workspace not 16-byte aligned */
  KD_ERR_INDEX_RANGE = 4,  /* (device) a topk_idx entry outside [0, V) */
  KD_ERR_WORKSPACE = 5,    /* workspace NULL or smaller than kd_kl_workspace_size() */
  KD_ERR_CUDA = 6,         /* a CUDA runtime or driver call failed */
  KD_ERR_TIMEOUT = 7,      /* (device) a bounded pipeline wait ran out; outputs undefined */
  KD_ERR_UNSUPPORTED = 8   /* the current device is not compute capability 10.3 */
} kd_status;

typedef struct {
  int64_t T;          /* tokens (rows of H) */
  int64_t d;          /* hidden size (columns of H and W); multiple of 8 */
  int64_t V;          /* vocabulary size (rows of W) */
  int32_t K;          /* cached teacher entries per token, 1..min(V, KDKL_MAX_K) */
  float temperature;  /* tau > 0; divides both student and teacher logits */
  int64_t chunk;      /* token-chunk size of the pages' method: bounds the
                         backward's gradient-of-logits buffer to chunk x V
                         bf16 elements, plus tile padding (the scheduler may
                         tile that budget as fewer tokens x more vocabulary,
                         in whole 256-wide vocabulary tiles; results are the
                         same) */
} kd_kl_problem;

/* Workspace bytes for kd_kl_forward (which = 0), kd_kl_backward (which = 1),
 * kd_kl_forward_ex (which = 2), kd_kl_backward_ex (which = 3) or
 * kd_kl_backward_reuse (which = 4).
 * Linear in T (no T x V term). Returns 0 if the problem is invalid. */
size_t kd_kl_workspace_size(const kd_kl_problem* prob, int which);

/* Forward: mean KL loss over unmasked tokens and the per-token logsumexp.
 *   H          [T, d] bf16        student hidden states
 *   W          [V, d] bf16        student output projection (LM head)
 *   topk_idx   [T, K] int32       teacher's cached ids, any order, in [0, V)
 *   topk_logit [T, K] fp32        teacher's cached logits (-inf allowed, not all)
 *   mask       [T] uint8 or NULL  nonzero = token counts (NULL: all count)
 *   loss       [1] fp32 out       sum_t m[t] KL[t] / N (0 when N = 0)
 *   lse        [T] fp32 out       log sum_v exp(z[t,v]/tau) of every counted token
 *   token_kl   [T] fp32 out or NULL   KL[t] of every counted token
 * The logits z are produced tile by tile inside the SMs and never written to
 * memory. With a mask, the counted tokens are compacted first (in order) and
 * every later step runs on them alone: a masked token costs no tensor-core
 * work, and its lse and token_kl read 0 (they are not computed). With a NULL
 * mask every token counts. */
kd_status kd_kl_forward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                        const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                        float* loss, float* lse, float* token_kl,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Backward: gradients of g * loss. Masked tokens are skipped as in the
 * forward (their dH rows are exact zeros).
 *   lse        [T] fp32           from kd_kl_forward on the same inputs
 *   grad_loss  g                  upstream dL_outer/dloss (host scalar)
 *   dH         [T, d] bf16 out    overwritten; fp32 accumulation inside, masked rows = 0
 *   dW         [V, d] fp32 out    overwritten, or added to when accumulate_dW != 0
 * Each logit tile is recomputed and turned into (softmax - P) in the GEMM
 * epilogue; the result is kept in a bf16 buffer of about chunk x V elements
 * (the block's vocabulary rounded up to whole 256-wide tiles) that feeds the
 * dH and dW tensor-core GEMMs. */
kd_status kd_kl_backward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                         const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                         const float* lse, float grad_loss,
                         uint16_t* dH, float* dW, int accumulate_dW,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Loss variant. The pages report ablations over the choice of loss without
 * printing one ("Making knowledge distillation cheap enough to run at scale",
 * closing section); this is the standard distillation mix:
 *   loss_t = alpha * c * KL_t(tau) + (1 - alpha) * CE_t,  c = tau^2 or 1,
 *   CE_t   = log sum_v exp(z[t,v]) - z[t, labels[t]]      (temperature 1),
 *   loss   = sum_t m[t] loss_t / N.
 * dL/dz[t,v] = m[t]/N * (alpha c (softmax(z/tau) - P)/tau + (1-alpha)(softmax(z) - onehot)).
 * Same kernels as the calls above, with the temperature-1 sum and the label
 * logit added to the GEMM epilogues. */
typedef struct {
  float alpha;            /* weight of the soft term, in [0, 1]; 1 = KL only */
  int32_t scale_tau_sq;   /* nonzero: the soft term and its gradient are scaled by tau^2 */
  const int32_t* labels;  /* [T] device, hard labels in [0, V); may be NULL when alpha == 1 */
} kd_kl_options;

/* Workspace: kd_kl_workspace_size(prob, 2) for the forward, (prob, 3) for the backward.
 *   lse        [T] fp32 out   logsumexp of z / tau (counted tokens; masked ones read 0)
 *   lse1       [T] fp32 out   logsumexp of z (temperature 1; equals lse when tau == 1)
 *   token_loss [T] fp32 out or NULL   alpha c KL_t + (1 - alpha) CE_t (counted tokens)
 * A counted token's label outside [0, V) is reported as KD_ERR_INDEX_RANGE by
 * kd_kl_check_status (masked tokens' labels and teacher ids are not read). */
kd_status kd_kl_forward_ex(const kd_kl_problem* prob, const kd_kl_options* opts,
                           const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                           const float* topk_logit, const uint8_t* mask, float* loss, float* lse,
                           float* lse1, float* token_loss, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Backward of grad_loss * loss. lse1 may be NULL when tau == 1 or alpha == 1. */
kd_status kd_kl_backward_ex(const kd_kl_problem* prob, const kd_kl_options* opts,
                            const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                            const float* topk_logit, const uint8_t* mask, const float* lse,
                            const float* lse1, float grad_loss, uint16_t* dH, float* dW,
                            int accumulate_dW, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Backward that reuses the teacher cache the forward already prepared. The
 * forward turns the cache into sorted (id, p) rows and counts the mask
 * (N) in its workspace; the pages compute the teacher side once and keep it
 * ("Making knowledge distillation cheap enough to run at scale", section "Two
 * system changes"), so the backward can read those rows instead of preparing
 * them again. Same results as kd_kl_backward / kd_kl_backward_ex.
 *   opts           NULL for the plain KL loss, else as kd_kl_backward_ex
 *   mask, lse, lse1  as kd_kl_backward(_ex); mask must be the forward's
 *   fwd_workspace  the workspace of the latest kd_kl_forward or
 *                  kd_kl_forward_ex call on the same problem (T, d, V, K and
 *                  temperature; chunk may differ), queued earlier on the same
 *                  stream and not reused since; read only
 *   workspace      kd_kl_workspace_size(prob, 4) bytes (no teacher region)
 * The library remembers, on the host, which problem each forward workspace
 * was last filled for; a fwd_workspace it does not know for this problem, or
 * fwd_workspace_bytes smaller than that call's, returns KD_ERR_INVALID_ARG
 * synchronously. The teacher cache was validated by the forward: its
 * device-detected errors are read from fwd_workspace, this call's (wait
 * timeouts) from workspace. */
kd_status kd_kl_backward_reuse(const kd_kl_problem* prob, const kd_kl_options* opts,
                               const uint16_t* H, const uint16_t* W, const uint8_t* mask,
                               const float* lse, const float* lse1, const void* fwd_workspace,
                               size_t fwd_workspace_bytes, float grad_loss, uint16_t* dH,
                               float* dW, int accumulate_dW, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Allocation-free forward. The paper has no counterpart to this call; it
 * exists for callers that cannot allocate device memory for a workspace: code
 * inside a host framework whose memory pool owns (and has typically reserved)
 * all free HBM, and loops with a latency budget that rules out cudaMalloc,
 * which can synchronise the device.
 * Same arguments, results and errors as kd_kl_forward, minus the workspace:
 * the scratch is a fixed array of KDKL_NOALLOC_SCRATCH_BYTES compiled into the
 * library, held on every GPU where the library's device code is loaded until
 * the process exits. Problems whose kd_kl_workspace_size(prob, 0) exceeds it
 * return KD_ERR_WORKSPACE before anything is queued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current), and so does the first
 *     call after a device reset; make that first call before any stream
 *     capture.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine (with
 *     per-kernel timing off, the default).
 *   - Every call on a device shares the one array and clears its header when
 *     it starts. Calls whose GPU work overlaps (other streams, other host
 *     threads) race on it: order them on one stream.
 *   - Device-detected errors (an id outside [0, V), a teacher row with no
 *     finite logit, a wait that ran out) go to the array's status word and are
 *     read with kd_kl_noalloc_check_status(); outputs are then undefined. */
#define KDKL_NOALLOC_SCRATCH_BYTES (64u << 20)
kd_status kd_kl_forward_noalloc(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                                const int32_t* topk_idx, const float* topk_logit,
                                const uint8_t* mask, float* loss, float* lse, float* token_kl,
                                void* stream);

/* BLOCKING: synchronises `stream`, then returns the first device-detected
 * error recorded by the latest kd_kl_forward_noalloc call on the current
 * device (KD_OK if none), like kd_kl_check_status does for a workspace. */
kd_status kd_kl_noalloc_check_status(void* stream);

/* ---------------------------------------------------------------------------
 * Second loss variant: reverse KL restricted to the cached ids. The pages
 * report ablations over the choice of loss without printing one ("Making
 * knowledge distillation cheap enough to run at scale", closing section);
 * this is the mode-seeking direction, taken over the same support as the
 * teacher cache (entries whose teacher logit is not finite are dropped from
 * both distributions):
 *   qt[t,k]  = softmax_k(z[t,idx[t,k]] / tau)      student, renormalised over the ids
 *   p[t,k]   = softmax_k(topk_logit[t,k] / tau)    teacher, as above
 *   RKL[t]   = sum_k qt[t,k] (log qt[t,k] - log p[t,k])
 *   loss     = sum_t m[t] RKL[t] / N              (0 when N = 0)
 *   grad_z[t,k] = dloss/dz[t,idx[t,k]] = m[t]/N * qt (log qt - log p - RKL[t]) / tau
 *               (0 for dropped entries)
 * Only the K cached logits of each token enter, so there is no vocabulary-wide
 * contraction: the kernels stream rows of W and H per (token, id) pair, on CUDA
 * cores, over the pairs sorted by id (forward, dW) or per token (dH). The problem struct
 * is kd_kl_problem; `chunk` is not used (any value >= 1); T * K < 2^31.
 * Both calls take a workspace of kd_rkl_workspace_size() bytes: linear in T,
 * plus 8 bytes per vocabulary row. */
size_t kd_rkl_workspace_size(const kd_kl_problem* prob);

/*   loss       [1] fp32 out           sum_t m[t] RKL[t] / N
 *   token_rkl  [T] fp32 out or NULL   RKL[t] before masking
 *   grad_z     [T, K] fp32 out or NULL   dloss/dz at the cached ids (upstream
 *                                     gradient 1); passing it to kd_rkl_backward
 *                                     saves the backward its logit recompute
 * Other arguments and errors as kd_kl_forward. */
kd_status kd_rkl_forward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                         const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                         float* loss, float* token_rkl, float* grad_z, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Gradients of grad_loss * loss.
 *   grad_z  [T, K] fp32 or NULL   from kd_rkl_forward on the same inputs; NULL:
 *                                 the backward recomputes it (the forward's z pass)
 *   dH      [T, d] bf16 out       overwritten (fp32 sums inside; masked rows = 0)
 *   dW      [V, d] fp32 out       overwritten, or added to when accumulate_dW != 0
 * The (id, token) pairs are sorted by id inside the call so that each dW row is
 * summed by one warp in token order: no atomics, and both outputs are bitwise
 * reproducible from run to run. An id outside [0, V) contributes nothing and is
 * reported as KD_ERR_INDEX_RANGE by kd_kl_check_status. */
kd_status kd_rkl_backward(const kd_kl_problem* prob, const uint16_t* H, const uint16_t* W,
                          const int32_t* topk_idx, const float* topk_logit, const uint8_t* mask,
                          const float* grad_z, float grad_loss, uint16_t* dH, float* dW,
                          int accumulate_dW, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ---------------------------------------------------------------------------
 * Offline teacher cache producer: for every row t of H, the K largest logits
 * z[t,v] = H[t] . W[v] over the full vocabulary, with their ids. This is the
 * cache the loss above consumes ("Making knowledge distillation cheap enough
 * to run at scale", section "Two system changes": compute the teacher's
 * output once and cache the 100 most likely tokens per position). The same
 * tensor-core GEMM produces each logit tile; its epilogue keeps per-row
 * candidate lists above a running threshold, so the logits are never stored.
 */
#define KDKL_TOPK_MAX_K 512

typedef struct {
  int64_t T;   /* rows of H (tokens) */
  int64_t d;   /* hidden size; multiple of 8 */
  int64_t V;   /* vocabulary (rows of W) */
  int32_t K;   /* entries kept per row, 1..min(V, KDKL_TOPK_MAX_K) */
  int32_t reserved;  /* set to 0 */
} kd_topk_problem;

/* Workspace bytes for kd_lmhead_topk; linear in T; 0 if the problem is invalid. */
size_t kd_lmhead_topk_workspace_size(const kd_topk_problem* prob);

/*   H          [T, d] bf16      hidden states (device)
 *   W          [V, d] bf16      output projection (device)
 *   topk_idx   [T, K] int32 out ids, per row by logit descending, ties to the smaller id
 *   topk_logit [T, K] fp32 out  the logits z (fp32 accumulation of the bf16 products)
 * Errors: KD_ERR_SHAPE (T < 0, d < 8, V < 1, K outside 1..min(V, KDKL_TOPK_MAX_K)),
 * KD_ERR_ALIGNMENT (d % 8 != 0 or misaligned pointers), KD_ERR_INVALID_ARG (null
 * pointers), KD_ERR_WORKSPACE, KD_ERR_CUDA, KD_ERR_UNSUPPORTED; device-detected
 * errors via kd_kl_check_status(workspace). */
kd_status kd_lmhead_topk(const kd_topk_problem* prob, const uint16_t* H, const uint16_t* W,
                         int32_t* topk_idx, float* topk_logit, void* workspace,
                         size_t workspace_bytes, void* stream);

/* BLOCKING: synchronises `stream`, then returns the first device-detected
 * error recorded in `workspace` by the latest call that used it (KD_OK if
 * none). Each forward/backward call clears the record when it starts. */
kd_status kd_kl_check_status(void* workspace, void* stream);

/* Human-readable name of a status code (static storage). */
const char* kd_status_string(kd_status status);

/* Number of kernels this library has launched in this process (all calls,
 * all devices). Lets a caller count launches inside a timed region. */
int64_t kd_launch_count(void);

/* Per-kernel timing. After kd_timing_begin(), every kernel the library
 * launches is bracketed by CUDA events recorded on its launch stream.
 * kd_timing_end() is BLOCKING: it synchronises those events, fills up to
 * `max_entries` rows (one per kernel name, in first-launch order), stores
 * the row count in *n_entries, and stops recording. */
typedef struct {
  char name[32];
  int64_t launches;
  double total_ms;
} kd_kernel_time;

kd_status kd_timing_begin(void);
kd_status kd_timing_end(kd_kernel_time* out, int max_entries, int* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* KDKL_H */
