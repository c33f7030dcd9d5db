/* Plain C consumer of the library's C ABI (include/kdkl.h), linked against
 * libkdkl.so with no Python in between. It needs no GPU: it exercises the
 * calls that are answered on the host (workspace sizing, argument checks,
 * status strings) and prints "ok" when every check passes, else the first
 * failing check, with exit status 1. Built and run by tests/test_c_abi.py. */
#include <math.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include "kdkl.h"

static int failures = 0;

#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

int main(void) {
  /* layout the header promises (int64 fields at 8-byte offsets) */
  CHECK(sizeof(kd_kl_problem) == 40);
  CHECK(offsetof(kd_kl_problem, K) == 24);
  CHECK(offsetof(kd_kl_problem, chunk) == 32);
  CHECK(sizeof(kd_topk_problem) == 32);

  kd_kl_problem p = {32768, 2880, 201088, 100, 1.0f, 2048};
  const size_t fwd = kd_kl_workspace_size(&p, 0);
  const size_t bwd = kd_kl_workspace_size(&p, 1);
  const size_t rkl = kd_rkl_workspace_size(&p);
  CHECK(fwd > 0 && bwd > 0 && rkl > 0);
  /* no T x V term: far below a bf16 logit grid, a few KB per token at most */
  kd_kl_problem half = p;
  half.T = p.T / 2;
  CHECK(kd_kl_workspace_size(&half, 0) < fwd && kd_kl_workspace_size(&half, 1) < bwd);
  /* (the forward also holds a bf16 copy of the counted tokens' rows of H) */
  CHECK(fwd < (size_t)p.T * (4096 + 2 * (size_t)p.d) && rkl < (size_t)p.T * 16384);
  CHECK(bwd < (size_t)2 * p.T * p.V / 8);

  /* invalid problems size to 0 and are rejected synchronously */
  kd_kl_problem bad = p;
  bad.d = 12; /* not a multiple of 8 */
  CHECK(kd_kl_workspace_size(&bad, 0) == 0);
  CHECK(kd_kl_forward(&bad, (const uint16_t*)16, (const uint16_t*)16, (const int32_t*)16,
                      (const float*)16, NULL, (float*)64, (float*)128, NULL, (void*)256,
                      (size_t)1 << 30, NULL) == KD_ERR_ALIGNMENT);
  bad = p;
  bad.K = 0;
  CHECK(kd_kl_backward(&bad, (const uint16_t*)16, (const uint16_t*)16, (const int32_t*)16,
                       (const float*)16, NULL, (const float*)64, 1.0f, (uint16_t*)4096,
                       (float*)8192, 0, (void*)256, (size_t)1 << 30, NULL) == KD_ERR_SHAPE);
  bad = p;
  bad.temperature = 0.0f;
  CHECK(kd_rkl_forward(&bad, (const uint16_t*)16, (const uint16_t*)16, (const int32_t*)16,
                       (const float*)16, NULL, (float*)64, NULL, NULL, (void*)256,
                       (size_t)1 << 30, NULL) == KD_ERR_INVALID_ARG);
  /* a missing workspace is reported before anything touches a device */
  CHECK(kd_kl_forward(&p, (const uint16_t*)16, (const uint16_t*)16, (const int32_t*)16,
                      (const float*)16, NULL, (float*)64, (float*)128, NULL, NULL, 0,
                      NULL) == KD_ERR_WORKSPACE);

  /* mixed loss: options are checked before anything else happens */
  CHECK(kd_kl_forward_ex(&p, NULL, (const uint16_t*)16, (const uint16_t*)16, (const int32_t*)16,
                         (const float*)16, NULL, (float*)64, (float*)128, (float*)192, NULL,
                         (void*)256, (size_t)1 << 30, NULL) == KD_ERR_INVALID_ARG);
  kd_kl_options opt = {1.5f, 0, NULL}; /* alpha outside [0, 1] */
  CHECK(kd_kl_backward_ex(&p, &opt, (const uint16_t*)16, (const uint16_t*)16,
                          (const int32_t*)16, (const float*)16, NULL, (const float*)64,
                          (const float*)192, 1.0f, (uint16_t*)4096, (float*)8192, 0, (void*)256,
                          (size_t)1 << 30, NULL) == KD_ERR_INVALID_ARG);
  CHECK(kd_kl_workspace_size(&p, 2) > 0 && kd_kl_workspace_size(&p, 3) > 0);

  kd_topk_problem tp = {4096, 2880, 201088, 100, 0};
  CHECK(kd_lmhead_topk_workspace_size(&tp) > 0);
  CHECK(kd_lmhead_topk(&tp, (const uint16_t*)16, (const uint16_t*)16, (int32_t*)64, (float*)128,
                       NULL, 0, NULL) == KD_ERR_WORKSPACE);
  tp.K = KDKL_TOPK_MAX_K + 1;
  CHECK(kd_lmhead_topk_workspace_size(&tp) == 0);
  CHECK(kd_lmhead_topk(&tp, (const uint16_t*)16, (const uint16_t*)16, (int32_t*)64, (float*)128,
                       (void*)256, (size_t)1 << 30, NULL) == KD_ERR_SHAPE);

  /* the backward that reuses a forward's teacher rows: smaller workspace, and
   * a forward workspace the library has not seen filled is refused on the host */
  CHECK(kd_kl_workspace_size(&p, 4) > 0 && kd_kl_workspace_size(&p, 4) < bwd);
  CHECK(kd_kl_backward_reuse(&p, NULL, (const uint16_t*)16, (const uint16_t*)16, NULL,
                             (const float*)64, NULL, (const void*)4096, (size_t)1 << 30, 1.0f,
                             (uint16_t*)4096, (float*)8192, 0, (void*)256, (size_t)1 << 30,
                             NULL) == KD_ERR_INVALID_ARG);
  CHECK(kd_kl_backward_reuse(&p, NULL, (const uint16_t*)16, (const uint16_t*)16, NULL,
                             (const float*)64, NULL, NULL, 0, 1.0f, (uint16_t*)4096, (float*)8192,
                             0, (void*)256, (size_t)1 << 30, NULL) == KD_ERR_INVALID_ARG);

  CHECK(strcmp(kd_status_string(KD_OK), "KD_OK") == 0);
  CHECK(strcmp(kd_status_string(KD_ERR_TIMEOUT), "KD_ERR_TIMEOUT") == 0);
  CHECK(kd_launch_count() >= 0);

  if (failures) return 1;
  printf("ok\n");
  return 0;
}
