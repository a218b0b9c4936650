/*
 * A plain C99 user of bsolve.h: the header compiles as C, every entry point links, and
 * the calls that return before any launch (empty batches, argument errors, unsupported
 * shapes, queries) give the documented statuses. No call below reaches the GPU, so the
 * program runs on a machine without one. Exit status: the number of failed checks.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "bsolve.h"

static int failures = 0;

#define CHECK(expr)                                              \
  do {                                                           \
    if (!(expr)) {                                               \
      fprintf(stderr, "%s:%d: failed: %s\n", __FILE__, __LINE__, #expr); \
      ++failures;                                                \
    }                                                            \
  } while (0)

/* Never dereferenced: every call that is given these returns before any copy or launch. */
static void* fake(uintptr_t offset) { return (void*)(uintptr_t)(0x10000u + offset); }

int main(void) {
  const uintptr_t M = 0x100000u;
  void* A = fake(0);
  void* B = fake(M);
  int32_t* ipiv = (int32_t*)fake(2 * M);
  int32_t* info = (int32_t*)fake(3 * M);
  bs_options o;

  /* the options struct as the binding marshals it: 32 bytes, fields at fixed offsets */
  CHECK(sizeof(bs_options) == 32);
  CHECK(offsetof(bs_options, pivot_threshold) == 0);
  CHECK(offsetof(bs_options, status_contract) == 8);
  CHECK(offsetof(bs_options, transposed_factor) == 12);
  CHECK(offsetof(bs_options, interleave) == 16);
  CHECK(offsetof(bs_options, scaling) == 24);

  /* queries */
  CHECK(bs_version() > 0);
  CHECK(strlen(bs_status_string(BS_OK)) > 0);
  CHECK(strcmp(bs_status_string(BS_OK), bs_status_string(BS_ERR_CUDA)) != 0);
  CHECK(bs_getrf_getrs_supported(BS_FP32, BS_ROW_MAJOR, 16, 4) == 1);
  CHECK(bs_getrf_getrs_supported(BS_FP64, BS_COL_MAJOR, 129, 1) == 0);
  CHECK(bs_potrf_potrs_supported(BS_FP64, BS_COL_MAJOR, BS_LOWER, 32, 1) == 1);
  CHECK(bs_bdsv_supported(BS_FP64, 32, 8) == 1);
  CHECK(bs_bdsv_supported(BS_FP64, 32, 9) == 0);
  CHECK(bs_getrf_getrs_host_workspace(BS_FP32, 16, 4, 8) > 0);
  CHECK(bs_getrf_getrs_host_workspace(BS_FP32, 16, 4, 0) == 0);
  CHECK(bs_potrf_potrs_host_workspace(BS_FP64, 32, 1, 8) > 0);
  CHECK(bs_bdsv_host_workspace(BS_FP64, 32, 8, 8) > 0);
  CHECK(bs_bdsv_host_workspace(BS_FP64, 32, 8, -1) == 0);

  /* empty batches launch nothing, whatever the pointers */
  CHECK(bs_getrf_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, 0, NULL, NULL, NULL, NULL,
                               NULL) == BS_OK);
  CHECK(bs_potrf_potrs_batched(BS_FP64, BS_COL_MAJOR, BS_LOWER, 32, 1, 0, NULL, NULL, NULL,
                               NULL) == BS_OK);
  CHECK(bs_bdsv_batched(BS_FP64, 32, 8, 0, NULL, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_getrf_batched(BS_FP32, BS_ROW_MAJOR, 16, 0, NULL, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, 0, NULL, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_potrf_batched(BS_FP64, BS_COL_MAJOR, BS_LOWER, 32, 0, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_potrs_batched(BS_FP64, BS_COL_MAJOR, BS_LOWER, 32, 1, 0, NULL, NULL, NULL) ==
        BS_OK);
  CHECK(bs_bdsv_factor_batched(BS_FP64, 32, 8, 0, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_bdsv_solve_batched(BS_FP64, 32, 8, 0, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_bdmv_batched(BS_FP64, 32, 8, 0, NULL, NULL, NULL, NULL) == BS_OK);
  CHECK(bs_bdmv2_batched(BS_FP64, 32, 8, 0, NULL, NULL, NULL, NULL, NULL) == BS_OK);

  /* argument errors and unsupported shapes */
  CHECK(bs_getrf_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, -1, A, B, ipiv, info, NULL) ==
        BS_ERR_INVALID_ARG);
  CHECK(bs_getrf_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, NULL, B, ipiv, info, NULL) ==
        BS_ERR_INVALID_ARG);
  CHECK(bs_getrf_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, fake(4), B, ipiv, info,
                               NULL) == BS_ERR_INVALID_ARG);
  CHECK(bs_getrf_getrs_batched(BS_FP32, BS_ROW_MAJOR, 129, 4, 5, A, B, ipiv, info, NULL) ==
        BS_ERR_UNSUPPORTED);
  CHECK(bs_getrf_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, fake(4096), ipiv, info,
                               NULL) == BS_ERR_INVALID_ARG); /* B inside A */
  CHECK(bs_potrf_potrs_batched(BS_FP64, BS_COL_MAJOR, (bs_fill)2, 32, 1, 5, A, B, info,
                               NULL) == BS_ERR_UNSUPPORTED);
  CHECK(bs_bdsv_batched(BS_FP64, 32, 9, 4, A, B, info, NULL) == BS_ERR_UNSUPPORTED);
  CHECK(bs_getrs_batched(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, ipiv, fake(16), NULL) ==
        BS_ERR_INVALID_ARG); /* B over the factor */
  CHECK(bs_bdmv_batched(BS_FP64, 32, 8, 4, A, B, B, NULL) == BS_ERR_INVALID_ARG);
  CHECK(bs_bdmv2_batched(BS_FP64, 32, 8, 4, A, B, ipiv, ipiv, NULL) == BS_ERR_INVALID_ARG);

  /* the contract options */
  memset(&o, 0, sizeof o);
  o.pivot_threshold = 0.0; /* outside (0, 1] */
  CHECK(bs_getrf_getrs_batched_ex(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, B, ipiv, info, &o,
                                  NULL) == BS_ERR_INVALID_ARG);
  o.pivot_threshold = 1.0;
  o.interleave = -2;
  CHECK(bs_getrf_getrs_batched_ex(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, B, ipiv, info, &o,
                                  NULL) == BS_ERR_INVALID_ARG);
  o.interleave = 4;
  o.transposed_factor = 1;
  o.status_contract = BS_CONTRACT_RUDA; /* the row-major reading: not with this contract */
  CHECK(bs_getrf_getrs_batched_ex(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, B, ipiv, info, &o,
                                  NULL) == BS_ERR_UNSUPPORTED);
  /* the split calls with options: the contract stays with the fused calls */
  CHECK(bs_getrf_batched_ex(BS_FP32, BS_ROW_MAJOR, 16, 5, A, ipiv, info, &o, NULL) ==
        BS_ERR_UNSUPPORTED);
  CHECK(bs_getrs_batched_ex(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, ipiv, B, &o, NULL) ==
        BS_ERR_UNSUPPORTED);
  o.status_contract = BS_CONTRACT_DEFAULT;
  CHECK(bs_potrf_batched_ex(BS_FP64, BS_COL_MAJOR, BS_LOWER, 32, 5, A, info, &o, NULL) ==
        BS_ERR_UNSUPPORTED); /* an LU option */
  o.transposed_factor = 0;
  CHECK(bs_potrs_batched_ex(BS_FP64, BS_COL_MAJOR, BS_LOWER, 200, 1, 5, A, B, &o, NULL) ==
        BS_ERR_UNSUPPORTED); /* interleaved Cholesky: n <= 128 */
  o.status_contract = 7;
  CHECK(bs_potrf_potrs_batched_ex(BS_FP64, BS_COL_MAJOR, BS_LOWER, 32, 1, 5, A, B, info, &o,
                                  NULL) == BS_ERR_INVALID_ARG);

  /* host-resident calls */
  CHECK(bs_getrf_getrs_batched_host(BS_FP32, BS_ROW_MAJOR, 16, 4, 5, A, B, ipiv, info,
                                    fake(4 * M), bs_getrf_getrs_host_workspace(BS_FP32, 16, 4, 8),
                                    0, NULL, NULL) == BS_ERR_INVALID_ARG); /* chunk 0 */
  CHECK(bs_getrf_getrs_batched_host_static(BS_FP32, BS_ROW_MAJOR, 129, 4, 5, A, B, ipiv, info,
                                           16, NULL, NULL) == BS_ERR_UNSUPPORTED);
  CHECK(bs_bdsv_batched_host(BS_FP64, 32, 8, 4, A, B, info, fake(4 * M), 16, 8, NULL, NULL) ==
        BS_ERR_INVALID_ARG); /* workspace too small */

  if (failures == 0) printf("bsolve C ABI: all checks passed\n");
  return failures;
}
