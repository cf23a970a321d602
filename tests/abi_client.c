/*
 * A plain C99 client of include/icp.h, built and run by test_abi_c.py.
 *
 * It compiles the header as C (not C++), links libicp.so like any C program
 * would, and calls only host paths that need no GPU: the sizing helpers,
 * calls with nothing to do, and argument checks that must reject before
 * anything reaches CUDA.  Exit status 0 when every check holds.
 */
#include <stdio.h>
#include <string.h>

#include "icp.h"

static int failures = 0;

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "abi_client: %s:%d: %s\n", __FILE__,       \
              __LINE__, #cond);                                  \
      ++failures;                                                \
    }                                                            \
  } while (0)

int main(void) {
  int32_t errors = 0;
  float out_s[16];
  int32_t out_i[16];

  /* status strings */
  CHECK(strcmp(icp_status_string(ICP_OK), "ok") == 0);
  CHECK(icp_status_string(ICP_ERR_INVALID_ARG) != NULL);
  CHECK(icp_status_string(12345) != NULL);
  CHECK(strstr(icp_status_string(ICP_ERR_TIMEOUT), "timed out") != NULL);
  CHECK(ICP_ERR_TIMEOUT != ICP_ERR_CUDA && ICP_ERR_TIMEOUT != ICP_ERR_UNSUPPORTED);

  /* plane width: B128 blocks (or local pages), padded to a multiple of 4 */
  CHECK(icp_score_columns(1000, 128, 1) == 8);
  CHECK(icp_score_columns(2500, 128, 1) == 20);
  CHECK(icp_score_columns(1000, 256, 1) == 8);   /* B128 blocks at P256, unsharded */
  CHECK(icp_score_columns(1000, 256, 2) == 4);   /* local pages at P256, sharded */
  CHECK(icp_score_columns(0, 128, 1) == 4);
  CHECK(icp_score_columns(-1, 128, 1) == -1);
  CHECK(icp_score_columns(1000, 64, 1) == -1);
  CHECK(icp_score_columns(1000, 128, 3) == -1);
  CHECK(icp_score_columns(8192 * 128, 128, 1) == 8192);
  CHECK(icp_score_columns(8192 * 128 + 1, 128, 1) == -1);

  /* scorer: an empty batch is a no-op; bad limits are rejected */
  CHECK(icp_score(NULL, NULL, 0, NULL, 0, NULL, NULL, 0, 4, 0, 1, 128, 1, 1, 0, NULL, NULL) ==
        ICP_OK);
  CHECK(icp_score(NULL, NULL, 0, NULL, 0, NULL, NULL, 0, 6, 0, 1, 128, 1, 1, 0, NULL, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* cols not a multiple of 4 */
  CHECK(icp_score(NULL, NULL, 0, NULL, 0, NULL, NULL, 0, 4, 0, 3, 128, 1, 1, 0, NULL, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* world size 3 */
  CHECK(icp_score(NULL, NULL, 0, NULL, 0, NULL, NULL, 0, 4, 0, 1, 128, 2, 1, 0, NULL, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* decode_query_len > max */
  CHECK(icp_score(NULL, NULL, 0, NULL, 0, NULL, NULL, 0, 4, 0, 1, 128, 1, 9, 0, NULL, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* 4 * max_decode_query_len > 32 */
  CHECK(icp_score(NULL, NULL, 1, NULL, 1, NULL, NULL, 1, 4, 0, 1, 128, 1, 1, 0, NULL, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* null buffers */

  /* select / publish / merge limits */
  CHECK(icp_top16_select(NULL, 0, 16, NULL, 1, 2, 1, 0, NULL, NULL, NULL) == ICP_OK);
  CHECK(icp_top16_select(NULL, 1, 12288, NULL, 1, 2, 1, 0, out_s, out_i, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* K >= 12288 */
  CHECK(icp_top16_select(NULL, 1, 16, NULL, 9, 8, 1, 0, out_s, out_i, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* init + local > 16 */
  CHECK(icp_publish_rows(NULL, 4, 16, NULL, NULL, &errors, 3, 0, 1, 4, 4, 1, 2, 100, 1, 0, 0,
                         NULL) == ICP_ERR_INVALID_ARG);   /* slot 3 */
  CHECK(icp_publish_rows(NULL, 5, 16, NULL, NULL, &errors, 0, 0, 1, 4, 4, 1, 2, 100, 1, 0, 0,
                         NULL) == ICP_ERR_INVALID_ARG);   /* T > capacity */
  CHECK(icp_merge(NULL, NULL, 1, 0, 3, 1, 4, 1, 2, 100, &errors, out_s, out_i, 0, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* world size 3 */
  CHECK(icp_merge(NULL, NULL, 1, 0, 2, 1, 4, 1, 2, 100, &errors, out_s, out_i, 0, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* heads_per_rank * world_size != 4 */

  /* fused path workspace and the prefill plan size */
  CHECK(icp_score_select_workspace_bytes(-1, 1) == 0);
  CHECK(icp_score_select_workspace_bytes(1, 9) == 0);
  CHECK(icp_score_select_workspace_bytes(4, 2) > 0);
  CHECK(icp_prefill_plan_words(1, 64) == 8 + 8 * 2);   /* one 64-token record + one spare */
  CHECK(icp_prefill_plan_words(2, 65) == 8 + 8 * 4);
  CHECK(icp_prefill_plan_words(-1, 0) == -1);
  CHECK(icp_prefill_merge(NULL, NULL, 0, 1, 4, 1, 2, NULL, NULL, NULL) == ICP_OK);
  CHECK(icp_prefill_merge(NULL, NULL, 1, 4, 4, 1, 2, out_s, out_i, NULL) ==
        ICP_ERR_INVALID_ARG);                    /* 4 ranks x 4 heads */

  if (failures == 0) printf("abi_client: ok\n");
  return failures == 0 ? 0 : 1;
}
