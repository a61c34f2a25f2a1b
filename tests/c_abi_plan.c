/* A plain C99 caller of the library's C ABI (include/zero.h), built and run by
 * tests/test_c_abi.py. It uses only the host-side entry points (plan, query, bucket ranges,
 * argument errors), so it runs without a GPU. One line per plan:
 *   plan psi n stage bucket_bytes | psi P S C n_buckets state[param grad master m v total]
 *        comm[rs ag_fwd ag_bwd total] ring fused | first and last bucket of the last rank
 * then one line per expected argument error: "error <code> <message>". Exit status 0 on
 * success, 1 if any call did not behave as the header states. */
#include <inttypes.h>
#include <stdio.h>
#include <string.h>

#include "zero.h"

static int failures = 0;

static void show_plan(uint64_t psi, int n, int stage, uint64_t bucket_bytes) {
  zero_plan_t* plan = NULL;
  zero_layout L;
  uint64_t b0 = 0, e0 = 0, b1 = 0, e1 = 0;
  if (zero_plan(psi, n, stage, bucket_bytes, &plan) != ZERO_OK || plan == NULL) {
    printf("plan-failed %s\n", zero_last_error());
    ++failures;
    return;
  }
  memset(&L, 0, sizeof(L));
  if (zero_plan_query(plan, &L) != ZERO_OK) ++failures;
  if (zero_bucket_range(plan, n - 1, 0, &b0, &e0) != ZERO_OK) ++failures;
  if (zero_bucket_range(plan, n - 1, L.n_buckets - 1, &b1, &e1) != ZERO_OK) ++failures;
  printf("plan %" PRIu64 " %d %d %" PRIu64 " | %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64, psi, n,
         stage, bucket_bytes, L.psi, L.psi_padded, L.shard_elems, L.bucket_elems, L.n_buckets);
  printf(" %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64, L.state_param_bytes,
         L.state_grad_bytes, L.state_master_bytes, L.state_m_bytes, L.state_v_bytes, L.state_total_bytes);
  printf(" %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64, L.comm_reduce_scatter,
         L.comm_all_gather_fwd, L.comm_all_gather_bwd, L.comm_total, L.ring_sent_elems, L.fused_step_bytes);
  printf(" | %" PRIu64 " %" PRIu64 " %" PRIu64 " %" PRIu64 "\n", b0, e0, b1, e1);
  if (zero_plan_destroy(plan) != ZERO_OK) ++failures;
}

static void expect_error(int rc, int want) {
  printf("error %d %s\n", rc, zero_last_error());
  if (rc != want || zero_last_error()[0] == '\0') ++failures;
}

int main(void) {
  zero_plan_t* plan = NULL;
  uint64_t b = 0, e = 0;
  printf("version %d\n", zero_version());
  show_plan(1000003u, 8, 2, 25u << 20);
  show_plan(13u, 3, 0, 6u);
  show_plan(124356864u, 8, 3, 25u << 20);
  show_plan(7241732096u, 8, 3, 50u << 20);
  show_plan(4099u, 5, ZERO_STAGE_MEGATRON, 1u << 10);
  /* argument errors come back as codes, with nothing launched */
  expect_error(zero_plan(1000u, 0, 2, 1u << 20, &plan), ZERO_ERR_INVALID_ARG);
  expect_error(zero_plan(1000u, ZERO_MAX_RANKS + 1, 2, 1u << 20, &plan), ZERO_ERR_INVALID_ARG);
  expect_error(zero_plan(1000u, 8, 2, 15u, &plan), ZERO_ERR_INVALID_ARG);
  if (zero_plan(1000u, 8, 2, 1u << 20, &plan) != ZERO_OK) ++failures;
  expect_error(zero_bucket_range(plan, 8, 0, &b, &e), ZERO_ERR_INVALID_ARG);
  expect_error(zero_plan_query(plan, NULL), ZERO_ERR_INVALID_ARG);
  zero_plan_destroy(plan);
  return failures ? 1 : 0;
}
