/* A plain C caller of libsp's host-only entry points, compiled and run by
 * tests/test_abi_host.py (no GPU needed).
 *
 * It plans two requests: request 0 is a 20-token shared state with two
 * question branches of 3 and 5 own tokens; request 1 is one 7-token branch.
 * Staged submission (LLM2Jev "shared prefix" page, the three printed rounds)
 * sends the first branch of each request, then the second branch of request
 * 0 once the shared state is cached: rounds {0, 2} and {1}.  The state is
 * counted in both of its branches' logical tokens and computed once.
 *
 * Then it runs the batcher over three copies of request 1 with a budget of
 * two of them, and checks the argument and limit errors.  Exit status 0 when
 * every check holds; otherwise the first failed check is printed. */
#include <stdio.h>
#include <stdlib.h>

#include "sp.h"

#define CHECK(c)                                                        \
  do {                                                                  \
    if (!(c)) {                                                         \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c);   \
      return 1;                                                         \
    }                                                                   \
  } while (0)

int main(void) {
  const sp_shape shape = {8, 2, 64, 16, 64, 100};
  int32_t tokens[23 + 25 + 7];
  int64_t off[4] = {0, 23, 48, 55};
  const int32_t req[3] = {0, 0, 1};
  for (int i = 0; i < 20; ++i) tokens[i] = tokens[23 + i] = 10 + i;  /* the shared state */
  for (int i = 0; i < 3; ++i) tokens[20 + i] = 50 + i;
  for (int i = 0; i < 5; ++i) tokens[43 + i] = 60 + i;
  for (int i = 0; i < 7; ++i) tokens[48 + i] = 70 + i;

  sp_plan* plan = NULL;
  CHECK(sp_plan_build(&shape, 3, req, off, tokens, 1000, 152, &plan) == SP_OK && plan);
  sp_plan_stats st;
  CHECK(sp_plan_get_stats(plan, &st) == SP_OK);
  CHECK(st.n_requests == 2 && st.n_branches == 3);
  CHECK(st.n_segments == 4 && st.n_shared_segments == 1);
  CHECK(st.logical_tokens == 55 && st.computed_tokens == 35 && st.reused_tokens == 20);
  CHECK(st.node_tokens == 35);
  CHECK(st.pages_used == 5); /* 2 pages for the state, one for each own segment */
  int32_t n_rounds = 0;
  const int32_t* r_off = NULL;
  const int32_t* r_br = NULL;
  CHECK(sp_plan_rounds(plan, &n_rounds, &r_off, &r_br) == SP_OK);
  CHECK(n_rounds == 2);
  CHECK(r_off[0] == 0 && r_off[1] == 2 && r_off[2] == 3);
  CHECK(r_br[0] == 0 && r_br[1] == 2 && r_br[2] == 1);
  sp_plan_free(plan);

  /* errors: a pool too small, an empty branch, a branch over 32768 tokens */
  plan = NULL;
  CHECK(sp_plan_build(&shape, 3, req, off, tokens, 4, 152, &plan) == SP_ERR_POOL_FULL);
  CHECK(plan == NULL);
  const int64_t off_empty[4] = {0, 23, 23, 30};
  CHECK(sp_plan_build(&shape, 3, req, off_empty, tokens, 1000, 152, &plan) == SP_ERR_ARG);
  int32_t* long_branch = (int32_t*)calloc(32769, sizeof(int32_t));
  CHECK(long_branch != NULL);
  const int64_t off_long[2] = {0, 32769};
  const int32_t req_long[1] = {0};
  CHECK(sp_plan_build(&shape, 1, req_long, off_long, long_branch, 1 << 20, 152, &plan) ==
        SP_ERR_LIMIT);
  free(long_branch);
  CHECK(sp_status_str(SP_ERR_LIMIT) != NULL);

  /* label CSRs: counts 2..64 and ids below the vocabulary */
  const int32_t lab_off[3] = {0, 2, 4};
  const int32_t lab_ok[4] = {1, 2, 3, 99};
  const int32_t lab_bad[4] = {1, 2, 3, 100};
  CHECK(sp_check_labels(lab_off, lab_ok, 2, 100) == SP_OK);
  CHECK(sp_check_labels(lab_off, lab_bad, 2, 100) == SP_ERR_ARG);
  CHECK(sp_label_workspace_bytes(2, 100, 152) > 0);

  /* the batcher: three 7-token requests, at most 14 node tokens per batch */
  sp_batcher* b = NULL;
  CHECK(sp_batcher_create(&shape, 14, 64, &b) == SP_OK && b);
  const int64_t off1[2] = {0, 7};
  for (int i = 0; i < 3; ++i) {
    int64_t id = -1, nt = -1;
    CHECK(sp_batcher_submit(b, 1, off1, tokens + 48, &id, &nt) == SP_OK);
    CHECK(id == i && nt == 7);
  }
  int32_t pending = 0;
  int64_t pending_tokens = 0;
  CHECK(sp_batcher_pending(b, &pending, &pending_tokens) == SP_OK);
  CHECK(pending == 3 && pending_tokens == 21);
  const int32_t want[2] = {2, 1};
  for (int k = 0; k < 2; ++k) {
    int32_t n = 0;
    const int64_t* ids = NULL;
    const int32_t* br_off = NULL;
    const int64_t* row_off = NULL;
    plan = NULL;
    CHECK(sp_batcher_next(b, 1000, 152, &plan, &n, &ids, &br_off, &row_off) == SP_OK);
    CHECK(n == want[k] && plan != NULL);
    CHECK(ids[0] == 2 * k);
    CHECK(row_off[0] == 0 && (n < 2 || row_off[1] == 7));
    sp_plan_free(plan);
  }
  CHECK(sp_batcher_pending(b, &pending, &pending_tokens) == SP_OK && pending == 0);
  sp_batcher_free(b);

  printf("c abi host checks passed\n");
  return 0;
}
