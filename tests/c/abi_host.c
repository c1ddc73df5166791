/* A plain C99 caller of the library's host-side entry points (no GPU is
 * needed for these): workspace sizes, status strings, the version, and
 * argument validation, which rejects bad calls before anything is enqueued.
 * Prints one "key value" line per check for the test that runs it. */
#include <stdio.h>

#include "mlp.h"

int main(void) {
  mlp_problem_t p = {2048, 4096, 11008, MLP_ACT_SWIGLU, 1.0f, 1.0f};
  printf("ws_fwd %zu\n", mlp_workspace_size(&p, MLP_MODE_FWD));
  printf("ws_bwd %zu\n", mlp_workspace_size(&p, MLP_MODE_BWD));
  printf("ws_null %zu\n", mlp_workspace_size(NULL, MLP_MODE_FWD));
  printf("status_ok %s\n", mlp_status_string(MLP_OK));
  printf("version %s\n", mlp_version());
  /* no problem, then a null required pointer: rejected before any launch */
  printf("fwd_null_problem %d\n",
         mlp_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL));
  printf("fwd_null_x %d\n", mlp_fwd(&p, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL));
  mlp_problem_t bad = p;
  bad.H = 4100; /* not a multiple of 8 */
  printf("fwd_bad_h %d\n", mlp_fwd(&bad, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL));
  return 0;
}
