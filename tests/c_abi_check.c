/* A plain C client of include/bsgemv.h: the header compiles as C11 and the library links.  Runs
 * only host-side entry points (no GPU needed): geometry queries, status strings and argument
 * errors.  Prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "bsgemv.h"

#define CHECK(cond)                                                    \
  do {                                                                 \
    if (!(cond)) {                                                     \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      return 1;                                                        \
    }                                                                  \
  } while (0)

int main(void) {
  bsgemv_geometry g;
  memset(&g, 0, sizeof g);
  CHECK(bsgemv_geometry_for(BSGEMV_INT8, 128, 1, 4096, 4096, 1, 152, &g) == BSGEMV_OK);
  CHECK(g.rows_per_tile == 64 && g.k_per_stage == 256 && g.tiles == 64 && g.ctas >= 1);
  CHECK(bsgemv_geometry_for(BSGEMV_INT4 | BSGEMV_ACT_BF16, 32, 0, 151936, 4096, 16, 152, &g) ==
        BSGEMV_OK);
  CHECK(bsgemv_geometry_for(BSGEMV_FP8_E4M3, 64, 0, 512, 2048, 1, 152, &g) == BSGEMV_ERR_UNSUPPORTED);
  CHECK(bsgemv_geometry_for(BSGEMV_NVFP4, 16, 0, 512, 2048, 33, 152, &g) == BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_dense_geometry_for(0, 1024, 2048, 8, 152, &g) == BSGEMV_OK && g.rows_per_tile == 64);
  CHECK(bsgemv_dense_geometry_for(1, 1, 2048, 8, 152, &g) == BSGEMV_OK && g.rows_per_tile == 8);
  CHECK(strcmp(bsgemv_status_string(BSGEMV_OK), "ok") == 0);
  CHECK(bsgemv_run(NULL, NULL, NULL, NULL, NULL, NULL, 1, NULL) == BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_destroy(NULL) == BSGEMV_OK && bsgemv_dense_destroy(NULL) == BSGEMV_OK);
  bsgemv_plan_t plan = NULL;
  CHECK(bsgemv_plan(&plan, BSGEMV_INT8, 48, 1, 64, 512, 1) == BSGEMV_ERR_UNSUPPORTED && !plan);
  CHECK(bsgemv_plan_set_test_fault(NULL, -1, 0) == BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_version() >= 100);
  printf("ok\n");
  return 0;
}
