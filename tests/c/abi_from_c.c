/* The qmoe C ABI used from plain C99 (no C++, no torch): size and schedule queries and
 * argument checks, which need no GPU.  Prints one line per check; exit code = failures. */
#include <math.h>
#include <stdio.h>

#include "qmoe.h"

static int fails = 0;
#define CHECK(cond)                                  \
  do {                                               \
    if (!(cond)) {                                   \
      printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #cond); \
      ++fails;                                       \
    }                                                \
  } while (0)

int main(void) {
  /* schedules and tiles */
  CHECK(qmoe_sched_tile_n(QMOE_SCHED_AUTO, 16, 8, 256) == 16);
  CHECK(qmoe_sched_tile_n(QMOE_SCHED_AUTO, 8192, 8, 256) == 320);
  CHECK(qmoe_max_tiles(8192, 8, 256, 320) == (65536 + 319) / 320 + 256);
  CHECK(qmoe_forward_kernel_count(16, 8, 256, QMOE_SCHED_AUTO) == 5);
  /* sizes */
  CHECK(qmoe_forward_workspace_size(16, 7168, 2048, 256, 8, QMOE_SCHED_AUTO) > 0);
  CHECK(qmoe_forward_workspace_size(4, 100, 128, 8, 2, QMOE_SCHED_AUTO) == 0);
  CHECK(qmoe_repacked_fp4_size(256, 4096, 7168) == (size_t)256 * 4096 * 3584);
  CHECK(qmoe_route_workspace_size(4, 2, 8, 16) >= 4);
  /* argument checks before any device work */
  CHECK(moe_nvfp4_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, 100,
                          128, 8, 2, QMOE_SCHED_AUTO, NULL, 0, NULL) == QMOE_ERR_SHAPE);
  CHECK(moe_nvfp4_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, 128,
                          128, 8, 2, QMOE_SCHED_AUTO, NULL, 0, NULL) == QMOE_ERR_ARG);
  CHECK(moe_nvfp4_forward_limit(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0,
                                128, 128, 8, 2, QMOE_SCHED_AUTO, -1.0f, NULL, 0,
                                NULL) == QMOE_ERR_ARG);
  CHECK(moe_nvfp4_forward_limit(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0,
                                128, 128, 8, 2, QMOE_SCHED_AUTO, INFINITY, NULL, 0,
                                NULL) == QMOE_OK);
  CHECK(moe_nvfp4_repack_layout(NULL, NULL, 1, 128, 128, QMOE_W13, 7, NULL, NULL, NULL) ==
        QMOE_ERR_ARG);
  printf("%s: %d failure(s)\n", fails ? "FAILED" : "ok", fails);
  return fails;
}
