/* Plain C99 user of include/flce.h: checks that the header compiles as C and
 * that the host-only entry points link and answer from a C program (no GPU
 * call is made).  Prints "ok" and exits 0 on success. */
#include <stdio.h>
#include <string.h>

#include "flce.h"

int main(void) {
  size_t ws = flce_workspace_size(8192, 3584, 152064);
  if (ws == 0 || flce_workspace_size(8, 12, 100) != 0) {
    printf("workspace size check failed\n");
    return 1;
  }
  if (strcmp(flce_status_string(FLCE_ERR_LABEL_OUT_OF_RANGE), "FLCE_ERR_LABEL_OUT_OF_RANGE") != 0) {
    printf("status string check failed\n");
    return 1;
  }
  /* host-detected argument errors return before any CUDA call */
  if (flce_forward(NULL, NULL, NULL, 64, 64, 100, 0, -100, 0, FLCE_REDUCTION_MEAN, NULL, NULL,
                   NULL, NULL, 0, NULL) != FLCE_ERR_INVALID_ARG) {
    printf("argument check failed\n");
    return 1;
  }
  if (flce_downcast_bf16(NULL, NULL, 12, NULL) != FLCE_ERR_INVALID_ARG) {
    printf("downcast argument check failed\n");
    return 1;
  }
  printf("ok %zu\n", ws);
  return 0;
}
