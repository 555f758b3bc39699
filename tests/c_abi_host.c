/* Plain C99 user of include/flce.h: compiles against the header, links the
 * library and calls the entry points that need no GPU (sizing, status strings,
 * argument validation).  Exit code 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "flce.h"

static int fails = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      ++fails;                                                   \
    }                                                            \
  } while (0)

int main(void) {
  const int64_t T = 65536, Hd = 2048, V = 124160;
  size_t fws = flce_forward_workspace_size(T, Hd, V);
  size_t bws = flce_backward_workspace_size(T, Hd, V);
  CHECK(flce_abi_version() == FLCE_ABI_VERSION);
  CHECK(fws > 256);
  CHECK(bws < (size_t)(T * V * 2)); /* never a [T x V] bf16 buffer */
  CHECK(flce_backward_chunk_tokens(T, Hd, V, bws) == 8192);
  CHECK(flce_score_workspace_size(T, Hd, V) > fws);
  CHECK(flce_combine_workspace_size(T, 2) > 0 && flce_combine_workspace_size(T, 65) == 0);
  CHECK(strcmp(flce_status_string(FLCE_ERR_TIMEOUT), "FLCE_ERR_TIMEOUT") == 0);
  CHECK(strcmp(flce_kernel_name(FLCE_KERNEL_BWD_DH_DW), "bwd_dh_dw") == 0);
  /* argument errors are returned before anything touches a device */
  char ws[512];
  void* ws_al = (void*)(((size_t)ws + 255) & ~(size_t)255);
  float f[4];
  flce_status st = flce_forward((const void*)16, (const void*)16, (const int64_t*)16, 10, 100, 50, -100,
                                FLCE_REDUCTION_MEAN, f, f, f, NULL, ws_al, 256, NULL);
  CHECK(st == FLCE_ERR_UNSUPPORTED); /* Hd not a multiple of 64 */
  st = flce_forward((const void*)16, (const void*)16, (const int64_t*)16, 10, 64, 50, 7, FLCE_REDUCTION_MEAN, f, f,
                    f, NULL, ws_al, 256, NULL);
  CHECK(st == FLCE_ERR_INVALID_ARG); /* ignore_index inside [0, V) */
  CHECK(strlen(flce_last_error()) > 0);
  st = flce_forward_shard((const void*)16, (const void*)16, (const int64_t*)16, 10, 64, 60, 50, 100, -100, f, f,
                          ws_al, 256, NULL);
  CHECK(st == FLCE_ERR_INVALID_ARG); /* shard [50, 110) outside [0, 100) */
  st = flce_forward_noalloc((const void*)16, (const void*)16, (const int64_t*)16, 300000, 64, 100, -100,
                            FLCE_REDUCTION_MEAN, f, f, f, NULL, NULL, NULL);
  CHECK(st == FLCE_ERR_WORKSPACE); /* beyond the built-in scratch */
  printf("%s\n", fails ? "FAILED" : "ok");
  return fails ? 1 : 0;
}
