/* A plain C caller of libmoe.so: compiles against include/moe.h alone and
 * exercises the host-side part of the boundary (no device memory is touched):
 * the version string, workspace sizes, status strings and argument checks. */
#include <stdio.h>
#include <string.h>

#include "moe.h"

static int fails = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "FAILED: %s (line %d)\n", #cond, __LINE__); \
      ++fails;                                                   \
    }                                                            \
  } while (0)

int main(void) {
  moe_shape_t s;
  memset(&s, 0, sizeof(s));
  s.T = 8192; s.d = 6144; s.E = 8; s.K = 2; s.F = 16384; s.dtype = MOE_BF16;
  s.drop = 1; s.capacity_factor = 1.0f; s.subseq_len = 4096; s.renorm = 1; s.Fs = 0;
  CHECK(moe_version() != NULL && strlen(moe_version()) >= 5);
  const size_t ws = moe_workspace_size(&s);
  CHECK(ws >= MOE_FFN_BWD_WORKSPACE_BYTES && ws % 256 == 0);
  CHECK(moe_padded_capacity(&s) == 2048);          /* 2 sub-sequences x 1024 */
  CHECK(strlen(moe_status_string(MOE_ERR_INVALID_ARG)) > 0);
  /* argument checks fail before any device access */
  void *fake = (void *)(size_t)(1 << 20);
  CHECK(moe_route(&s, NULL, fake, NULL, NULL, fake, NULL, fake, fake, fake, fake, fake, 0) ==
        MOE_ERR_INVALID_ARG);
  CHECK(moe_sum_partials(MOE_BF16, 0, 8, 64, fake, fake, 0) == MOE_ERR_INVALID_ARG);
  s.E = 65;                                         /* above the 64-expert limit */
  CHECK(moe_workspace_size(&s) == 0);
  s.E = 8; s.drop = 0;
  CHECK(moe_padded_capacity(&s) == 0);             /* dropless: no fixed capacity */
  if (fails == 0) printf("c abi probe ok\n");
  return fails == 0 ? 0 : 1;
}
