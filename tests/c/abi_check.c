/* Plain C99 use of the library's C ABI (include/mok.h): size queries, status strings and
 * host-side argument checks, none of which launches a kernel.  Built and run by
 * tests/test_abi.py to show that the boundary needs no C++ or PyTorch types. */
#include <stdio.h>
#include <string.h>

#include "mok.h"

static int fail(const char *what) {
  fprintf(stderr, "abi_check: %s\n", what);
  return 1;
}

int main(void) {
  mok_dims d;
  memset(&d, 0, sizeof d);
  d.T = 4096;
  d.d = 7168;
  d.E = 256;
  d.k = 8;
  d.F = 2048;
  d.F_shared = 2048;
  d.n_shared = 1;
  d.dtype = MOK_BF16;
  if (mok_workspace_size(&d, MOK_PASS_FORWARD) == 0) return fail("forward workspace size");
  if (mok_workspace_size(&d, MOK_PASS_BACKWARD) == 0) return fail("backward workspace size");
  if (mok_saved_size(&d) == 0) return fail("saved size");
  if (mok_prepared_size(&d) != 0 || mok_prepared_bwd_size(&d) != 0) return fail("bf16 prepared sizes");
  d.dtype = MOK_MXFP8;
  if (mok_prepared_size(&d) == 0 || mok_prepared_bwd_size(&d) == 0) return fail("mxfp8 prepared sizes");
  d.d = 100; /* not a multiple of 128 */
  if (mok_workspace_size(&d, MOK_PASS_FORWARD) != 0) return fail("bad dims accepted");
  if (mok_route(&d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) != MOK_ERR_UNSUPPORTED)
    return fail("bad dims not reported");
  d.d = 7168;
  if (mok_route(&d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) != MOK_ERR_INVALID_ARG)
    return fail("null pointers not reported");
  if (strncmp(mok_status_string(MOK_ERR_WORKSPACE), "MOK_ERR_WORKSPACE", 17) != 0)
    return fail("status string");
  printf("abi_check ok\n");
  return 0;
}
