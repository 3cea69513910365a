/* A plain C99 client of the library: compiles against include/fa.h alone, links
 * libfa_sm103.so, and calls the entry points that need no GPU (status strings, workspace size,
 * argument checks that return before any device work). */
#include <stdio.h>

#include "fa.h"

int main(void) {
  const size_t ws = fa_bwd_workspace_size(1, 1, 128, 64);
  const fa_status unsupported = fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 96, 0, -1.0f,
                                       NULL, NULL);
  const fa_status invalid = fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 0, 64, 0, -1.0f, NULL,
                                   NULL);
  printf("status_string %s\n", fa_status_string(FA_ERR_TIMEOUT));
  printf("workspace %zu\n", ws);
  printf("unsupported %d\n", (int)unsupported);
  printf("invalid %d\n", (int)invalid);
  return 0;
}
