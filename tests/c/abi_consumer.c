/*
 * A plain C99 consumer of the library's C ABI: includes the public header,
 * links against libsls.so and makes calls that need no GPU (version, stats,
 * workspace sizes, and calls that fail host-side validation before any
 * launch).  Prints one "name=value" line per result for the test to check.
 */
#include <stdint.h>
#include <stdio.h>

#include "sls.h"

int main(void) {
  sls_attn_desc d = {2, 8, 2, 128, 16, 1024, SLS_DTYPE_BF16, 0, 0.0f};
  const void* dev = (const void*)(uintptr_t)0x1000; /* never dereferenced */
  printf("version=%d\n", (int)sls_version());
  printf("select_ws=%zu\n", sls_select_pages_workspace_size(&d));
  printf("null_desc=%d\n", (int)sls_pagemeta_build(NULL, dev, dev, (void*)dev, (void*)dev, NULL));
  printf("null_cache=%d\n", (int)sls_pagemeta_build(&d, NULL, dev, (void*)dev, (void*)dev, NULL));
  printf("error=%s\n", sls_last_error());
  printf("misaligned=%d\n",
         (int)sls_pagemeta_build(&d, (const void*)(uintptr_t)0x1002, dev, (void*)dev, (void*)dev, NULL));
  d.head_dim = 96;
  printf("bad_dim=%d\n", (int)sls_pagemeta_build(&d, dev, dev, (void*)dev, (void*)dev, NULL));
  sls_stats st;
  printf("stats_null=%d\n", (int)sls_get_stats(NULL, 0));
  (void)st;
  return 0;
}
