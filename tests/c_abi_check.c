/* A C99 client of the library: include/awq.h must compile as plain C and the
 * host-only entry points (defaults, status strings, size queries) must work
 * without a GPU. Built and run by tests/test_abi.py. */
#include <stdio.h>
#include <string.h>

#include "awq.h"

int main(void) {
  awq_config cfg;
  size_t bytes = 0;
  awq_config_default(&cfg);
  if (cfg.w_bit != 4 || cfg.group != 128 || cfg.n_grid != 20 || cfg.zero_point != 1) return 1;
  if (strcmp(awq_status_string(AWQ_OK), awq_status_string(AWQ_ERR_TIMEOUT)) == 0) return 2;
  if (awq_workspace_size(4096, 4096, 4096, &cfg, &bytes) != AWQ_OK || bytes == 0) return 3;
  if (awq_workspace_size(0, 4096, 4096, &cfg, &bytes) != AWQ_ERR_INVALID_ARG) return 4;
  if (awq_packed_bytes(4096, 4096, &cfg) != (size_t)4096 * 4096 / 2 + 2 * 2 * 4096 * 32) return 5;
  cfg.group = 96;
  if (awq_workspace_size(4096, 4096, 4096, &cfg, &bytes) != AWQ_ERR_UNSUPPORTED) return 6;
  printf("c abi ok\n");
  return 0;
}
