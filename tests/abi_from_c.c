/* Compiled as C99 by tests/test_abi_host.py and linked against libkvsel.so:
 * the header must be plain C, and the host-only entry points must be callable
 * from C. Prints one line per check; exits non-zero on the first failure.
 * Needs no GPU: nothing here launches a kernel. */
#include <stdio.h>
#include <string.h>

#include "kvsel.h"

#define CHECK(cond, what)                      \
  do {                                         \
    if (!(cond)) {                             \
      printf("FAIL %s\n", what);               \
      return 1;                                \
    }                                          \
    printf("ok %s\n", what);                   \
  } while (0)

int main(void) {
  /* "KV cache offloading", section "Why the cache leaves the GPU": 32 layers,
   * 2 KV heads, d 128, bf16 give 32768 bytes per token */
  CHECK(kvsel_kv_bytes_per_token(32, 2, 128, 2) == 32768, "kv bytes per token");
  CHECK(kvsel_kv_bytes_per_token(-1, 2, 128, 2) == -1, "kv bytes rejects a negative count");
  CHECK(strncmp(kvsel_version(), "kvsel", 5) == 0, "version string");

  kvsel_budget_in in;
  memset(&in, 0, sizeof in);
  in.block_size = 64; in.kv_heads = 2; in.head_dim = 128; in.elem_bytes = 2;
  in.hidden = 4096; in.n_blocks = 2048;
  in.h2d_bytes_per_s = 64e9; in.recompute_flop_per_s = 1e15; in.kappa = 2.0;
  in.keep_floor = 0.05; in.gamma = 0.8; in.tau_s = 0.0; in.keep_override = 0.125;
  kvsel_budget_out out;
  CHECK(kvsel_budget(&in, &out) == KVSEL_OK, "budget accepts valid input");
  /* one block of one layer: 64 * 2 * 128 * 2 = 32768 B; copy cost 2 * S / BW */
  CHECK(out.c_copy_s == 2.0 * 32768.0 / 64e9, "budget copy cost");
  CHECK(out.k == 256, "budget k from the override ratio (0.125 of 2048)");
  CHECK(out.dense == 0, "budget: 256 of 2048 is not dense at gamma 0.8");
  in.h2d_bytes_per_s = 0.0;
  CHECK(kvsel_budget(&in, &out) == KVSEL_ERR_INVALID_ARG, "budget rejects a zero bandwidth");
  CHECK(kvsel_last_error() != NULL && kvsel_last_error()[0] != '\0', "last error message");

  kvsel_problem p = {16, 32, 8, 128, 32, 1024, 128};
  CHECK(kvsel_workspace_size(&p, KVSEL_WS_SCORE_TOPK) >= (size_t)16 * 1024 * 4, "score workspace size");
  CHECK(kvsel_workspace_size(&p, KVSEL_WS_SPARSE_DECODE) > 0, "decode workspace size");
  kvsel_problem bad = p;
  bad.head_dim = 96;
  CHECK(kvsel_workspace_size(&bad, KVSEL_WS_SCORE_TOPK) == 0, "unsupported shape has no workspace");
  CHECK(kvsel_score_topk(&bad, NULL, NULL, NULL, NULL, 1.0f, 0.0f, NULL, NULL, NULL, NULL, NULL,
                         NULL, NULL, NULL, 0, NULL) == KVSEL_ERR_UNSUPPORTED,
        "score_topk rejects an unsupported shape before touching the device");
  printf("all ok\n");
  return 0;
}
