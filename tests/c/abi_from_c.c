/* A plain C caller of libsmla.so: no Python, no CUDA headers.  It plans the
 * FP8 decode of 128 tokens x 128 heads over 2176 columns for a 152-SM device,
 * sizes the workspace of a long-context split, and checks that host-detectable
 * mistakes come back as statuses before any CUDA call.  Prints one line per
 * check; exits non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "smla.h"

static int failures = 0;

#define CHECK(cond, ...)                       \
  do {                                         \
    if (cond) {                                \
      printf("ok   ");                         \
    } else {                                   \
      printf("FAIL ");                         \
      failures++;                              \
    }                                          \
    printf(__VA_ARGS__);                       \
    printf("\n");                              \
  } while (0)

static smla_args base(int sum_q, int width) {
  smla_args a;
  memset(&a, 0, sizeof(a));
  a.sum_q = sum_q;
  a.batch = sum_q;
  a.num_heads = 128;
  a.width = width;
  a.dtype = SMLA_E4M3;
  a.swa_rows = 128 * 128;
  a.comp_rows = 262144;
  return a;
}

int main(void) {
  CHECK(smla_abi_version() == SMLA_ABI_VERSION, "abi version %d", smla_abi_version());
  CHECK(strcmp(smla_status_string(SMLA_ERR_WORKSPACE_TOO_SMALL), "SMLA_ERR_WORKSPACE_TOO_SMALL") == 0,
        "status string");

  smla_args a = base(128, 2176);
  smla_plan p;
  smla_status st = smla_plan_decode_for_sm_count(&a, 152, &p);
  CHECK(st == SMLA_OK && p.kernel == SMLA_KERNEL_TCGEN05_SLOT_SPLIT && p.num_splits == 1 && p.grid == 256 &&
            p.clusters == 0 && p.workspace_bytes == 0,
        "plan 128 tokens: kernel %d splits %d grid %d clusters %d threads %d smem %d", p.kernel, p.num_splits,
        p.grid, p.clusters, p.threads, p.smem_bytes);

  /* balanced schedule: 76 pairs with equal column shares; pieces of cut
     tokens in 2 x 76 x 128 BF16 rows of 512, their LSEs (a copy per CTA) and
     2 x 76 counters */
  a.schedule = SMLA_SCHEDULE_BALANCED;
  st = smla_plan_decode_for_sm_count(&a, 152, &p);
  size_t pieces = (size_t)2 * 76 * 128;
  size_t want_pieces = (pieces * 512 * 2 + 255) / 256 * 256 + (2 * pieces * 4 + 255) / 256 * 256 +
                       (2 * 76 * 4 + 255) / 256 * 256;
  CHECK(st == SMLA_OK && p.num_splits == 1 && p.grid == 152 && p.clusters == 76 && p.workspace_bytes == want_pieces,
        "plan 128 tokens, balanced: splits %d grid %d clusters %d workspace %zu", p.num_splits, p.grid, p.clusters,
        p.workspace_bytes);
  a.schedule = SMLA_SCHEDULE_AUTO;

  smla_args b = base(4, 128 + 16384);
  st = smla_plan_decode_for_sm_count(&b, 152, &p);
  size_t rows = (size_t)4 * 128 * 19;
  size_t want = (rows * 512 * 2 + 255) / 256 * 256 + (rows * 4 + 255) / 256 * 256;
  CHECK(st == SMLA_OK && p.num_splits == 19 && p.grid == 152 && p.clusters == 0 && p.workspace_bytes == want,
        "plan 4 long tokens: splits %d grid %d workspace %zu", p.num_splits, p.grid, p.workspace_bytes);

  /* host-detectable mistakes: statuses, no CUDA call */
  smla_args c = base(128, 2176);
  c.num_heads = 96;
  st = smla_decode(&c, NULL);
  CHECK(st == SMLA_ERR_UNSUPPORTED && strstr(smla_last_error(), "num_heads") != NULL, "96 heads: %s",
        smla_last_error());
  c = base(128, 2176);
  st = smla_decode(&c, NULL); /* every pointer NULL */
  CHECK(st == SMLA_ERR_INVALID_ARG && strstr(smla_last_error(), "required") != NULL, "missing pointers: %s",
        smla_last_error());
  st = smla_decode(NULL, NULL);
  CHECK(st == SMLA_ERR_INVALID_ARG, "NULL args: %s", smla_last_error());
  c = base(0, 2176);
  c.batch = 1;
  CHECK(smla_decode(&c, NULL) == SMLA_OK, "empty batch is a no-op");
  c.batch = 0;
  CHECK(smla_decode(&c, NULL) == SMLA_ERR_INVALID_ARG, "batch 0: %s", smla_last_error());
  st = smla_plan_decode_for_sm_count(&a, 0, &p);
  CHECK(st == SMLA_ERR_INVALID_ARG, "sm_count 0: %s", smla_last_error());
  return failures == 0 ? 0 : 1;
}
