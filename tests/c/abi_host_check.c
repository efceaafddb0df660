/* Uses the library from plain C99 through include/cs_chain.h alone, without a
 * GPU: the header compiles as C, the structs and enums mean the same as in the
 * library, and the host-only entry points (desc defaults, validation, the
 * dispatch order, the tuning table) behave as documented.  Prints "ok" and
 * exits 0, or names the first failed check and exits 1. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "cs_chain.h"

#define CHECK(cond)                                                      \
  do {                                                                   \
    if (!(cond)) {                                                       \
      fprintf(stderr, "check failed at line %d: %s (%s)\n", __LINE__, #cond, \
              cs_last_error_string());                                   \
      return 1;                                                          \
    }                                                                    \
  } while (0)

static int stage_of(uint32_t u) { return (int)(u >> 30); }
static int mtile_of(uint32_t u) { return (int)((u >> 14) & 0xFFFu); }

int main(int argc, char** argv) {
  cs_chain_desc d;
  size_t n = 0;
  uint32_t* units;
  size_t i;
  int seen_consumer_of_row0 = 0, entry = -2, count = -1;
  cs_chain_desc resolved;
  cs_chain_t plan = (cs_chain_t)0x1;

  CHECK(cs_abi_version() == CS_ABI_VERSION);
  CHECK(cs_chain_desc_init(&d) == CS_OK);
  CHECK(d.kind == CS_CHAIN_MLP_GELU && d.dtype == CS_F16 && d.policy == CS_SYNC_TILE && d.lag == -1);
  CHECK(d.tuned == 0 && d.out_release == 0 && d.head_dim == 128);

  /* the GPT-3 shard at M = 2048 on 152 SMs: every producer unit precedes the
     consumers of its rows, and the count matches 512 x 256 tiles */
  d.M = 2048;
  d.H = 12288;
  d.F = 6144;
  d.weight_layout = CS_WEIGHTS_NK;
  CHECK(cs_schedule_build(&d, 152, NULL, 0, &n) == CS_OK);
  CHECK(n == 4 * (24 + 48));
  units = (uint32_t*)malloc(n * sizeof(uint32_t));
  CHECK(units != NULL);
  CHECK(cs_schedule_build(&d, 152, units, n, &n) == CS_OK);
  for (i = 0; i < n; ++i) {
    if (stage_of(units[i]) == 1 && mtile_of(units[i]) == 0) seen_consumer_of_row0 = 1;
    if (stage_of(units[i]) == 0 && mtile_of(units[i]) == 0) CHECK(!seen_consumer_of_row0);
  }
  CHECK(seen_consumer_of_row0);
  free(units);

  /* the GPT-3 shard at one row with six K-splits in K-range order: the first
     consumer units listed are K-split 0 of consecutive column tiles, and
     cs_chain_plan_info reports the order and the first stage's own splits */
  {
    cs_chain_desc k = d;
    cs_chain_info info;
    size_t first = 0;
    k.M = 1;
    k.tile_m = 128;
    k.tile_n = 128;
    k.split_k = 3;
    k.split_k_first = 6;
    k.raster = 3;
    k.tuned = -1;
    CHECK(cs_chain_plan_info(&k, 152, &info) == CS_OK);
    CHECK(info.raster == 3 && info.split_k[0] == 6 && info.split_k[1] == 3);
    CHECK(cs_schedule_build(&k, 152, NULL, 0, &n) == CS_OK);
    CHECK(n == (size_t)(48 * 6 + 96 * 3));
    units = (uint32_t*)malloc(n * sizeof(uint32_t));
    CHECK(units != NULL);
    CHECK(cs_schedule_build(&k, 152, units, n, &n) == CS_OK);
    while (first < n && stage_of(units[first]) == 0) ++first;
    CHECK(first == 48 * 6);
    for (i = 0; i < 96; ++i) CHECK(units[first + i] == (uint32_t)((1u << 30) | i));
    free(units);
    k.raster = 4;
    CHECK(cs_schedule_build(&k, 152, NULL, 0, &n) == CS_ERR_INVALID_ARG);
  }

  /* validation: status codes and a message, no abort */
  d.tile_m = 64;
  CHECK(cs_schedule_build(&d, 152, NULL, 0, &n) == CS_ERR_INVALID_ARG);
  CHECK(strlen(cs_last_error_string()) > 0);
  d.tile_m = 0;
  CHECK(cs_chain_plan(NULL, &plan) == CS_ERR_INVALID_ARG);
  CHECK(cs_chain_destroy(NULL) == CS_OK);

  /* the tuning table named on the command line (the shipped one) */
  CHECK(cs_tune_clear() == CS_OK && cs_tune_size() == 0);
  CHECK(cs_tune_match(&d, 152, &entry, &resolved) == CS_OK && entry == -1);
  if (argc > 1) {
    CHECK(cs_tune_load(argv[1], &count) == CS_OK && count > 0 && cs_tune_size() == count);
    d.policy = CS_SYNC_AUTO;
    CHECK(cs_tune_match(&d, 152, &entry, &resolved) == CS_OK && entry >= 0);
    CHECK(resolved.policy == CS_SYNC_TILE || resolved.policy == CS_SYNC_ROW || resolved.policy == CS_SYNC_STRIDED);
    CHECK(cs_tune_load("/nonexistent/table.json", &count) == CS_ERR_INVALID_ARG && cs_tune_size() > 0);
    CHECK(cs_tune_clear() == CS_OK);
  }
  printf("ok\n");
  return 0;
}
