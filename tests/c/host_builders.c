/* A plain C11 program against libunip's C ABI (include/unip.h, include/unip_sched.h):
 * packs the prompts given on the command line with unip_ffd_pack, then runs a
 * chunked-prefill schedule with the step builder, printing one line per bin and
 * per step.  Host calls only: no GPU is needed. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "unip.h"
#include "unip_sched.h"

int main(int argc, char **argv) {
  if (argc < 3) return 2;
  const int32_t capacity = (int32_t)atoi(argv[1]);
  const int32_t n = argc - 2;
  int32_t lengths[64], order[64], bin_cu[65], num_bins = 0;
  if (n > 64) return 2;
  for (int32_t i = 0; i < n; ++i) lengths[i] = (int32_t)atoi(argv[i + 2]);
  int32_t rc = unip_ffd_pack(lengths, n, capacity, order, bin_cu, &num_bins);
  printf("pack %d %s\n", rc, unip_status_string(rc));
  if (rc != UNIP_OK) return 1;
  for (int32_t b = 0; b < num_bins; ++b) {
    printf("bin");
    for (int32_t k = bin_cu[b]; k < bin_cu[b + 1]; ++k) printf(" %d", order[k]);
    printf("\n");
  }
  /* every prompt as a request sampling 2 tokens, 8-token budget, 4-token pages */
  unip_step_builder *sb = NULL;
  rc = unip_step_builder_create(8, 4, 256, 64, 8, 1, &sb);
  if (rc != UNIP_OK) return 1;
  for (int32_t i = 0; i < n; ++i) {
    int32_t id = -1;
    if (lengths[i] > 0 && unip_step_builder_add(sb, lengths[i], 2, &id) != UNIP_OK) return 1;
  }
  int32_t cu[9], pos[8], slots[8], bt[8 * 64], ids[8], fin[8];
  uint8_t mask[8];
  unip_step_buffers buf = {cu, pos, slots, bt, ids, mask, fin};
  for (int step = 0; step < 1000; ++step) {
    unip_step_counts c;
    if (unip_step_builder_next(sb, &buf, &c) != UNIP_OK) return 1;
    if (c.num_segs == 0) break;
    printf("step");
    for (int32_t s = 0; s < c.num_segs; ++s)
      printf(" [%d %d %d %d]", ids[s], pos[cu[s]], cu[s + 1] - cu[s], (int)mask[s]);
    printf("\n");
  }
  unip_step_builder_destroy(sb);
  printf("bad %s\n", unip_status_string(unip_ffd_pack(lengths, n, 0, order, bin_cu, &num_bins)));
  return 0;
}
