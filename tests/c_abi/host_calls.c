/*
 * A plain C caller of the library's C ABI (include/pagedkv.h): no CUDA or
 * PyTorch headers, only the declared entry points with host pointers and
 * sizes. It runs without a GPU: the block allocator and the scheduler are
 * host code, and the attention entry points are only called with arguments
 * they must reject before touching the device.
 *
 * Checks, printing "ok" on success (exit status 0) or the first failure:
 *  - the worked allocation example (three requests of 3, 5 and 2 tokens in
 *    4-token blocks take ceil(T/B) blocks each, 3 + 5 + 2 = 10 slots of the
 *    16 reserved), copy-on-write on a shared, partly filled block, and the
 *    pool's free + used block count;
 *  - a scheduler loop: every request runs to its token budget, every block
 *    returns to the free list;
 *  - argument validation of the decode, merge and block-copy calls.
 */
#include <stdio.h>
#include <stdlib.h>

#include "pagedkv.h"

#define CHECK(cond, what)                                   \
  do {                                                      \
    if (!(cond)) {                                          \
      printf("FAIL %s (line %d)\n", (what), __LINE__);      \
      return 1;                                             \
    }                                                       \
  } while (0)

static int allocator_example(void) {
  pkv_allocator* a = NULL;
  CHECK(pkv_alloc_create(16, 4, 7, &a) == PKV_OK, "create");
  const int lens[3] = {3, 5, 2};
  int ids[3];
  int64_t slots[8];
  int32_t pairs[16];
  int n_cow = 0;
  for (int r = 0; r < 3; ++r) {
    CHECK(pkv_seq_new(a, &ids[r]) == PKV_OK, "seq_new");
    CHECK(pkv_seq_append(a, ids[r], lens[r], slots, pairs, &n_cow) == PKV_OK, "append");
    CHECK(n_cow == 0, "no copy for a private sequence");
    int32_t table[4];
    int nb = 0;
    CHECK(pkv_seq_block_table(a, ids[r], table, 4, &nb) == PKV_OK, "table");
    CHECK(nb == (lens[r] + 3) / 4, "ceil(T/B) blocks");
    for (int t = 0; t < lens[r]; ++t)
      CHECK(slots[t] == (int64_t)table[t / 4] * 4 + t % 4, "slot = block * B + offset");
  }
  int free_blocks = 0, used_blocks = 0;
  long long used_slots = 0;
  CHECK(pkv_alloc_stats(a, &free_blocks, &used_blocks, &used_slots) == PKV_OK, "stats");
  CHECK(used_blocks == 4 && used_slots == 10 && free_blocks == 12, "3 + 5 + 2 tokens in 4 blocks");
  /* a fork shares the 5-token sequence's blocks; its first append writes
   * into the shared, partly filled second block and gets a copy */
  int child = -1;
  CHECK(pkv_seq_fork(a, ids[1], &child) == PKV_OK, "fork");
  CHECK(pkv_seq_append(a, child, 1, slots, pairs, &n_cow) == PKV_OK, "child append");
  CHECK(n_cow == 1, "one copy-on-write pair");
  int32_t pt[2], ct[2];
  int np = 0, nc = 0;
  CHECK(pkv_seq_block_table(a, ids[1], pt, 2, &np) == PKV_OK, "parent table");
  CHECK(pkv_seq_block_table(a, child, ct, 2, &nc) == PKV_OK, "child table");
  CHECK(pt[0] == ct[0] && pairs[0] == pt[1] && pairs[1] == ct[1] && pt[1] != ct[1],
        "the copy goes from the shared block to the child's new one");
  CHECK(pkv_alloc_stats(a, &free_blocks, &used_blocks, NULL) == PKV_OK, "stats");
  CHECK(free_blocks + used_blocks == 16, "free + used = pool");
  for (int r = 0; r < 3; ++r) CHECK(pkv_seq_free(a, ids[r]) == PKV_OK, "free");
  CHECK(pkv_seq_free(a, child) == PKV_OK, "free child");
  CHECK(pkv_alloc_stats(a, &free_blocks, &used_blocks, NULL) == PKV_OK, "stats");
  CHECK(free_blocks == 16 && used_blocks == 0, "all blocks back");
  pkv_alloc_destroy(a);
  return 0;
}

static int scheduler_loop(void) {
  pkv_allocator* a = NULL;
  pkv_scheduler* s = NULL;
  CHECK(pkv_alloc_create(64, 16, 3, &a) == PKV_OK, "create");
  CHECK(pkv_sched_create(a, 16, 4, &s) == PKV_OK, "sched");
  for (int r = 0; r < 10; ++r)
    CHECK(pkv_sched_add_request(s, r, 20 + 13 * r, 5 + r) == PKV_OK, "add");
  CHECK(pkv_sched_add_request(s, 3, 10, 2) == PKV_ERR_INVALID_ARG, "id in use");
  int running = 0, admitted = 0, finished = 0, done = 0, iters = 0;
  int waiting = 1;
  while ((waiting > 0 || running > 0) && iters < 10000) {
    CHECK(pkv_sched_step(s, &running, &admitted, &finished) == PKV_OK, "step");
    done += finished;
    CHECK(running <= 4, "batch bound");
    int32_t ctx[4];
    CHECK(pkv_sched_running(s, NULL, ctx, NULL, 4) == PKV_OK, "running");
    CHECK(pkv_sched_counts(s, &waiting, &running, NULL) == PKV_OK, "counts");
    ++iters;
  }
  CHECK(pkv_sched_step(s, &running, &admitted, &finished) == PKV_OK, "last step");
  done += finished;
  CHECK(done == 10, "every request finished");
  int free_blocks = 0;
  CHECK(pkv_alloc_stats(a, &free_blocks, NULL, NULL) == PKV_OK, "stats");
  CHECK(free_blocks == 64, "every block returned");
  pkv_sched_destroy(s);
  pkv_alloc_destroy(a);
  return 0;
}

static int validation(void) {
  void* fake = (void*)(uintptr_t)0x10000; /* never dereferenced: rejected first */
  pkv_cache_desc c = {8, 16, 2, 128, PKV_DTYPE_BF16};
  /* group of 9 query heads per KV head: unsupported */
  CHECK(pkv_paged_attention_decode(fake, fake, fake, fake, c, NULL, NULL, fake, 64, fake, 4, 18,
                                   100, 0.088f, 0, NULL, 0, NULL, NULL) == PKV_ERR_UNSUPPORTED,
        "group 9");
  /* split form without a workspace */
  CHECK(pkv_paged_attention_decode(fake, fake, fake, fake, c, NULL, NULL, fake, 64, fake, 4, 8,
                                   100, 0.088f, 64, NULL, 0, NULL, NULL) == PKV_ERR_INVALID_ARG,
        "no workspace");
  CHECK(pkv_paged_attention_reduce(fake, NULL, 0, fake, 4, 8, 96, 100, 64, NULL) ==
            PKV_ERR_UNSUPPORTED,
        "head_dim 96");
  CHECK(pkv_copy_blocks(fake, fake, c, NULL, 3, NULL) == PKV_ERR_INVALID_ARG, "no pairs");
  CHECK(pkv_split_partition_size(1033, 16, 512) == 528, "split size");
  {
    const int32_t lens[5] = {3, 9, 1, 9, 5};
    int32_t order[5];
    CHECK(pkv_longest_first_order(lens, 5, order) == PKV_OK && order[0] == 1 && order[1] == 3 &&
              order[2] == 4 && order[3] == 0 && order[4] == 2,
          "longest first");
  }
  CHECK(pkv_decode_workspace_bytes(8, 24, 256, 131072, 512) ==
            (size_t)8 * 24 * 256 * (256 + 2) * 4,
        "workspace bytes");
  return 0;
}

int main(void) {
  if (allocator_example() || scheduler_loop() || validation()) return 1;
  printf("ok\n");
  return 0;
}
