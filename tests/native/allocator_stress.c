/* Random-operation stress of the host allocator through the C ABI, built with
 * AddressSanitizer and UndefinedBehaviorSanitizer by tests/test_allocator_sanitized.py.
 *
 * Every call of include/pkv.h that touches only host state is driven from one
 * seeded generator: create (+ append), fork, free, single and batch appends
 * (short pools make some fail, which must change nothing; batches may repeat
 * a sequence), preemption, admission with a
 * watermark, prefix-cache hits, full and incremental batch tables.  After
 * every step the invariants the pages fix are checked:
 *   - a block's reference count is the number of tables holding it, so the
 *     counts sum to the tables' total length;
 *   - a block on the free stack has count 0;
 *   - a table holds exactly ceil(len / block_size) blocks (a block is taken
 *     only when the previous one is full);
 *   - pkv_block_tables_update leaves the same rows as pkv_block_tables.
 * Exit status 0 when all hold; otherwise the failing check's number.
 *
 * usage: allocator_stress <seed> <steps> <caching 0|1>
 */
#include "pkv.h"

#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#define NUM_BLOCKS 96
#define T 16
#define MAX_SEQS 48
#define MAX_BLOCKS NUM_BLOCKS
#define VOCAB 3

static uint64_t g_state;

static uint32_t next_u32(void) {
  g_state = g_state * 6364136223846793005ULL + 1442695040888963407ULL;
  return (uint32_t)(g_state >> 33);
}

static int below(int n) { return n > 0 ? (int)(next_u32() % (uint32_t)n) : 0; }

static int64_t live[MAX_SEQS];
static int n_live;
static int64_t next_id = 1;

static void forget(int64_t id) {
  for (int i = 0; i < n_live; ++i)
    if (live[i] == id) {
      live[i] = live[--n_live];
      return;
    }
}

/* rows kept across steps for pkv_block_tables_update */
static int32_t rows_tables[MAX_SEQS * MAX_BLOCKS];
static int64_t rows_state[MAX_SEQS * 2];

static int check(pkv_pool* p) {
  int64_t sum_rc = 0, sum_len = 0;
  for (int32_t b = 0; b < NUM_BLOCKS; ++b) {
    int32_t rc = -1;
    if (pkv_block_refcount(p, b, &rc) != PKV_OK || rc < 0) return 10;
    sum_rc += rc;
  }
  static int32_t tab[MAX_BLOCKS];
  for (int i = 0; i < n_live; ++i) {
    int32_t nb = 0;
    int64_t len = 0;
    if (pkv_seq_table(p, live[i], tab, MAX_BLOCKS, &nb, &len) != PKV_OK) return 11;
    if ((int64_t)nb != (len + T - 1) / T) return 12;
    sum_len += nb;
  }
  if (sum_rc != sum_len) return 13;
  static int32_t stack[NUM_BLOCKS];
  int32_t n_free = 0;
  if (pkv_free_stack(p, stack, NUM_BLOCKS, &n_free) != PKV_OK) return 14;
  for (int32_t i = 0; i < n_free; ++i) {
    int32_t rc = -1;
    if (pkv_block_refcount(p, stack[i], &rc) != PKV_OK || rc != 0) return 15;
  }
  /* a batch of up to all live sequences, in a shuffled order */
  int64_t batch[MAX_SEQS];
  const int n = n_live ? 1 + below(n_live) : 0;
  memcpy(batch, live, sizeof(int64_t) * (size_t)n_live);
  for (int i = n_live - 1; i > 0; --i) {
    const int j = below(i + 1);
    const int64_t x = batch[i];
    batch[i] = batch[j];
    batch[j] = x;
  }
  static int32_t want[MAX_SEQS * MAX_BLOCKS];
  int32_t want_ctx[MAX_SEQS], got_ctx[MAX_SEQS];
  if (pkv_block_tables(p, batch, n, MAX_BLOCKS, want, want_ctx) != PKV_OK) return 16;
  if (pkv_block_tables_update(p, batch, n, MAX_BLOCKS, rows_tables, rows_state, got_ctx) != PKV_OK)
    return 17;
  if (memcmp(want, rows_tables, sizeof(int32_t) * (size_t)n * MAX_BLOCKS) != 0) return 18;
  if (memcmp(want_ctx, got_ctx, sizeof(int32_t) * (size_t)n) != 0) return 19;
  return 0;
}

static void tokens_for(int32_t* ids, int n, int variant) {
  /* prompts from a tiny vocabulary, so that full blocks repeat across requests */
  for (int i = 0; i < n; ++i) ids[i] = (i / T + variant) % VOCAB;
}

int main(int argc, char** argv) {
  if (argc != 4) return 2;
  g_state = strtoull(argv[1], NULL, 10) * 2654435761ULL + 1;
  const int steps = atoi(argv[2]);
  const int caching = atoi(argv[3]);
  pkv_pool* p = NULL;
  if (pkv_pool_create(NUM_BLOCKS, T, NULL, &p) != PKV_OK) return 3;
  if (caching && pkv_pool_enable_prefix_cache(p) != PKV_OK) return 4;
  static int64_t slots[MAX_SEQS * 64];
  static int32_t cow[2 * MAX_SEQS];
  static int32_t ids[8 * T];
  int64_t preempted[MAX_SEQS];
  for (int step = 0; step < steps; ++step) {
    const int op = below(10);
    int32_t n_cow = 0, n_pre = 0;
    if (op == 0 || n_live == 0) {
      if (n_live < MAX_SEQS) {
        const int64_t id = next_id++;
        if (caching && below(2)) {
          const int n = 1 + below(8 * T - 1);
          int32_t have = 0;
          tokens_for(ids, n, below(2));
          if (pkv_seq_create_cached(p, id, ids, n, &have) != PKV_OK) return 20;
          live[n_live++] = id;
          if (have < n) pkv_seq_append_tokens(p, id, ids + have, n - have, slots, cow, 1, &n_cow);
        } else if (below(2)) {
          if (pkv_seq_admit(p, id, below(40), 2 + below(4), slots) == PKV_OK) live[n_live++] = id;
        } else {
          if (pkv_seq_create(p, id) != PKV_OK) return 21;
          live[n_live++] = id;
          pkv_seq_append(p, id, below(50), slots, cow, 1, &n_cow);
        }
      }
    } else if (op == 1) {
      if (n_live < MAX_SEQS) {
        const int64_t id = next_id++;
        if (pkv_seq_fork(p, live[below(n_live)], id) != PKV_OK) return 22;
        live[n_live++] = id;
      }
    } else if (op == 2) {
      const int64_t id = live[below(n_live)];
      if (pkv_seq_free(p, id) != PKV_OK) return 23;
      forget(id);
      if (below(2)) { /* the same id again: a new sequence */
        if (pkv_seq_create(p, id) != PKV_OK) return 24;
        live[n_live++] = id;
      }
    } else if (op <= 4) {
      pkv_seq_append(p, live[below(n_live)], 1 + below(30), slots, cow, 1, &n_cow);
    } else if (op <= 7) {
      int64_t batch[MAX_SEQS];
      const int n = 1 + below(n_live);
      /* half the batches name some sequences twice: such a sequence takes
         one token per mention, in batch order */
      const int repeat = below(2);
      for (int i = 0; i < n; ++i) batch[i] = repeat ? live[below(n_live)] : live[i];
      const pkv_status st = pkv_batch_append(p, batch, n, slots, cow, n, &n_cow);
      if (st != PKV_OK && st != PKV_ERR_OUT_OF_BLOCKS) return 25;
      if (st != PKV_OK && n_cow != 0) return 26;
    } else if (op == 8) {
      int64_t batch[MAX_SEQS];
      const int n = n_live;
      memcpy(batch, live, sizeof(int64_t) * (size_t)n);
      if (pkv_batch_append_preempt(p, batch, n, slots, cow, n, &n_cow, preempted, &n_pre) != PKV_OK)
        return 27;
      for (int i = 0; i < n_pre; ++i) forget(preempted[i]);
    } else {
      /* a sequence that does not exist: an error and no change */
      if (pkv_seq_append(p, -5, 1, slots, cow, 1, &n_cow) != PKV_ERR_UNKNOWN_SEQ) return 28;
    }
    const int bad = check(p);
    if (bad) {
      fprintf(stderr, "step %d op %d: check %d failed (%s)\n", step, op, bad, pkv_last_error());
      pkv_pool_destroy(p);
      return bad;
    }
  }
  pkv_pool_destroy(p);
  printf("ok %d steps\n", steps);
  return 0;
}
