/* A plain C11 user of the C ABI's host calls: the block allocator (slots
 * through the table, fork, copy-on-write, tables) and SHA-256.  Built and run
 * by tests/test_abi_library.py; prints "ok" and exits 0 when every check
 * holds, else exits with the number of the failed check. */
#include <stdio.h>
#include <string.h>

#include "pa.h"

#define CHECK(n, cond)                                   \
  do {                                                   \
    if (!(cond)) {                                       \
      fprintf(stderr, "check %d failed: %s\n", n, #cond); \
      return n;                                          \
    }                                                    \
  } while (0)

int main(void) {
  const int32_t order[16] = {9, 3, 14, 0, 7, 11, 2, 5, 12, 1, 15, 6, 8, 13, 4, 10};
  pa_allocator* a = NULL;
  CHECK(1, pa_alloc_create(16, 4, order, &a) == PA_OK && a != NULL);
  CHECK(2, pa_alloc_num_free(a) == 16 && pa_alloc_block_size(a) == 4);

  int32_t s0 = -1, s1 = -1;
  CHECK(3, pa_alloc_seq_create(a, &s0) == PA_OK);
  int64_t slots[6];
  CHECK(4, pa_alloc_append_tokens(a, s0, 6, slots) == PA_OK);
  int32_t table[4], n = 0;
  CHECK(5, pa_alloc_block_table(a, s0, table, 4, &n) == PA_OK && n == 2);
  /* the free list is taken from the front: blocks 9 then 3 */
  CHECK(6, table[0] == 9 && table[1] == 3);
  for (int p = 0; p < 6; ++p) CHECK(7, slots[p] == (int64_t)table[p / 4] * 4 + p % 4);

  /* a fork shares both blocks; the child's next token lands in the shared,
     partly filled last block, so it is copied on write */
  CHECK(8, pa_alloc_fork(a, s0, &s1) == PA_OK);
  CHECK(9, pa_alloc_refcount(a, 9) == 2 && pa_alloc_refcount(a, 3) == 2);
  int64_t slot = -1;
  int32_t src = -1, dst = -1;
  CHECK(10, pa_alloc_append_slot(a, s1, &slot, &src, &dst) == PA_OK);
  CHECK(11, src == 3 && dst == 14 && slot == 14 * 4 + 2);
  CHECK(12, pa_alloc_refcount(a, 3) == 1 && pa_alloc_refcount(a, 14) == 1 && pa_alloc_refcount(a, 9) == 2);

  int32_t seqs[2] = {s0, s1}, tables[2 * 3], lens[2];
  CHECK(13, pa_alloc_export_tables(a, seqs, 2, tables, 3, lens, -1) == PA_OK);
  CHECK(14, lens[0] == 6 && lens[1] == 7);
  CHECK(15, tables[0] == 9 && tables[1] == 3 && tables[2] == -1);
  CHECK(16, tables[3] == 9 && tables[4] == 14 && tables[5] == -1);

  /* freeing returns blocks whose count reaches zero to the back of the list */
  CHECK(17, pa_alloc_free_seq(a, s0) == PA_OK);
  CHECK(18, pa_alloc_refcount(a, 3) == 0 && pa_alloc_refcount(a, 9) == 1);
  CHECK(19, pa_alloc_num_free(a) == 16 - 2);
  pa_alloc_destroy(a);

  /* SHA-256 of "abc" (FIPS 180-2, appendix B.1) */
  static const uint8_t want[32] = {0xba, 0x78, 0x16, 0xbf, 0x8f, 0x01, 0xcf, 0xea, 0x41, 0x41, 0x40,
                                   0xde, 0x5d, 0xae, 0x22, 0x23, 0xb0, 0x03, 0x61, 0xa3, 0x96, 0x17,
                                   0x7a, 0x9c, 0xb4, 0x10, 0xff, 0x61, 0xf2, 0x00, 0x15, 0xad};
  uint8_t got[32];
  CHECK(20, pa_sha256("abc", 3, got) == PA_OK && memcmp(got, want, 32) == 0);
  CHECK(21, strcmp(pa_status_string(PA_ERR_OOM), "PA_ERR_OOM") == 0);
  printf("ok\n");
  return 0;
}
