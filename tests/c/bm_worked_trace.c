/* The worked allocation trace of "PagedAttention, simply explained" ("How PagedAttention
 * solves it": 100 frames of 10 token slots, free list 0..99, prompts A:8 B:5 C:12 D:9,
 * then three decode steps) driven through the C ABI from plain C99.  Prints, one line
 * each: every step's slots, every sequence's final table and length, the head of the
 * free list, and the pool's memory accounting. */
#include <stdint.h>
#include <stdio.h>

#include "pa.h"

#define CHECK(x)                                                  \
  do {                                                            \
    int rc_ = (x);                                                \
    if (rc_ < 0) {                                                \
      printf("error %d (%s) at %s\n", rc_, pa_strerror(rc_), #x); \
      return 1;                                                   \
    }                                                             \
  } while (0)

int main(void) {
  pa_bm* bm = NULL;
  const int32_t prompts[4] = {8, 5, 12, 9};
  int32_t slots[16];
  int64_t ids[4] = {0, 1, 2, 3};
  int32_t copies[8];
  int32_t n_copies = 0;
  int32_t table[4];
  int32_t n = 0, len = 0, nb = 0, free_list[100];
  pa_bm_usage_t u;
  int s, i, step;

  CHECK(pa_bm_create(100, 10, NULL, &bm));
  for (s = 0; s < 4; ++s) CHECK(pa_bm_add_seq(bm, ids[s], prompts[s], slots));
  for (step = 0; step < 3; ++step) {
    CHECK(pa_bm_step(bm, ids, 4, slots, copies, &n_copies));
    printf("step %d slots", step + 1);
    for (i = 0; i < 4; ++i) printf(" %d", (int)slots[i]);
    printf(" copies %d\n", (int)n_copies);
  }
  for (s = 0; s < 4; ++s) {
    CHECK(pa_bm_table(bm, ids[s], table, 4, &n));
    CHECK(pa_bm_seq_info(bm, ids[s], &len, &nb));
    printf("seq %d len %d table", s, (int)len);
    for (i = 0; i < n; ++i) printf(" %d", (int)table[i]);
    printf("\n");
  }
  if (pa_bm_free_list(bm, free_list, 3, &n) != PA_ERR_CAPACITY) return 2; /* too small a buffer */
  CHECK(pa_bm_free_list(bm, free_list, 100, &n));
  printf("free %d head %d %d %d last %d\n", (int)n, (int)free_list[0], (int)free_list[1], (int)free_list[2],
         (int)free_list[n - 1]);
  CHECK(pa_bm_usage(bm, &u));
  printf("usage %lld %lld %lld %lld %lld\n", (long long)u.frames_in_use, (long long)u.slots_filled,
         (long long)u.tokens_logical, (long long)u.table_entries, (long long)u.max_seq_waste);
  pa_bm_destroy(bm);
  return 0;
}
