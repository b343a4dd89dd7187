/* A plain C99 consumer of include/oomb.h: the header is valid C, and the calls
 * below exercise only host-side paths of liboomb.so (argument checks, the page
 * allocator, status strings), so the program runs on a machine without a GPU.
 * The pool's buffer pointers are placeholders that no call dereferences.
 * Exit status 0 = every check held; otherwise the number of the failed check. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "oomb.h"

#define CHECK(id, cond)                                        \
  do {                                                         \
    if (!(cond)) {                                             \
      fprintf(stderr, "check %d failed: %s\n", (id), #cond);   \
      return (id);                                             \
    }                                                          \
  } while (0)

static void* fake(uintptr_t i) { return (void*)(uintptr_t)((i + 1) << 20); }

int main(void) {
  oomb_pool_desc d;
  oomb_pool* pool = NULL;
  int32_t order[4] = {2, 0, 3, 1};
  int32_t table[8];
  memset(&d, 0, sizeof(d));
  d.n_q_heads = 28;
  d.n_kv_heads = 4;
  d.head_dim = 128;
  d.page_size = 128;
  d.num_phys_pages = 4;
  d.max_logical_pages = 8;
  d.dtype = OOMB_BF16;
  d.k_pool = fake(0);
  d.v_pool = fake(1);
  d.dk_pool = (float*)fake(2);
  d.dv_pool = (float*)fake(3);
  d.summary = (float*)fake(4);
  d.page_table = (int32_t*)fake(5);
  d.error_word = (uint32_t*)fake(6);
  d.page_order = order;

  CHECK(1, strcmp(oomb_status_str(OOMB_ERR_OUT_OF_PAGES), "out of pages") == 0);
  d.n_kv_heads = 3; /* 28 query heads do not split into 3 groups */
  CHECK(2, oomb_pool_create(&d, &pool) == OOMB_ERR_ARG && pool == NULL);
  d.n_kv_heads = 4;
  CHECK(3, oomb_pool_create(&d, &pool) == OOMB_OK && pool != NULL);
  CHECK(4, oomb_pool_free_pages(pool) == 4 && oomb_pool_tokens(pool) == 0);
  CHECK(5, oomb_uses_tensor_cores(pool) == 1);
  /* refused before any device work */
  CHECK(6, oomb_kv_append(pool, fake(9), fake(9), 64, 128, NULL) == OOMB_ERR_ARG);      /* not at the end */
  CHECK(7, oomb_kv_append(pool, fake(9), fake(9), 0, 5 * 128, NULL) == OOMB_ERR_OUT_OF_PAGES);
  CHECK(8, oomb_page_free(pool, 0, 1, NULL) == OOMB_ERR_ARG);                          /* nothing appended */
  CHECK(9, oomb_window_select(pool, 0, 128, -1, 1, (int32_t*)fake(9), (int32_t*)fake(9), 8, NULL) == OOMB_ERR_ARG);
  CHECK(10, oomb_prefetch(pool, (int32_t*)fake(9), (int32_t*)fake(9), 8, 0, NULL) == OOMB_ERR_UNSUPPORTED);
  CHECK(11, oomb_workspace_size(pool, OOMB_OP_SELECT, 4096) > 0);
  CHECK(12, oomb_workspace_size(pool, OOMB_OP_BWD, 4096) >= (size_t)28 * 4096 * 4);
  CHECK(13, oomb_page_table_host(pool, table, 8) == 8);
  for (int i = 0; i < 8; ++i) CHECK(14, table[i] == -1);
  oomb_pool_destroy(pool);
  printf("c abi host checks: ok\n");
  return 0;
}
