/* The boundary used from plain C: plan rejects (checked before any CUDA call) and the host page
 * allocator, linked against libpg.so with no Python or torch involved. Exit status 0 = pass. */
#include <stdint.h>
#include <stdio.h>

#include "pg.h"
#include "pg_kv.h"

int main(void) {
  pg_plan_t plan = NULL;
  int64_t qo[2] = {0, 4}, kvp[2] = {0, 1}, start[1] = {0};
  int32_t pages[1] = {0}, last[1] = {5};
  /* one page holding 5 positions for a 4-token step at position 0: coverage fails */
  int rc = pg_plan_paged_prefill(&plan, 1, qo, kvp, pages, last, start, 16, 8, 256, 16, NULL);
  if (rc != PG_ERR_COVERAGE || plan != NULL) return 1;
  rc = pg_plan_paged_prefill(&plan, 1, qo, kvp, pages, last, start, 16, 0, 256, 16, NULL);
  if (rc != PG_ERR_ZERO_KV_HEADS || plan != NULL) return 2;
  if (pg_status_string(PG_ERR_COVERAGE) == NULL) return 3;
  pg_plan_destroy(NULL); /* a no-op */

  pg_kv_server_t srv = NULL;
  if (pg_kv_server_create(&srv, 4, 4, 16, 100, 1, 1024) != PG_KV_OK) return 4;
  int64_t rid = 0;
  if (pg_kv_request_open(srv, &rid) != PG_KV_OK || rid <= 0) return 5;
  if (pg_kv_admit_step(srv, rid, 20) != PG_KV_OK) return 6;
  int32_t frontier = 0, nl = 0, ng = 0, nfree = 0;
  if (pg_kv_request_info(srv, rid, &frontier, &nl, &ng) != PG_KV_OK) return 7;
  if (frontier != 0 || nl != 2 || ng != 2) return 8;  /* reserved, not committed */
  if (pg_kv_abort_step(srv, rid) != PG_KV_OK) return 12;
  if (pg_kv_free_pages(srv, PG_KV_LOCAL, &nfree) != PG_KV_OK || nfree != 4) return 13;
  if (pg_kv_admit_step(srv, rid, 20) != PG_KV_OK || pg_kv_commit_step(srv, rid) != PG_KV_OK) return 14;
  if (pg_kv_request_info(srv, rid, &frontier, &nl, &ng) != PG_KV_OK) return 15;
  if (frontier != 20 || nl != 2 || ng != 2) return 16;
  if (pg_kv_admit_step(srv, rid, 100) != PG_KV_ERR_WINDOW) return 9; /* fails closed */
  if (pg_kv_request_close(srv, rid) != PG_KV_OK) return 10;
  if (pg_kv_free_pages(srv, PG_KV_LOCAL, &nfree) != PG_KV_OK || nfree != 4) return 11;
  pg_kv_server_destroy(srv);
  printf("c abi ok\n");
  return 0;
}
