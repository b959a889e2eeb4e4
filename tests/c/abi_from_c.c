/* The C ABI used from plain C99: only include/mfsdp.h and the shared library.
 * Host-only calls (planner, sizes, strings, argument checks, an owner-shard
 * checkpoint written to argv[1] and read back), so it runs without a GPU.
 * Prints "ok" and returns 0, or names the first failed check. */
#include <stdio.h>
#include <string.h>

#include "mfsdp.h"

#define CHECK(cond)                                          \
  do {                                                       \
    if (!(cond)) {                                           \
      printf("failed: %s (line %d)\n", #cond, __LINE__);     \
      return 1;                                              \
    }                                                        \
  } while (0)

int main(int argc, char** argv) {
  /* a 4096-wide block: two square matrices, a tall and a wide one, two vectors */
  const mfsdp_param params[6] = {
      {4096, 1, MFSDP_KIND_TAIL, 0},    {4096, 4096, MFSDP_KIND_MATRIX, 0}, {14336, 4096, MFSDP_KIND_MATRIX, 0},
      {4096, 14336, MFSDP_KIND_MATRIX, 0}, {4096, 4096, MFSDP_KIND_MATRIX, 0}, {4096, 1, MFSDP_KIND_TAIL, 0}};
  mfsdp_matrix_shard m[4];
  mfsdp_tail_shard t[2];
  int32_t n_m = 0, n_t = 0;
  int64_t mat_elems[2], tail_elems[2];
  CHECK(mfsdp_plan_owners(params, 6, 2, 5, 128, m, &n_m, t, &n_t, mat_elems, tail_elems) == MFSDP_OK);
  CHECK(n_m == 4 && n_t == 2);
  for (int i = 0; i < n_m; ++i) {
    CHECK(m[i].offset % 128 == 0);
    CHECK(m[i].transposed == (m[i].rows > m[i].cols));
    CHECK(m[i].offset + m[i].rows * m[i].cols <= mat_elems[m[i].owner]);
  }
  /* LPT: the two equal-cost 14336-long matrices go to ranks 0 and 1, then the two
   * 4096^2 ones to ranks 0 and 1 again (ties to the lower rank id) */
  int per_rank[2] = {0, 0};
  for (int i = 0; i < n_m; ++i) per_rank[m[i].owner] += 1;
  CHECK(per_rank[0] == 2 && per_rank[1] == 2);
  CHECK(mfsdp_plan_owners(params, 6, 0, 5, 128, m, &n_m, t, &n_t, mat_elems, tail_elems) == MFSDP_ERR_INVALID_ARG);

  /* rank 0's matrices: contiguous in the planner's (owner, offset) order */
  int first = 0, count = 0;
  while (first < n_m && m[first].owner != 0) ++first;
  while (first + count < n_m && m[first + count].owner == 0) ++count;
  CHECK(count > 0);
  CHECK(mfsdp_muon_workspace_bytes(m + first, count) > 0);
  uint64_t dense = 0, executed = 0;
  CHECK(mfsdp_muon_step_flops(m + first, count, 5, &dense, &executed) == MFSDP_OK);
  CHECK(dense > 0 && executed > 0);
  CHECK(mfsdp_host_step_groups(m + first, count, MFSDP_DTYPE_BF16, MFSDP_DTYPE_BF16, 0, NULL) >= 1);

  /* argument checks happen on the host, before anything touches a device */
  CHECK(mfsdp_muon_owner_step(m + first, count, NULL, MFSDP_DTYPE_BF16, NULL, NULL, MFSDP_DTYPE_BF16,
                              mat_elems[0], 0.95, 0, 5, 3.4445, -4.7750, 2.0315, 1e-7, NULL, 0, NULL) ==
        MFSDP_ERR_INVALID_ARG);
  CHECK(mfsdp_adamw_tail_step(NULL, NULL, NULL, NULL, 16, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, NULL) ==
        MFSDP_ERR_INVALID_ARG);

  /* an owner-shard checkpoint of a small plan's rank 1: its shards, momentum and tail */
  if (argc > 1) {
    const mfsdp_param small[4] = {{64, 96, MFSDP_KIND_MATRIX, 0}, {40, 1, MFSDP_KIND_TAIL, 0},
                                  {40, 40, MFSDP_KIND_MATRIX, 0}, {96, 64, MFSDP_KIND_MATRIX, 0}};
    mfsdp_matrix_shard sm[3], back[3];
    mfsdp_tail_shard st[1], tback[1];
    int32_t nm = 0, nt = 0;
    int64_t me[2], te[2];
    CHECK(mfsdp_plan_owners(small, 4, 2, 5, 128, sm, &nm, st, &nt, me, te) == MFSDP_OK);
    int f = 0, c = 0, ft = 0, ct = 0;
    while (f < nm && sm[f].owner != 1) ++f;
    while (f + c < nm && sm[f + c].owner == 1) ++c;
    while (ft < nt && st[ft].owner != 1) ++ft;
    while (ft + ct < nt && st[ft + ct].owner == 1) ++ct;
    static float mom[8192], mom2[8192], tp[256], tm[256], tv[256], tp2[256], tm2[256], tv2[256];
    CHECK(me[1] <= 8192 && te[1] <= 256 && c >= 1);
    for (int i = 0; i < 8192; ++i) mom[i] = (float)i * 0.5f - 7.0f;
    for (int i = 0; i < 256; ++i) { tp[i] = (float)i; tm[i] = -(float)i; tv[i] = 0.25f * (float)i; }
    mfsdp_checkpoint_header h;
    memset(&h, 0, sizeof h);
    h.world = 2; h.rank = 1; h.ns_steps = 5; h.n_matrix = c; h.n_tail = ct;
    h.align_elems = 128; h.matrix_elems = me[1]; h.tail_elems = te[1]; h.adam_step = 3;
    CHECK(mfsdp_checkpoint_write(argv[1], &h, sm + f, st + ft, mom, tp, tm, tv) == MFSDP_OK);
    mfsdp_checkpoint_header r;
    CHECK(mfsdp_checkpoint_read_header(argv[1], &r) == MFSDP_OK);
    CHECK(r.world == 2 && r.rank == 1 && r.n_matrix == c && r.matrix_elems == me[1] && r.adam_step == 3);
    CHECK(mfsdp_checkpoint_bytes(&r) == 64 + 48 * (size_t)c + 24 * (size_t)ct + 4 * (size_t)(me[1] + 3 * te[1]) + 8);
    CHECK(mfsdp_checkpoint_read(argv[1], &r, back, 3, tback, 1, mom2, 8192, tp2, tm2, tv2, 256) == MFSDP_OK);
    CHECK(memcmp(back, sm + f, (size_t)c * sizeof(mfsdp_matrix_shard)) == 0);
    CHECK(ct == 0 || memcmp(tback, st + ft, (size_t)ct * sizeof(mfsdp_tail_shard)) == 0);
    CHECK(memcmp(mom, mom2, (size_t)me[1] * sizeof(float)) == 0);
    CHECK(memcmp(tv, tv2, (size_t)te[1] * sizeof(float)) == 0);
    CHECK(mfsdp_checkpoint_read(argv[1], &r, back, c - 1, tback, 1, mom2, 8192, tp2, tm2, tv2, 256) ==
          MFSDP_ERR_WORKSPACE_TOO_SMALL);
  }

  const char* s = mfsdp_status_string(MFSDP_ERR_WORKSPACE_TOO_SMALL);
  CHECK(s != NULL && strlen(s) > 0);
  const char* v = mfsdp_version();
  CHECK(v != NULL && strchr(v, '.') != NULL);
  printf("ok %s\n", v);
  return 0;
}
