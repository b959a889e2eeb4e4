// Balance-aware owner planner and MatrixShard table.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: each 2D weight is owned whole by one data-parallel rank
// (the others hold empty shards), non-matrix tensors are packed into tail
// owners, and a balance-aware owner planner produces the MatrixShard metadata.
// The pages give no algorithm; this is longest-processing-time-first on the
// dense Newton-Schulz FLOP count, with a tail pass that fills the ranks with
// the least Newton-Schulz work first, and a deterministic layout in
// declaration order.  Integer arithmetic only, so every rank that runs it gets
// the same plan.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "mfsdp.h"

namespace {

// cost = T * (4 s^2 l + 2 s^3); false on uint64 overflow.
bool ns_cost(int64_t rows, int64_t cols, int32_t steps, uint64_t* out) {
  const unsigned __int128 s = (unsigned __int128)std::min(rows, cols);
  const unsigned __int128 l = (unsigned __int128)std::max(rows, cols);
  const unsigned __int128 c = (unsigned __int128)steps * (4 * s * s * l + 2 * s * s * s);
  if (c > (unsigned __int128)UINT64_MAX) return false;
  *out = (uint64_t)c;
  return true;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Rank with the lexicographically smallest (primary[r], secondary[r], r).
int argmin_rank(const std::vector<uint64_t>& primary, const std::vector<uint64_t>* secondary) {
  int best = 0;
  for (int r = 1; r < (int)primary.size(); ++r) {
    if (primary[r] < primary[best]) {
      best = r;
    } else if (primary[r] == primary[best] && secondary && (*secondary)[r] < (*secondary)[best]) {
      best = r;
    }
  }
  return best;
}

}  // namespace

extern "C" int mfsdp_plan_owners(const mfsdp_param* params, int32_t n_params, int32_t world,
                                 int32_t ns_steps, int64_t align_elems,
                                 mfsdp_matrix_shard* out_m, int32_t* n_m,
                                 mfsdp_tail_shard* out_t, int32_t* n_t,
                                 int64_t* rank_matrix_elems, int64_t* rank_tail_elems) {
  if (n_params < 0 || world < 1 || ns_steps < 0 || align_elems < 1) return MFSDP_ERR_INVALID_ARG;
  if (n_params > 0 && !params) return MFSDP_ERR_INVALID_ARG;
  if (!n_m || !n_t) return MFSDP_ERR_INVALID_ARG;

  std::vector<int> mats, tails;
  std::vector<uint64_t> cost(n_params, 0);
  for (int i = 0; i < n_params; ++i) {
    const mfsdp_param& p = params[i];
    if (p.kind != MFSDP_KIND_MATRIX && p.kind != MFSDP_KIND_TAIL) return MFSDP_ERR_INVALID_ARG;
    if (p.rows < 1 || p.cols < 1) return MFSDP_ERR_UNSUPPORTED_SHAPE;
    if (p.rows > (INT64_MAX / p.cols)) return MFSDP_ERR_UNSUPPORTED_SHAPE;
    if (p.kind == MFSDP_KIND_MATRIX) {
      if (!ns_cost(p.rows, p.cols, ns_steps, &cost[i])) return MFSDP_ERR_UNSUPPORTED_SHAPE;
      mats.push_back(i);
    } else {
      tails.push_back(i);
    }
  }
  if ((!mats.empty() && !out_m) || (!tails.empty() && !out_t)) return MFSDP_ERR_INVALID_ARG;

  // Matrix pass: longest processing time first.
  std::vector<int> order = mats;
  std::sort(order.begin(), order.end(), [&](int x, int y) {
    return cost[x] != cost[y] ? cost[x] > cost[y] : x < y;
  });
  std::vector<uint64_t> load(world, 0);
  std::vector<int> owner(n_params, -1);
  for (int i : order) {
    const int r = argmin_rank(load, nullptr);
    owner[i] = r;
    load[r] += cost[i];
  }

  // Tail pass: largest tensors first, to the rank with the least tail, then the
  // least Newton-Schulz work.
  auto numel = [&](int i) { return (uint64_t)(params[i].rows * params[i].cols); };
  order = tails;
  std::sort(order.begin(), order.end(), [&](int x, int y) {
    return numel(x) != numel(y) ? numel(x) > numel(y) : x < y;
  });
  std::vector<uint64_t> tload(world, 0);
  for (int i : order) {
    const int r = argmin_rank(tload, &load);
    owner[i] = r;
    tload[r] += numel(i);
  }

  // Layout: per rank, ascending param id (mats/tails are already ascending).
  int cm = 0, ct = 0;
  for (int r = 0; r < world; ++r) {
    int64_t off = 0;
    for (int i : mats) {
      if (owner[i] != r) continue;
      off = round_up(off, align_elems);
      mfsdp_matrix_shard& s = out_m[cm++];
      std::memset(&s, 0, sizeof(s));
      s.param_id = i;
      s.owner = r;
      s.offset = off;
      s.rows = params[i].rows;
      s.cols = params[i].cols;
      s.transposed = params[i].rows > params[i].cols ? 1 : 0;
      s.cost = cost[i];
      off += params[i].rows * params[i].cols;
    }
    if (rank_matrix_elems) rank_matrix_elems[r] = round_up(off, align_elems);
    off = 0;
    for (int i : tails) {
      if (owner[i] != r) continue;
      off = round_up(off, align_elems);
      mfsdp_tail_shard& s = out_t[ct++];
      std::memset(&s, 0, sizeof(s));
      s.param_id = i;
      s.owner = r;
      s.offset = off;
      s.numel = (int64_t)numel(i);
      off += (int64_t)numel(i);
    }
    if (rank_tail_elems) rank_tail_elems[r] = round_up(off, align_elems);
  }
  *n_m = cm;
  *n_t = ct;
  return MFSDP_OK;
}
