// TP Micro-Group planner behind cz_plan_microgroups.
//
// Canzona summary page (paper-graph-ui), section 3.4, "The TP Hierarchical
// Partitioning and Scheduling (Micro-Group Construction)": a deterministic
// global LPT sort by (W(p), ID) descending, greedy packing of tensors into the
// current candidate group, each candidate simulated by the MinHeapSolver (LPT
// over R host ranks with a min-heap of (load, rank)), and a rollback that
// finalises the group when the simulated makespan would exceed C_max.  All
// arithmetic is on int64 costs, so the result is exact and identical on every
// rank that runs it.

#include <algorithm>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "cz.h"

namespace {

// Makespan L_max of the LPT assignment of `items` (parameter ids) to R ranks;
// optionally records each item's rank.  Items are taken by (cost, id) descending;
// equal loads go to the smaller rank index.
int64_t min_heap_solver(std::vector<int64_t>& items, const int64_t* costs, int32_t R, int32_t* host) {
  std::sort(items.begin(), items.end(), [&](int64_t a, int64_t b) {
    if (costs[a] != costs[b]) return costs[a] > costs[b];
    return a > b;
  });
  using Slot = std::pair<int64_t, int32_t>;   // (load, rank)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> pq;
  for (int32_t r = 0; r < R; ++r) pq.push({0, r});
  for (int64_t p : items) {
    Slot s = pq.top();
    pq.pop();
    if (host) host[p] = s.second;
    pq.push({s.first + costs[p], s.second});
  }
  int64_t l_max = 0;
  while (!pq.empty()) {
    l_max = std::max(l_max, pq.top().first);
    pq.pop();
  }
  return l_max;
}

}  // namespace

extern "C" int cz_plan_microgroups(const int64_t* costs, int64_t n_params, int32_t R, int64_t c_max,
                                   int32_t* group_out, int32_t* host_out, int64_t* n_groups_out) {
  if (!costs || n_params <= 0 || R < 1 || c_max <= 0 || !group_out || !host_out || !n_groups_out)
    return CZ_ERR_INVALID;
  for (int64_t i = 0; i < n_params; ++i)
    if (costs[i] <= 0) return CZ_ERR_INVALID;
  std::vector<int64_t> order(n_params);
  for (int64_t i = 0; i < n_params; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    if (costs[a] != costs[b]) return costs[a] > costs[b];
    return a > b;
  });
  std::vector<std::vector<int64_t>> groups;
  std::vector<int64_t> curr, test;
  for (int64_t p : order) {
    if (curr.empty()) {
      curr.push_back(p);
      continue;
    }
    test = curr;
    test.push_back(p);
    if (min_heap_solver(test, costs, R, nullptr) <= c_max) {
      curr.push_back(p);
    } else {
      groups.push_back(curr);   // rollback: finalise without p; p seeds the next group
      curr.assign(1, p);
    }
  }
  if (!curr.empty()) groups.push_back(curr);
  for (size_t g = 0; g < groups.size(); ++g) {
    min_heap_solver(groups[g], costs, R, host_out);
    for (int64_t p : groups[g]) group_out[p] = (int32_t)g;
  }
  *n_groups_out = (int64_t)groups.size();
  return CZ_OK;
}
