// Dependency-aware order of the fused Newton-Schulz launch's tiles: list scheduling
// on a model of the launch.  Host code only, no CUDA types (the CPU tests compile it
// on its own).
//
// The launch runs, per matrix, a chain of stages: Gram, Poly, Update of step 1, of
// step 2, and so on, the last Update being the apply.  A tile may start once every
// tile of its matrix's previous stage has finished and the hand-off (store
// completion, counter release, poll, first operand load) is over.  Walking fixed
// per-(step, product) lists, a unit stops at a tile whose matrix is not ready
// although later tiles of other matrices are.  Here a model of the units (a tile
// takes its k-blocks plus kSchedTileOverhead; a hand-off takes kSchedHandoff
// k-blocks) assigns tiles as units free up: ready tiles first, by the longest
// remaining chain of stages of their matrix (critical path), then the most
// k-blocks, then the lower matrix index, then list order.  Each unit's sequence is
// in model time order, and every tile's dependencies finish before it starts in the
// model, so the real launch cannot wait in a cycle: the earliest blocked tile's
// dependencies are always running or queued behind tiles that are not blocked.
#pragma once

#include <stdint.h>

#include <algorithm>
#include <functional>
#include <queue>
#include <tuple>
#include <utility>
#include <vector>

namespace cz {

constexpr int64_t kSchedTileOverhead = 2;   // k-blocks: tile start and accumulator hand-off
constexpr int64_t kSchedHandoff = 36;       // k-blocks: stage hand-off (about 12 us at 2 GHz)
constexpr int kSchedLists = 7;              // Gram (X buffer 0, 1), Poly, Update (0, 1), Apply (0, 1)

// One tile of one of the seven lists: the entry the kernel walks (problem index in
// the launch's table, matrix within the problem, tile row, tile column), its global
// matrix and its k-blocks.
struct SchedTile {
  int32_t prob, mat, tile_m, tile_n;
  int32_t gm;
  int64_t kb;
};

// An entry of a unit's sequence: {problem | step << 8, matrix, tile_m, tile_n}.
struct SchedEntry {
  int32_t x, y, z, w;
};

// The list a (step, product) takes its tiles from: Gram of X buffer t & 1, Poly,
// Update of X buffer t & 1, or the Apply in the last step.
inline int sched_list_of(int t, int slot, int steps) {
  return slot == 0 ? (t & 1) : slot == 1 ? 2 : (t + 1 == steps ? 5 : 3) + (t & 1);
}

// lists[li]: the tiles of list li (every matrix of every list has at least one
// tile); n_mats global matrices; per_unit receives each unit's sequence.  Returns
// false (the caller then walks the lists) if the model ever had no tile to start
// and no stage to wait for, which the stage chains rule out.
inline bool schedule_fused(const std::vector<SchedTile> lists[kSchedLists], int steps, int units, int n_mats,
                           std::vector<std::vector<SchedEntry>>& per_unit) {
  std::vector<std::vector<std::vector<const SchedTile*>>> by(kSchedLists,
                                                             std::vector<std::vector<const SchedTile*>>(n_mats));
  std::vector<int64_t> maxkb((size_t)n_mats * 3, 0);
  for (int li = 0; li < kSchedLists; ++li) {
    const int slot = li < 2 ? 0 : li == 2 ? 1 : 2;
    for (const SchedTile& t : lists[li]) {
      if (t.gm < 0 || t.gm >= n_mats) return false;
      by[li][t.gm].push_back(&t);
      maxkb[(size_t)t.gm * 3 + slot] = std::max(maxkb[(size_t)t.gm * 3 + slot], t.kb);
    }
  }
  const int64_t n_stages = (int64_t)steps * 3;
  auto rem = [&](int32_t gm, int64_t stage) {   // model time from this stage's start to the chain's end
    int64_t r = 0;
    for (int64_t q = stage; q < n_stages; ++q) r += maxkb[(size_t)gm * 3 + q % 3] + kSchedTileOverhead + kSchedHandoff;
    return r;
  };
  std::vector<int64_t> left((size_t)n_mats * n_stages, 0), last((size_t)n_mats * n_stages, 0);
  for (int32_t gm = 0; gm < n_mats; ++gm)
    for (int64_t q = 0; q < n_stages; ++q)
      left[(size_t)gm * n_stages + q] = (int64_t)by[sched_list_of((int)(q / 3), (int)(q % 3), steps)][gm].size();
  struct Ready {
    int64_t prio, kb;
    int32_t gm;
    int64_t seq, stage;
    SchedEntry e;
  };
  auto rless = [](const Ready& a, const Ready& b) {   // largest first: priority, k-blocks, -matrix, -sequence
    if (a.prio != b.prio) return a.prio < b.prio;
    if (a.kb != b.kb) return a.kb < b.kb;
    if (a.gm != b.gm) return a.gm > b.gm;
    return a.seq > b.seq;
  };
  std::priority_queue<Ready, std::vector<Ready>, decltype(rless)> ready(rless);
  using Rel = std::tuple<int64_t, int32_t, int64_t>;   // (time, matrix, stage)
  std::priority_queue<Rel, std::vector<Rel>, std::greater<Rel>> release;
  using Unit = std::pair<int64_t, int>;                // (free time, unit)
  std::priority_queue<Unit, std::vector<Unit>, std::greater<Unit>> free_units;
  for (int32_t gm = 0; gm < n_mats; ++gm)
    if (left[(size_t)gm * n_stages] > 0) release.emplace(0, gm, 0);
  for (int u = 0; u < units; ++u) free_units.emplace(0, u);
  per_unit.assign((size_t)units, {});
  int64_t seq = 0, todo = 0;
  for (int64_t x : left) todo += x;
  while (todo > 0) {
    const Unit fu = free_units.top();
    free_units.pop();
    const int64_t tf = fu.first;
    const int u = fu.second;
    while (!release.empty() && std::get<0>(release.top()) <= tf) {
      const Rel rl = release.top();
      release.pop();
      const int32_t gm = std::get<1>(rl);
      const int64_t q = std::get<2>(rl);
      const int t = (int)(q / 3);
      const int64_t pr = rem(gm, q);
      for (const SchedTile* it : by[sched_list_of(t, (int)(q % 3), steps)][gm])
        ready.push({pr, it->kb, gm, seq++, q, SchedEntry{it->prob | (t << 8), it->mat, it->tile_m, it->tile_n}});
    }
    if (ready.empty()) {        // nothing can start before the next stage is released
      if (release.empty()) return false;
      free_units.emplace(std::get<0>(release.top()), u);
      continue;
    }
    const Ready r = ready.top();
    ready.pop();
    per_unit[(size_t)u].push_back(r.e);
    const int64_t end = tf + r.kb + kSchedTileOverhead;
    const size_t k = (size_t)r.gm * n_stages + r.stage;
    last[k] = std::max(last[k], end);
    if (--left[k] == 0 && r.stage + 1 < n_stages)   // the matrix's next stage (every stage has tiles)
      release.emplace(last[k] + kSchedHandoff, r.gm, r.stage + 1);
    --todo;
    free_units.emplace(end, u);
  }
  return true;
}

}  // namespace cz
