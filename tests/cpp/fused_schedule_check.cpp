// CPU check of the fused launch's schedule (zero_sharded_gb300/csrc/fused_schedule.h).
//
// Builds the seven tile lists of a shard the way the step program does (symmetric
// Gram and Poly tiles of 256 x 256, Update and Apply tiles over m x n), schedules
// them for a step count, and checks that
//   1. every (step, product, matrix) gets exactly its list's tiles, from the list of
//      the right X buffer, once;
//   2. replaying the units' sequences with random tile durations and hand-off
//      latencies never blocks for good: each unit runs its entries in order, and an
//      entry waits until its matrix's previous stage is complete.
// Usage: fused_schedule_check <units> <steps> <m>x<n>[,<m>x<n>...]   (m = min, n = max)
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <string>
#include <tuple>
#include <vector>

#include "fused_schedule.h"

using namespace cz;

int main(int argc, char** argv) {
  if (argc < 4) return 2;
  const int units = atoi(argv[1]), steps = atoi(argv[2]);
  std::vector<std::pair<int, int>> mats;
  for (std::string s = argv[3]; !s.empty();) {
    const size_t c = s.find(','), x = s.find('x');
    mats.push_back({atoi(s.substr(0, x).c_str()), atoi(s.substr(x + 1, c - x - 1).c_str())});
    s = c == std::string::npos ? "" : s.substr(c + 1);
  }
  const int n_mats = (int)mats.size();
  // one problem per matrix in every list; list li's problems are numbered from li * n_mats
  std::vector<SchedTile> lists[kSchedLists];
  std::vector<int64_t> kb_of((size_t)kSchedLists * n_mats, 0);   // k-blocks of each problem's tiles
  for (int gm = 0; gm < n_mats; ++gm) {
    const int m = mats[gm].first, n = mats[gm].second;
    const int T = (m + 255) / 256, TN = (n + 255) / 256;
    for (int li = 0; li < kSchedLists; ++li) {
      const int prob = li * n_mats + gm;
      const int64_t kb = li < 2 ? (n + 63) / 64 : (m + 63) / 64;   // Gram: K = n; Poly, Update: K = m
      kb_of[(size_t)prob] = kb;
      if (li <= 2) {
        for (int a = 0; a < T; ++a)
          for (int b = a; b < T; ++b) lists[li].push_back({prob, 0, a, b, gm, kb});
      } else {
        for (int b = 0; b < TN; ++b)
          for (int a = 0; a < T; ++a) lists[li].push_back({prob, 0, a, b, gm, kb});
      }
    }
  }
  std::vector<int> count[kSchedLists];
  for (int li = 0; li < kSchedLists; ++li) {
    count[li].assign(n_mats, 0);
    for (const SchedTile& t : lists[li]) count[li][t.gm]++;
  }
  std::vector<std::vector<SchedEntry>> per_unit;
  if (!schedule_fused(lists, steps, units, n_mats, per_unit)) {
    printf("schedule failed\n");
    return 1;
  }
  // 1. coverage
  std::map<std::tuple<int, int, int>, int> seen;
  size_t total = 0;
  for (const auto& v : per_unit)
    for (const SchedEntry& e : v) {
      const int prob = e.x & 0xFF, t = e.x >> 8, li = prob / n_mats, gm = prob % n_mats;
      const int slot = li < 2 ? 0 : li == 2 ? 1 : 2;
      if (t < 0 || t >= steps || li != sched_list_of(t, slot, steps)) {
        printf("entry from the wrong list: step %d list %d\n", t, li);
        return 1;
      }
      seen[{t, slot, gm}]++;
      ++total;
    }
  size_t expect = 0;
  for (int t = 0; t < steps; ++t)
    for (int slot = 0; slot < 3; ++slot)
      for (int gm = 0; gm < n_mats; ++gm) {
        const int want = count[sched_list_of(t, slot, steps)][gm];
        expect += want;
        if (seen[{t, slot, gm}] != want) {
          printf("step %d product %d matrix %d: %d tiles, want %d\n", t, slot, gm, seen[{t, slot, gm}], want);
          return 1;
        }
      }
  if (total != expect) return 1;
  // 2. replays with random durations and hand-offs
  std::mt19937 rng(7);
  const int trials = total > 10000 ? 40 : 200;
  for (int trial = 0; trial < trials; ++trial) {
    std::uniform_real_distribution<double> jit(0.5, 2.0), hand(0.0, 80.0);
    std::vector<size_t> pos((size_t)units, 0);
    std::vector<double> tfree((size_t)units, 0.0);
    std::map<std::tuple<int, int, int>, int> done;
    std::map<std::tuple<int, int, int>, double> fin, lastend;
    for (size_t left = total; left > 0; --left) {
      int best = -1;
      double bstart = 0;
      for (int u = 0; u < units; ++u) {
        if (pos[u] >= per_unit[u].size()) continue;
        const SchedEntry& e = per_unit[u][pos[u]];
        const int prob = e.x & 0xFF, t = e.x >> 8, li = prob / n_mats, gm = prob % n_mats;
        const int slot = li < 2 ? 0 : li == 2 ? 1 : 2;
        double ready = 0;
        if (t > 0 || slot > 0) {
          const auto dep = slot == 0 ? std::make_tuple(t - 1, 2, gm) : std::make_tuple(t, slot - 1, gm);
          const auto it = fin.find(dep);
          if (it == fin.end()) continue;
          ready = it->second;
        }
        const double st = std::max(tfree[u], ready);
        if (best < 0 || st < bstart) {
          best = u;
          bstart = st;
        }
      }
      if (best < 0) {
        printf("replay %d: every unit waits for good (%zu entries left)\n", trial, left);
        return 1;
      }
      const SchedEntry& e = per_unit[best][pos[best]++];
      const int prob = e.x & 0xFF, t = e.x >> 8, li = prob / n_mats, gm = prob % n_mats;
      const int slot = li < 2 ? 0 : li == 2 ? 1 : 2;
      const double end = bstart + (double)(kb_of[(size_t)prob] + kSchedTileOverhead) * jit(rng);
      tfree[best] = end;
      const auto key = std::make_tuple(t, slot, gm);
      lastend[key] = std::max(lastend[key], end);
      if (++done[key] == count[li][gm]) fin[key] = lastend[key] + hand(rng);
    }
  }
  size_t lo = SIZE_MAX, hi = 0;
  for (const auto& v : per_unit) {
    lo = std::min(lo, v.size());
    hi = std::max(hi, v.size());
  }
  printf("ok: %zu entries over %d units (%zu..%zu each), %d replays\n", total, units, lo, hi, trials);
  return 0;
}
