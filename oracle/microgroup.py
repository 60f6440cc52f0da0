"""Oracle for the TP Micro-Group planner (test infrastructure only; see package header).

Written from the summary page "Canzona: A Unified, Asynchronous, and
Load-Balanced Framework for Distributed Matrix-based Optimizers"
(paper-graph-ui), section 3.4, "The TP Hierarchical Partitioning and
Scheduling (Micro-Group Construction)":

* Phase 1, deterministic global LPT sort of all parameters by the key
  (W(p), ID_p), descending.
* Phase 2, greedy packing with rollback: add the next tensor to the current
  candidate group, simulate the group with the MinHeapSolver, accept when the
  simulated makespan L_max <= C_max, otherwise finalise the current group and
  start the next one with this tensor.
* MinHeapSolver (the page's "Algorithm 4"): sort the group's items by cost,
  descending (a local sort), then give each item to the least-loaded rank from a
  min-heap of (load, rank) pairs initialised with (0, r); L_max is the largest
  load afterwards.
* Objectives reported per group: Phi_1 = max_r L_{k,r} - min_r L_{k,r} and
  Phi_2 = sum_r L_{k,r}.

Readings where the page is loose (listed in the design notes):
* "(W, ID) descending" is read literally: equal costs put the larger ID first;
  the solver's local sort uses the same key;
* heap ties (equal loads) go to the smaller rank index (tuple order);
* on a violation the current group is finalised and the violating tensor seeds
  the next group; a tensor whose cost alone exceeds C_max therefore forms a group
  of its own (retrying it as a seed could not succeed otherwise).
"""

from __future__ import annotations

import heapq
from typing import List, Sequence, Tuple


def _lpt_key(costs: Sequence[int]):
    return lambda i: (-int(costs[i]), -i)


def min_heap_solver(items: Sequence[int], costs: Sequence[int], R: int) -> Tuple[int, dict, List[int]]:
    """Assign the given parameter ids to R host ranks; returns (L_max, {id: rank}, loads)."""
    if R < 1:
        raise ValueError("R must be >= 1")
    order = sorted(items, key=_lpt_key(costs))
    pq = [(0, r) for r in range(R)]
    heapq.heapify(pq)
    assign = {}
    for p in order:
        load, r = heapq.heappop(pq)
        assign[p] = r
        heapq.heappush(pq, (load + int(costs[p]), r))
    loads = [0] * R
    for load, r in pq:
        loads[r] = load
    return max(loads), assign, loads


def plan_microgroups(costs: Sequence[int], R: int, c_max: int):
    """Returns (groups, host) where groups is a list of parameter-id lists in creation
    order and host[p] is the host rank of parameter p inside its group."""
    if R < 1:
        raise ValueError("R must be >= 1")
    if c_max <= 0:
        raise ValueError("c_max must be positive")
    if any(int(c) <= 0 for c in costs):
        raise ValueError("costs must be positive")
    order = sorted(range(len(costs)), key=_lpt_key(costs))
    groups: List[List[int]] = []
    curr: List[int] = []
    for p in order:
        if not curr:
            curr = [p]
            continue
        l_max, _, _ = min_heap_solver(curr + [p], costs, R)
        if l_max <= c_max:
            curr.append(p)
        else:
            groups.append(curr)
            curr = [p]
    if curr:
        groups.append(curr)
    host = [0] * len(costs)
    for g in groups:
        _, assign, _ = min_heap_solver(g, costs, R)
        for p, r in assign.items():
            host[p] = r
    return groups, host


def group_objectives(groups, host, costs, R):
    """Per group: (Phi_1 = max - min rank load, Phi_2 = total load, L_max)."""
    out = []
    for g in groups:
        loads = [0] * R
        for p in g:
            loads[host[p]] += int(costs[p])
        out.append((max(loads) - min(loads), sum(loads), max(loads)))
    return out
