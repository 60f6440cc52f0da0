"""Oracle for the DP partition planner (test infrastructure only; see package header).

Written from the Canzona summary page "Canzona: A Unified, Asynchronous, and
Load-Balanced Framework for Distributed Matrix-based Optimizers"
(paper-graph-ui), section 3.4:

* "Paradigm 3: Static Partitioning", Eq. 1 -- the start-index ownership rule
  (r-1)*S <= Start_Index(p) < r*S with stride S = |B|/R.
* "The DP Load-Balance Optimization Problem" -- loads L_{i,r}, the objectives
  J_DP (Eq. 2) and J_Comm, the cumulative load Phi_i(u).
* "The alpha-Balanced Greedy LPT Algorithm (Algorithm 1)" -- LPT bucket order,
  deficits d_r, blended target v* = (1-alpha) v_even + alpha v_fill, atomic
  discretisation by argmin |Phi_k(u) - C|, last rank takes the remainder.

Readings taken where the pages are silent or inconsistent (all listed in the
design notes):
* ranks are 0-based: owner = floor(start / S)   (the worked example calls
  1*S <= start < 2*S "rank 1");
* Start_Index is an element offset relative to the bucket start, S per bucket;
* empty shards are allowed (s_{i,r-1} <= s_{i,r});
* argmin domain u in [s_{k,r-1}, n_k], ties go to the smaller u;
* buckets are formed by walking parameters in buffer order and closing a
  bucket once its element count reaches the cap (a parameter is never split).

All arithmetic is Python int (exact) and IEEE double, in the operation order
written below; the C++ planner must reproduce it bit for bit.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence


def make_buckets(numels: Sequence[int], cap: int) -> List[int]:
    """Parameters per bucket, consecutive in buffer order.

    A bucket is closed as soon as its element count is >= cap; a parameter is
    never split.  A trailing partial bucket is kept.  (Section 3.4 says only
    that buckets are ordered, non-splittable parameter sequences.)
    """
    if cap <= 0:
        raise ValueError("cap must be positive")
    counts: List[int] = []
    cur_n = 0
    cur_el = 0
    for ne in numels:
        cur_n += 1
        cur_el += int(ne)
        if cur_el >= cap:
            counts.append(cur_n)
            cur_n = 0
            cur_el = 0
    if cur_n:
        counts.append(cur_n)
    return counts


@dataclass
class Plan:
    """A Global Partition Map Pi plus what the planner derives from it."""

    R: int
    bucket_sizes: List[int]                 # params per bucket
    param_cuts: List[List[int]]             # per bucket, s_{i,0..R} in parameter indices
    elem_cuts: List[List[int]]              # per bucket, element offsets of the cuts
    owner: List[int] = field(default_factory=list)       # per parameter, 0-based rank
    rank_load: List[int] = field(default_factory=list)   # sum of W(p) per rank
    rank_elems: List[int] = field(default_factory=list)  # sum of numel(p) per rank


def _bucket_prefix(numels: Sequence[int], bucket_sizes: Sequence[int], costs=None):
    """Per bucket: its parameters' costs W(p) (numel(p) unless given), Phi_i(u)
    for u = 0..n_i in cost units, and the element prefix for the same cuts."""
    out = []
    pos = 0
    for nb in bucket_sizes:
        e = [int(x) for x in numels[pos:pos + nb]]
        w = e if costs is None else [int(x) for x in costs[pos:pos + nb]]
        phi = [0]
        for x in w:
            phi.append(phi[-1] + x)
        ephi = [0]
        for x in e:
            ephi.append(ephi[-1] + x)
        out.append((pos, w, phi, ephi))
        pos += nb
    return out


def _check(numels, bucket_sizes, R, costs=None):
    if R < 1:
        raise ValueError("R must be >= 1")
    if any(int(x) <= 0 for x in numels):
        raise ValueError("numel must be positive")
    if costs is not None and (len(costs) != len(numels) or any(int(x) <= 0 for x in costs)):
        raise ValueError("costs must be positive, one per parameter")
    if any(int(b) <= 0 for b in bucket_sizes):
        raise ValueError("bucket sizes must be positive")
    if sum(int(b) for b in bucket_sizes) != len(numels):
        raise ValueError("bucket sizes must cover all parameters")


def _finish(numels, bucket_sizes, R, param_cuts, elem_cuts, costs=None) -> Plan:
    owner = [0] * len(numels)
    load = [0] * R
    elems = [0] * R
    pos = 0
    for i, nb in enumerate(bucket_sizes):
        s = param_cuts[i]
        for r in range(R):
            for u in range(s[r], s[r + 1]):
                owner[pos + u] = r
                load[r] += int(numels[pos + u] if costs is None else costs[pos + u])
                elems[r] += int(numels[pos + u])
        pos += nb
    return Plan(R=R, bucket_sizes=list(bucket_sizes), param_cuts=param_cuts,
                elem_cuts=elem_cuts, owner=owner, rank_load=load, rank_elems=elems)


def plan_naive(numels: Sequence[int], bucket_sizes: Sequence[int], R: int) -> Plan:
    """Eq. 1, start-index rule, per bucket with S = |B_i| / R (exact rational).

    Parameter p with element offset o inside bucket B_i goes to the 0-based rank
    r with r*|B_i|/R <= o < (r+1)*|B_i|/R, i.e. r = floor(o*R / |B_i|).
    """
    _check(numels, bucket_sizes, R)
    param_cuts, elem_cuts = [], []
    for _, w, phi, _ in _bucket_prefix(numels, bucket_sizes):
        size = phi[-1]
        owners = [(phi[u] * R) // size for u in range(len(w))]
        # s_{i,r} = first parameter whose owner is >= r
        s = []
        for r in range(R + 1):
            u = 0
            while u < len(w) and owners[u] < r:
                u += 1
            s.append(u)
        s[0] = 0
        s[R] = len(w)
        param_cuts.append(s)
        elem_cuts.append([phi[u] for u in s])
    return _finish(numels, bucket_sizes, R, param_cuts, elem_cuts)


def plan_partition(numels: Sequence[int], bucket_sizes: Sequence[int], R: int,
                   alpha: float, costs: Sequence[int] = None) -> Plan:
    """Algorithm 1, alpha-Balanced Greedy LPT.  Cost W(p) = numel(p) by default; any
    positive integer cost per parameter (e.g. the Newton-Schulz FLOPs of the tensor,
    the non-linear cost of the pages' appendix D.5) can be given instead.  Loads,
    deficits and cut targets are in cost units; shard sizes stay in elements."""
    _check(numels, bucket_sizes, R, costs)
    if not (0.0 <= alpha <= 1.0):
        raise ValueError("alpha must lie in [0, 1]")
    buckets = _bucket_prefix(numels, bucket_sizes, costs)
    N = len(buckets)
    Wb = [b[2][-1] for b in buckets]                 # W^i, exact ints
    total = 0
    for x in Wb:
        total += x
    mu = float(total) / R                            # mu_load
    order = sorted(range(N), key=lambda i: (-Wb[i], i))   # LPT: W desc, index asc
    L = [0.0] * R
    param_cuts: List[List[int]] = [None] * N  # type: ignore[list-item]
    for k in order:
        phi = buckets[k][2]
        nk = len(phi) - 1
        # step 1: deficits, taken at the start of this bucket
        d = [max(0.0, mu - L[r]) for r in range(R)]
        D = 0.0
        for r in range(R):
            D += d[r]
        # steps 2-3: blended target v*
        if D > 0.0:
            v = [(1.0 - alpha) * (1.0 / R) + alpha * (d[r] / D) for r in range(R)]
        else:
            v = [1.0 / R for _ in range(R)]
        t = [float(Wb[k]) * v[r] for r in range(R)]
        # step 4: atomic discretisation onto parameter boundaries
        s = [0] * (R + 1)
        C = 0.0
        for r in range(R - 1):
            C += t[r]
            best_u = s[r]
            best = abs(float(phi[best_u]) - C)
            for u in range(s[r] + 1, nk + 1):
                dist = abs(float(phi[u]) - C)
                if dist < best:          # strict: ties keep the smaller u
                    best = dist
                    best_u = u
            s[r + 1] = best_u
            L[r] += float(phi[s[r + 1]] - phi[s[r]])
        s[R] = nk
        L[R - 1] += float(phi[s[R]] - phi[s[R - 1]])
        param_cuts[k] = s
    elem_cuts = [[buckets[i][3][u] for u in param_cuts[i]] for i in range(N)]
    return _finish(numels, bucket_sizes, R, param_cuts, elem_cuts, costs)


def metrics(plan: Plan) -> dict:
    """R_LB = max/avg rank load; J_DP = max_r |L_r - mu|; J_Comm = sum |S_{i,r} - |B_i|/R|.

    J_DP and J_Comm follow section 3.4 ("Objective 1", "Objective 2"); R_LB is
    the max/avg load-balance ratio the experiments report.  Sizes are elements
    (single dtype), so bytes and elements differ by a constant factor.
    """
    R = plan.R
    total = sum(plan.rank_load)
    mu = float(total) / R
    r_lb = (max(plan.rank_load) / mu) if total > 0 else 1.0
    j_dp = max(abs(float(x) - mu) for x in plan.rank_load)
    j_comm = 0.0
    for ec in plan.elem_cuts:
        size = ec[-1]
        for r in range(R):
            j_comm += abs(float(ec[r + 1] - ec[r]) - float(size) / R)
    return {"r_lb": r_lb, "j_dp": j_dp, "j_comm": j_comm}
