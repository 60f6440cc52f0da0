"""Planner report: load balance and planning time on the Qwen3-32B layout.

    python -m zero_sharded_gb300.plan_report

Everything here is host work through the C-ABI planner (no GPU):
* alpha sweep (Algorithm 1, R = 32): max/avg load ratio R_LB, J_DP, J_Comm, against
  the start-index split of Eq. 1 -- the analogue of the pages' alpha ablation;
* R sweep (16 .. 128) at alpha = 1 -- the analogue of their DP-size scaling of R_LB;
* cost model: W(p) = numel(p) against W(p) = Newton-Schulz FLOPs of the tensor,
  both judged by the FLOPs each rank then has to do (the heaviest rank sets the
  step time) -- the analogue of their numel-vs-FLOPs comparison;
* TP micro-groups (Qwen3-32B tensors, TP = 8 host ranks) for several capacities
  C_max: number of groups and the worst in-group imbalance;
* planning time of each planner.
"""

from __future__ import annotations

import time

from . import cz
from . import workloads as wl


def ns_flops(r: int, c: int, steps: int = 5) -> int:
    m, n = min(r, c), max(r, c)
    return steps * (4 * m * m * n + 2 * m * m * m)


def _row(cells):
    return "| " + " | ".join(str(x) for x in cells) + " |"


def report() -> str:
    w = wl.qwen3_32b_reverse()
    buckets = cz.cz_make_buckets(w.numels, w.bucket_cap)
    flops = [ns_flops(r, c) for r, c in w.shapes]
    out = [f"Layout: {w.name}: {len(w.numels)} tensors, {len(buckets)} buckets of >= {w.bucket_cap:,} elements, "
           f"{w.total:,} elements.", ""]

    out += ["**alpha sweep** (R = 32, cost = numel)", "",
            _row(["planner", "alpha", "R_LB (max/avg)", "J_DP (elements)", "J_Comm (elements)"]),
            _row(["---"] * 5)]
    naive = cz.cz_plan_naive(w.numels, buckets, 32).metrics()
    out.append(_row(["Eq. 1 start-index", "—", f"{naive['r_lb']:.3f}", f"{naive['j_dp']:.3e}",
                     f"{naive['j_comm']:.3e}"]))
    for a in (0.0, 0.25, 0.5, 0.75, 1.0):
        m = cz.cz_plan_partition(w.numels, buckets, 32, a).metrics()
        out.append(_row(["Alg. 1", a, f"{m['r_lb']:.3f}", f"{m['j_dp']:.3e}", f"{m['j_comm']:.3e}"]))

    out += ["", "**R sweep** (alpha = 1, cost = numel)", "",
            _row(["R", "R_LB Alg. 1", "R_LB Eq. 1", "heaviest rank (elements)", "plan time (ms)"]),
            _row(["---"] * 5)]
    for R in (16, 32, 64, 128):
        t0 = time.perf_counter()
        p = cz.cz_plan_partition(w.numels, buckets, R, 1.0)
        dt = (time.perf_counter() - t0) * 1e3
        out.append(_row([R, f"{p.metrics()['r_lb']:.3f}", f"{cz.cz_plan_naive(w.numels, buckets, R).metrics()['r_lb']:.3f}",
                         f"{max(p.rank_load()):,}", f"{dt:.2f}"]))

    out += ["", "**cost model** (R = 32, alpha = 1): FLOPs per rank under each plan", "",
            _row(["W(p)", "R_LB in FLOPs", "heaviest rank TFLOP", "R_LB in elements"]), _row(["---"] * 4)]
    for name, plan in (("numel", cz.cz_plan_partition(w.numels, buckets, 32, 1.0)),
                       ("NS FLOPs", cz.cz_plan_partition_cost(w.numels, flops, buckets, 32, 1.0))):
        own = plan.owner()
        fl = [0] * 32
        for o, f in zip(own, flops):
            fl[o] += f
        el = plan.rank_elems()
        out.append(_row([name, f"{max(fl) / (sum(fl) / 32):.3f}", f"{max(fl) / 1e12:.1f}",
                         f"{max(el) / (sum(el) / 32):.3f}"]))

    out += ["", "**TP micro-groups** (Qwen3-32B tensors as compute tasks, TP = 8 host ranks, W = numel)", "",
            _row(["C_max (elements)", "groups", "largest group", "worst max-min load / C_max", "plan time (ms)"]),
            _row(["---"] * 5)]
    for cmax in (64 << 20, 128 << 20, 256 << 20, 512 << 20):
        t0 = time.perf_counter()
        grp, host, ng = cz.cz_plan_microgroups(w.numels, 8, cmax)
        dt = (time.perf_counter() - t0) * 1e3
        loads = {}
        sizes = [0] * ng
        for p, (g, h) in enumerate(zip(grp, host)):
            loads.setdefault(g, [0] * 8)[h] += w.numels[p]
            sizes[g] += 1
        worst = max((max(v) - min(v)) for v in loads.values()) / cmax
        out.append(_row([f"{cmax:,}", ng, max(sizes), f"{worst:.3f}", f"{dt:.2f}"]))
    return "\n".join(out)


if __name__ == "__main__":
    print(report())
