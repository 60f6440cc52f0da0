"""TP Micro-Group planner: oracle pins and the C-ABI planner bit-exact against the oracle.

Pins: hand-worked examples of the greedy rollback, Graham's LPT bound for the
MinHeapSolver against a brute-force optimum on tiny inputs, closed-form cases,
and the maximality of every rollback.
"""

import itertools
import json
import os
import random

import pytest

from oracle import microgroup as MG
from oracle import planner as P
from zero_sharded_gb300 import cz

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _groups_to_index(groups, n):
    idx = [0] * n
    for g, members in enumerate(groups):
        for p in members:
            idx[p] = g
    return idx


def test_golden_examples_oracle_and_abi():
    g = json.load(open(os.path.join(GOLDEN, "microgroup_examples.json")))
    for case in g["cases"]:
        groups, host = MG.plan_microgroups(case["costs"], case["R"], case["c_max"])
        assert _groups_to_index(groups, len(case["costs"])) == case["group"], case["name"]
        assert host == case["host"], case["name"]
        assert len(groups) == case["n_groups"]
        cg, ch, n = cz.cz_plan_microgroups(case["costs"], case["R"], case["c_max"])
        assert (cg, ch, n) == (case["group"], case["host"], case["n_groups"]), case["name"]


def _opt_makespan(costs, R):
    best = None
    for assign in itertools.product(range(R), repeat=len(costs)):
        loads = [0] * R
        for c, r in zip(costs, assign):
            loads[r] += c
        m = max(loads)
        best = m if best is None else min(best, m)
    return best


def test_min_heap_solver_graham_bound_and_closed_forms():
    rng = random.Random(5)
    for _ in range(200):
        n = rng.randint(1, 7)
        R = rng.randint(1, 3)
        costs = [rng.randint(1, 50) for _ in range(n)]
        lmax, assign, loads = MG.min_heap_solver(list(range(n)), costs, R)
        opt = _opt_makespan(costs, R)
        assert opt <= lmax <= (4.0 / 3.0 - 1.0 / (3.0 * R)) * opt + 1e-9     # Graham (1969)
        assert sum(loads) == sum(costs)
        assert lmax == max(loads)
    assert MG.min_heap_solver([0, 1, 2], [3, 4, 5], 1)[0] == 12                 # R = 1: the sum
    assert MG.min_heap_solver(list(range(7)), [6] * 7, 3)[0] == 18              # ceil(7/3) * 6


def test_rollback_properties_random():
    rng = random.Random(11)
    for _ in range(300):
        n = rng.randint(1, 40)
        R = rng.randint(1, 8)
        costs = [rng.choice([rng.randint(1, 10), rng.randint(1, 1000), rng.randint(1, 10 ** 6)]) for _ in range(n)]
        c_max = rng.randint(1, max(2, sum(costs) // rng.randint(1, 6)))
        groups, host = MG.plan_microgroups(costs, R, c_max)
        order = sorted(range(n), key=lambda i: (-costs[i], -i))
        assert [p for g in groups for p in g] == order          # groups are consecutive runs of the LPT order
        for k, g in enumerate(groups):
            lmax, _, _ = MG.min_heap_solver(g, costs, R)
            assert lmax <= c_max or len(g) == 1                # only a singleton may exceed C_max
            if k + 1 < len(groups):                           # maximal: the next tensor would not fit
                assert MG.min_heap_solver(g + [groups[k + 1][0]], costs, R)[0] > c_max
        objs = MG.group_objectives(groups, host, costs, R)
        for (phi1, phi2, lm), g in zip(objs, groups):
            assert phi2 == sum(costs[p] for p in g) and phi1 >= 0 and lm <= max(c_max, max(costs[p] for p in g))
        cg, ch, ng = cz.cz_plan_microgroups(costs, R, c_max)
        assert cg == _groups_to_index(groups, n) and ch == host and ng == len(groups)


def test_microgroup_invalid_inputs():
    with pytest.raises(ValueError):
        MG.plan_microgroups([1, 2], 0, 5)
    with pytest.raises(ValueError):
        MG.plan_microgroups([1, 0], 2, 5)
    with pytest.raises(cz.CzError):
        cz.cz_plan_microgroups([1, 2], 0, 5)
    with pytest.raises(cz.CzError):
        cz.cz_plan_microgroups([1, -2], 2, 5)
    with pytest.raises(cz.CzError):
        cz.cz_plan_microgroups([1, 2], 2, 0)


def test_flops_cost_alg1_golden_and_abi():
    g = json.load(open(os.path.join(GOLDEN, "planner_flops_cost.json")))
    pc = P.plan_partition(g["numels"], g["bucket_sizes"], g["R"], g["alpha"], costs=g["costs"])
    assert pc.owner == g["owner_cost"] and pc.rank_load == g["rank_load_cost"] and pc.rank_elems == g["rank_elems_cost"]
    pn = P.plan_partition(g["numels"], g["bucket_sizes"], g["R"], g["alpha"])
    assert pn.owner == g["owner_numel"] and pn.rank_load == g["rank_load_numel"]
    c = cz.cz_plan_partition_cost(g["numels"], g["costs"], g["bucket_sizes"], g["R"], g["alpha"])
    assert c.owner() == g["owner_cost"] and c.rank_load() == g["rank_load_cost"]
    assert c.rank_elems() == g["rank_elems_cost"]


def test_flops_cost_alg1_bit_exact_random():
    rng = random.Random(17)
    for _ in range(500):
        n = rng.randint(1, 30)
        numels = [rng.randint(1, 10 ** 6) for _ in range(n)]
        costs = [rng.randint(1, 10 ** 12) for _ in range(n)]
        buckets = P.make_buckets(numels, rng.randint(1, sum(numels)))
        R = rng.choice([1, 2, 3, 8, 32])
        alpha = rng.choice([0.0, 1.0, rng.random()])
        o = P.plan_partition(numels, buckets, R, alpha, costs=costs)
        c = cz.cz_plan_partition_cost(numels, costs, buckets, R, alpha)
        pc, ec = c.cuts()
        assert pc == o.param_cuts and ec == o.elem_cuts
        assert c.owner() == o.owner and c.rank_load() == o.rank_load and c.rank_elems() == o.rank_elems
        m, om = c.metrics(), P.metrics(o)
        assert m == om
