"""The bench's reference arm on the CPU: one JSON line with the contract's keys.

`bench.py --impl reference` times the fp64 oracle on the host cores (the one leg of
the bench that runs without a GPU); its line must carry the same metric, unit and
direction as the GPU arm, plus `impl`, `cpu_baseline` and a zero-copy `e2e`.
"""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "ms" and d["higher_is_better"] is False
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "tiny-6" and d["config"]["matrices"] == 6
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "timed whole" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_qwen3_32b_shard_workloads():
    """The headline shard and the two shards of the cost comparison, picked through libcz's planner and
    through the oracle's (the reference arm's) alike."""
    sys.path.insert(0, ROOT)
    import bench

    for planner in ("cz", "oracle"):
        w, buckets, R, alpha, run_rank, ex = bench.build_workload("qwen3-32b-shard", 1, 0, planner=planner)
        # the heaviest planned load (numel): 8 FFN matrices of 5120 x 25600, both orientations
        assert sorted({(min(s), max(s)) for s in w.shapes}) == [(5120, 25600)] and len(w.shapes) == 8
        assert {s[0] > s[1] for s in w.shapes} == {True, False}
        assert w.total == 1_048_576_000 and ex["R"] == 32 and ex["cost"] == "numel"
        assert buckets == [8] and R == 1 and run_rank == 0
        heavy = ex["plan_rank"]
        # the numel plan's slowest rank carries more Newton-Schulz flops than its heaviest-load rank
        w2, *_, ex2 = bench.build_workload("qwen3-32b-shard-numel-maxflops", 1, 0, planner=planner)
        assert bench.ns_flops(w2.shapes) > bench.ns_flops(w.shapes)
        # under the flops cost no rank carries more flops than the heaviest-load shard of the numel plan
        w3, *_, ex3 = bench.build_workload("qwen3-32b-shard-flops", 1, 0, planner=planner)
        assert ex3["cost"] == "flops" and bench.ns_flops(w3.shapes) <= bench.ns_flops(w.shapes)
        if planner == "cz":
            ref = (heavy, ex2["plan_rank"], ex3["plan_rank"], w2.shapes, w3.shapes)
        else:
            assert ref == (heavy, ex2["plan_rank"], ex3["plan_rank"], w2.shapes, w3.shapes)
    # GPU rank k of a multi-GPU run takes the k-th heaviest plan rank
    ws = [bench.build_workload("qwen3-32b-shard", 4, k)[5]["plan_rank"] for k in range(4)]
    assert ws[0] == heavy and len(set(ws)) == 4


def test_executed_flops_by_kind_sum_to_the_total():
    sys.path.insert(0, ROOT)
    import bench

    for shapes in ([(5120, 25600), (25600, 5120)], [(2048, 2048), (1024, 2048), (6144, 2048), (2048, 6144)],
                   [(300, 520), (64, 64), (256, 768)]):
        k = bench.ns_flops_executed_by_kind(shapes)
        tiled = [s for s in shapes if not bench._is_small(*s)]
        assert k["ns_gram"] + k["ns_poly"] + k["ns_update"] + k["ns_update_apply"] == k["ns_fused"]
        assert k["ns_fused"] == bench.ns_flops_executed(tiled)
        assert k["ns_small"] == bench.ns_flops_executed([s for s in shapes if bench._is_small(*s)])
        # the Update products are dense: executed = algorithmic when the sizes are multiples of the tile
        if all(min(s) % 256 == 0 and max(s) % 256 == 0 for s in tiled):
            a = bench.ns_flops_by_kind(shapes)
            assert k["ns_update"] == a["ns_update"] and k["ns_update_apply"] == a["ns_update_apply"]
            assert k["ns_gram"] < a["ns_gram"] and k["ns_poly"] < a["ns_poly"]
