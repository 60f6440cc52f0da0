"""C-ABI planner (libcz) against the planner oracle, bit for bit, plus ABI surface checks.

No GPU needed: the planner is host code and the library loads without a device.
"""

import math
import os
import random
import re

import pytest
import torch

from oracle import planner as O
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "cz.h")


def _same_plan(c_plan, o_plan):
    pc, ec = c_plan.cuts()
    assert pc == o_plan.param_cuts
    assert ec == o_plan.elem_cuts
    assert c_plan.owner() == o_plan.owner
    assert c_plan.rank_load() == o_plan.rank_load
    cm, om = c_plan.metrics(), O.metrics(o_plan)
    for k in ("r_lb", "j_dp", "j_comm"):
        assert cm[k] == om[k], k          # bit-exact doubles


def test_header_symbols_exported():
    text = open(HEADER).read()
    names = sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|void)\s+(cz_\w+)\s*\(", text, re.M)))
    assert len(names) >= 15
    lib = cz.load()
    for n in names:
        assert hasattr(lib, n), n
    assert cz.cz_version().endswith("sm_103a")


def test_tiny_config_bit_exact():
    w = wl.tiny()
    for buckets in ([6], [1] * 6, [2, 4], [3, 3]):
        for alpha in (0.0, 0.25, 0.5, 1.0):
            _same_plan(cz.cz_plan_partition(w.numels, buckets, 2, alpha), O.plan_partition(w.numels, buckets, 2, alpha))
        _same_plan(cz.cz_plan_naive(w.numels, buckets, 2), O.plan_naive(w.numels, buckets, 2))


def test_qwen3_32b_layout_bit_exact():
    w = wl.qwen3_32b_reverse()
    b_c = cz.cz_make_buckets(w.numels, w.bucket_cap)
    b_o = O.make_buckets(w.numels, w.bucket_cap)
    assert b_c == b_o and len(b_c) == 320
    for R, alpha in ((32, 1.0), (32, 0.5), (16, 1.0), (128, 1.0), (32, 0.0)):
        _same_plan(cz.cz_plan_partition(w.numels, b_c, R, alpha), O.plan_partition(w.numels, b_o, R, alpha))
    _same_plan(cz.cz_plan_naive(w.numels, b_c, 32), O.plan_naive(w.numels, b_o, 32))


def test_random_layouts_bit_exact():
    rng = random.Random(1234)
    for it in range(2000):
        n = rng.randint(1, 40)
        numels = [rng.choice([rng.randint(1, 50), rng.randint(1, 5000), rng.randint(1, 10 ** 7)]) for _ in range(n)]
        cap = rng.randint(1, max(1, sum(numels)))
        buckets = O.make_buckets(numels, cap)
        assert cz.cz_make_buckets(numels, cap) == buckets
        R = rng.choice([1, 2, 3, 5, 8, 13, 32])
        alpha = rng.choice([0.0, 1.0, rng.random()])
        _same_plan(cz.cz_plan_partition(numels, buckets, R, alpha), O.plan_partition(numels, buckets, R, alpha))
        if it % 4 == 0:
            _same_plan(cz.cz_plan_naive(numels, buckets, R), O.plan_naive(numels, buckets, R))


def test_goldens_through_the_abi():
    import json
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "planner_alpha_blend.json")))
    for case in g["cases"]:
        p = cz.cz_plan_partition(g["numels"], g["bucket_sizes"], g["R"], case["alpha"])
        assert p.cuts()[0] == case["param_cuts"]
        assert p.rank_load() == case["rank_load"]
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "eq1_start_index_example.json")))
    assert cz.cz_plan_naive(g["numels"], g["bucket_sizes"], g["R"]).owner() == g["owner"]


def test_host_validation_returns_errors():
    lib = cz.load()
    with pytest.raises(cz.CzError) as e:
        cz.cz_plan_partition([1, 2], [2], 0, 1.0)
    assert e.value.status == cz.CZ_ERR_INVALID
    for bad in (([1, 2], [2], 2, -0.1), ([1, 2], [2], 2, 1.01), ([1, 2], [1], 2, 1.0), ([1, -2], [2], 2, 1.0),
                ([1, 2], [3], 2, 1.0), ([1, 2], [1, 0, 1], 2, 1.0)):
        with pytest.raises(cz.CzError):
            cz.cz_plan_partition(*bad)
    with pytest.raises(cz.CzError):
        cz.cz_plan_partition([1, 2], [2], 2, math.nan)
    with pytest.raises(cz.CzError):
        cz.cz_make_buckets([1, 2], 0)
    assert lib.cz_plan_info(None, None, None, None) == cz.CZ_ERR_INVALID
    lib.cz_plan_free(None)


def test_step_validation_before_any_gpu_work():
    """Invalid step arguments are rejected on the host (no device is touched)."""
    w = wl.tiny()
    p = cz.cz_plan_partition(w.numels, [6], 2, 1.0)
    args = cz.StepArgs(w.offsets, w.shapes)
    fake = 0x1000
    for rank in (-1, 2):
        with pytest.raises(cz.CzError) as e:
            cz.cz_muon_step(p, rank, fake, fake, fake, args, 0.02, 0.95, 5)
        assert e.value.status == cz.CZ_ERR_INVALID
    with pytest.raises(cz.CzError) as e:
        cz.cz_muon_step(p, 0, fake, fake, fake, args, 0.02, 0.95, 0)
    assert e.value.status == cz.CZ_ERR_INVALID
    bad_shapes = cz.StepArgs(w.offsets, [(64, 64)] * 6)
    with pytest.raises(cz.CzError) as e:
        cz.cz_muon_step(p, 0, fake, fake, fake, bad_shapes, 0.02, 0.95, 5)
    assert e.value.status == cz.CZ_ERR_PLAN_MISMATCH
    overlap = cz.StepArgs([0] * 6, w.shapes)
    with pytest.raises(cz.CzError) as e:
        cz.cz_muon_step(p, 0, fake, fake, fake, overlap, 0.02, 0.95, 5)
    assert e.value.status == cz.CZ_ERR_PLAN_MISMATCH
    with pytest.raises(cz.CzError) as e:
        cz.cz_muon_step(p, 0, None, fake, fake, args, 0.02, 0.95, 5)
    assert e.value.status == cz.CZ_ERR_INVALID
    # base addresses must allow 16-byte vectors (a view at an odd element offset is refused, not run)
    for bad in ((fake + 4, fake, fake), (fake, fake + 8, fake), (fake, fake, fake + 4)):
        with pytest.raises(cz.CzError) as e:
            cz.cz_muon_step(p, 0, *bad, args, 0.02, 0.95, 5)
        assert e.value.status == cz.CZ_ERR_INVALID
    for o in (cz.make_opts(param_bf16=fake + 2), cz.make_opts(debug_update_out=fake + 4),
              cz.make_opts(grad_is_bf16=True), cz.make_opts(lr_device=fake + 2)):
        pg = fake + 4 if o.grad_is_bf16 else fake        # a bf16 gradient needs 8-byte alignment
        with pytest.raises(cz.CzError) as e:
            cz.cz_muon_step_ex(p, 0, fake, pg, fake, args, 0.02, 0.95, 5, None, o)
        assert e.value.status == cz.CZ_ERR_INVALID


def test_workspace_size_grows_with_shard():
    w = wl.qwen3_1p7b_layers(1)
    p1 = cz.cz_plan_partition(w.numels, [len(w.numels)], 1, 1.0)
    p2 = cz.cz_plan_partition(w.numels, [len(w.numels)], 2, 1.0)
    s1 = cz.cz_workspace_size(p1, 0, w.shapes)
    s2 = sum(cz.cz_workspace_size(p2, r, w.shapes) for r in range(2))
    # two bf16 X buffers (m x n), A and B' (m x m) per tensor dominate: ~4 mn + 4 m^2 bytes
    approx = sum(4 * r * c + 4 * min(r, c) ** 2 for r, c in w.shapes)
    assert approx <= s1 <= approx * 1.05
    assert s2 >= s1 * 0.95


def test_bucket_pack_validation_before_any_gpu_work():
    """cz_bucket_pack / cz_bucket_unpack reject bad layouts on the host (never touching the buffers, which are
    host tensors standing in for device ones); a zero-sized block is a no-op."""
    import ctypes
    lib = cz.load()
    b = torch.zeros(10)
    p = torch.zeros(20)
    bad = [([1, 10], 10), ([0, 6, 4], 10), ([0, 6, 10], 5), ([0, 10], -1)]
    for cuts, block in bad:
        for fn in (cz.cz_bucket_pack, cz.cz_bucket_unpack):
            with pytest.raises(cz.CzError) as e:
                fn(b, cuts, block, p)
            assert e.value.status == cz.CZ_ERR_INVALID
    cut_arr = (ctypes.c_int64 * 2)(0, 10)
    for elem_bytes in (0, 3, 16):
        assert lib.cz_bucket_pack(b.data_ptr(), elem_bytes, cut_arr, 1, 10, p.data_ptr(), None) == cz.CZ_ERR_INVALID
    assert lib.cz_bucket_pack(None, 4, cut_arr, 1, 10, p.data_ptr(), None) == cz.CZ_ERR_INVALID
    assert lib.cz_bucket_unpack(p.data_ptr(), 4, cut_arr, 1, 10, None, None) == cz.CZ_ERR_INVALID
    many = (ctypes.c_int64 * 1026)(*([0] * 1026))
    assert lib.cz_bucket_pack(b.data_ptr(), 4, many, 1025, 0, p.data_ptr(), None) == cz.CZ_ERR_INVALID  # > 1024 ranks
    empty = (ctypes.c_int64 * 3)(0, 0, 0)
    assert lib.cz_bucket_pack(b.data_ptr(), 4, empty, 2, 0, p.data_ptr(), None) == cz.CZ_OK      # nothing to move


def test_apply_validation_before_any_gpu_work():
    """cz_apply_update rejects bad arguments on the host; an empty list is a no-op."""
    fake = 0x1000
    cz.cz_apply_update(None, None, None, [], [], 0.02)          # n_tensors = 0: nothing to do
    cases = [
        dict(offsets=[0, 10], shapes=[(4, 4), (2, 2)]),          # overlapping tensors
        dict(offsets=[-4], shapes=[(2, 2)]),                     # negative offset
        dict(offsets=[0], shapes=[(0, 3)]),                      # empty shape
        dict(offsets=[0], shapes=[(2, 2)], lr=math.inf),         # non-finite lr
        dict(offsets=[0], shapes=[(2, 2)], param=None),          # missing buffer
        dict(offsets=[0], shapes=[(2, 2)], param=fake + 2),      # fp32 buffer not 4-byte aligned
    ]
    for cse in cases:
        with pytest.raises(cz.CzError) as e:
            cz.cz_apply_update(cse.get("param", fake), None, fake, cse["offsets"], cse["shapes"], cse.get("lr", 0.02))
        assert e.value.status == cz.CZ_ERR_INVALID, cse
    st = cz.load().cz_apply_update(fake, None, fake, cz._i64([0]), cz._i64([2, 2]), 1, 0.02, 2, None)
    assert st == cz.CZ_ERR_INVALID                               # shape_scale must be 0 or 1


def test_empty_shard_is_a_no_op_without_a_device():
    """A rank that owns no tensor (more ranks than single-tensor buckets) returns CZ_OK before any
    device work: the call succeeds here, where there is no GPU to launch on."""
    numels = [64 * 64, 32 * 128]
    shapes = [(64, 64), (32, 128)]
    p = cz.cz_plan_partition(numels, [1, 1], 4, 1.0)
    owner = p.owner()
    empty = [r for r in range(4) if r not in owner]
    assert empty
    fake = 0x1000
    built = cz.cz_step_programs_built()
    for r in empty:
        cz.cz_muon_step(p, r, fake, fake, fake, cz.StepArgs([0, 4096], shapes), 0.02, 0.95, 5)
    with pytest.raises(cz.CzError):                     # rejected on the host: nothing is built either
        cz.cz_muon_step(p, 0, fake + 4, fake, fake, cz.StepArgs([0, 4096], shapes), 0.02, 0.95, 5)
    assert cz.cz_step_programs_built() == built
