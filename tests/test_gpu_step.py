"""GPU parity of the Muon step (through the C-ABI) against the fp64 CPU oracle.

Bars: momentum within 1e-6 relative; per-tensor update delta within 2e-2 relative
Frobenius error (bf16 Newton-Schulz vs fp64); the bf16 parameter copy equals RNE
of the GPU's own fp32 master bit for bit; untouched tensors bit-identical.
"""

import numpy as np
import pytest
import torch

from oracle import muon as OM
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

UPDATE_TOL = 2e-2
MOM_TOL = 1e-6
LR, MU = 0.02, 0.95


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


class Run:
    """One cz_muon_step_ex on the GPU with a debug delta buffer and a bf16 copy."""

    def __init__(self, shapes, R=1, alpha=1.0, buckets=None, seed=0, grad_std=1.0, grad_bf16=False,
                 param_std=0.02):
        self.shapes = list(shapes)
        self.numels = [r * c for r, c in self.shapes]
        self.offsets = list(np.cumsum([0] + self.numels[:-1]))
        buckets = buckets or [len(self.shapes)]
        self.plan = cz.cz_plan_partition(self.numels, buckets, R, alpha)
        self.owner = self.plan.owner()
        p = wl.draw(self.shapes, param_std, seed)
        g = wl.draw(self.shapes, grad_std, seed + 1, dtype=torch.bfloat16 if grad_bf16 else torch.float32)
        self.grad_bf16 = grad_bf16
        self.p0 = p.clone()
        self.g = g.clone()
        self.m0 = torch.zeros_like(p)
        dev = torch.device("cuda")
        self.P = p.to(dev)
        self.G = g.to(dev)
        self.M = self.m0.to(dev)
        self.PB = torch.zeros(p.numel(), dtype=torch.bfloat16, device=dev)
        self.D = torch.zeros(p.numel(), dtype=torch.float32, device=dev)
        self.args = cz.StepArgs(self.offsets, self.shapes)

    def step(self, rank=0, ns_steps=5, coeffs=None, nesterov=True):
        opts = cz.make_opts(param_bf16=self.PB, debug_update_out=self.D, grad_is_bf16=self.grad_bf16,
                            coeffs=coeffs, nesterov=nesterov)
        cz.cz_muon_step_ex(self.plan, rank, self.P, self.G, self.M, self.args, LR, MU, ns_steps, None, opts)
        assert cz.cz_device_status(None, None) == cz.CZ_OK
        torch.cuda.synchronize()

    def tensor(self, buf, i):
        r, c = self.shapes[i]
        o = self.offsets[i]
        return buf[o:o + r * c].reshape(r, c)


def check_against_oracle(run, owned, p_before, m_before, ns_steps=5, coeffs=OM.QUINTIC, tol=UPDATE_TOL,
                         nesterov=True):
    P = run.P.cpu()
    M = run.M.cpu()
    D = run.D.cpu()
    PB = run.PB.cpu()
    g = run.g.float() if run.grad_bf16 else run.g
    worst = 0.0
    for i in range(len(run.shapes)):
        Wg = run.tensor(P, i).numpy()
        if not owned[i]:
            assert torch.equal(run.tensor(P, i), run.tensor(p_before, i))
            assert torch.equal(run.tensor(M, i), run.tensor(m_before, i))
            continue
        gi = run.tensor(g, i).numpy()
        mi = run.tensor(m_before, i).numpy()
        m_new, u = OM.momentum(gi, mi, MU)
        if not nesterov:
            u = m_new.astype(np.float64)
        X = OM.orthogonalise(u, ns_steps, coeffs)
        r, c = run.shapes[i]
        delta = LR * OM.shape_scale(r, c) * X
        mg = run.tensor(M, i).numpy()
        assert rel_fro(mg, m_new) <= MOM_TOL, ("momentum", i)
        dg = run.tensor(D, i).numpy()
        e = rel_fro(dg, delta)
        worst = max(worst, e)
        t = tol[i] if isinstance(tol, (list, tuple)) else tol
        assert e <= t, ("update", i, run.shapes[i], e, t)
        # the master moved by exactly the delta the kernel reports (fp32 rounding)
        W0 = run.tensor(p_before, i).numpy().astype(np.float64)
        assert np.allclose(W0 - dg.astype(np.float64), Wg, rtol=0, atol=2e-7 * max(1.0, np.abs(W0).max()))
        # bf16 copy = RNE(fp32 master), bit for bit
        want = OM.bf16_rne(Wg)
        got = run.tensor(PB, i).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), ("bf16 copy", i)
    return worst


def test_tiny_config_single_rank():
    w = wl.tiny()
    run = Run(w.shapes, R=1)
    run.step()
    check_against_oracle(run, [True] * 6, run.p0, run.m0)


def test_tiny_config_two_ranks_partition_and_cross_rank_bit_identity():
    w = wl.tiny()
    run = Run(w.shapes, R=2)
    assert run.owner == [0, 0, 0, 1, 1, 1]
    run.step(rank=0)
    after0 = run.P.cpu().clone()
    check_against_oracle(run, [o == 0 for o in run.owner], run.p0, run.m0)
    run.step(rank=1)
    both = run.P.cpu()
    # the same tensors updated by a single rank owning everything give bit-identical results
    single = Run(w.shapes, R=1)
    single.step()
    assert torch.equal(both, single.P.cpu())
    assert torch.equal(run.M.cpu(), single.M.cpu())
    assert not torch.equal(after0, both)


@pytest.mark.parametrize("shapes", [
    [(300, 520), (520, 300), (136, 1000), (1000, 136)],          # several tiles, ragged tails, tall and wide
    [(129, 257), (257, 129), (7, 9), (1, 33), (33, 1)],           # odd sizes: scalar paths, tiny, vectors
    [(512, 512), (384, 1280), (1280, 384), (640, 128)],           # exact tiles, mixed groups
])
@pytest.mark.parametrize("grad_bf16", [False, True])
def test_ragged_and_multi_tile_shapes(shapes, grad_bf16):
    # bf16 gradients: 8-column vectors where offset and width allow, scalar loads elsewhere
    run = Run(shapes, R=1, seed=3, grad_std=1e-3 if grad_bf16 else 1.0, grad_bf16=grad_bf16)
    run.step()
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0)


def test_many_same_shape_tensors_and_bf16_grads():
    shapes = [(256, 768)] * 5 + [(768, 256)] * 4 + [(128, 128)] * 6
    run = Run(shapes, R=1, seed=5, grad_std=1e-3, grad_bf16=True)
    run.step()
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0)


def test_three_steps_teacher_forced():
    shapes = [(256, 512), (512, 256), (384, 384)]
    run = Run(shapes, R=1, seed=7, grad_std=1e-3)
    for step in range(3):
        p_before = run.P.cpu().clone()
        m_before = run.M.cpu().clone()
        if step:
            g = wl.draw(shapes, 1e-3, 100 + step)
            run.g = g
            run.G.copy_(g.cuda())
        run.step()
        check_against_oracle(run, [True] * 3, p_before, m_before)


def test_single_ns_step_and_other_coefficients():
    shapes = [(192, 320), (320, 192)]
    run = Run(shapes, R=1, seed=11)
    run.step(ns_steps=1)
    check_against_oracle(run, [True, True], run.p0, run.m0, ns_steps=1)
    # the cubic Newton-Schulz iteration through the same kernels
    run2 = Run(shapes, R=1, seed=11)
    run2.step(ns_steps=8, coeffs=OM.CUBIC)
    check_against_oracle(run2, [True, True], run2.p0, run2.m0, ns_steps=8, coeffs=OM.CUBIC)


def test_plain_momentum_without_nesterov():
    shapes = [(256, 256), (128, 384)]
    run = Run(shapes, R=1, seed=13)
    run.step(nesterov=False)
    check_against_oracle(run, [True, True], run.p0, run.m0, nesterov=False)


def test_qwen3_1p7b_layer_full_size():
    """The bench workload at full size: every tensor checked against the fp64 oracle."""
    w = wl.qwen3_1p7b_layers(1)
    run = Run(w.shapes, R=1, seed=0, grad_std=w.grad_std)
    run.step()
    worst = check_against_oracle(run, [True] * len(w.shapes), run.p0, run.m0)
    assert worst < UPDATE_TOL


def test_deterministic_repeat():
    shapes = [(384, 1024), (1024, 384), (256, 256)]
    a = Run(shapes, R=1, seed=17)
    b = Run(shapes, R=1, seed=17)
    a.step()
    b.step()
    assert torch.equal(a.P.cpu(), b.P.cpu())
    assert torch.equal(a.D.cpu(), b.D.cpu())


def test_caller_workspace_reused_between_calls():
    """A caller workspace whose memory is overwritten between calls (as when an
    allocator hands the same block to another tensor) gives the same results as
    the library's own workspace: the step re-sends its tables on every call."""
    shapes = [(256, 768), (768, 256), (128, 128)]
    a = Run(shapes, R=1, seed=23)
    b = Run(shapes, R=1, seed=23)
    ws_bytes = cz.cz_workspace_size(a.plan, 0, shapes)
    WS = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    for call in range(2):
        a.step()
        opts = cz.make_opts(param_bf16=b.PB, debug_update_out=b.D, workspace=WS, workspace_bytes=ws_bytes)
        cz.cz_muon_step_ex(b.plan, 0, b.P, b.G, b.M, b.args, LR, MU, 5, None, opts)
        assert cz.cz_device_status(None, WS) == cz.CZ_OK
        assert torch.equal(a.P.cpu(), b.P.cpu())
        assert torch.equal(a.M.cpu(), b.M.cpu())
        WS[256:].fill_(0xA5)        # scribble over everything but the status word


_CHILD = r"""
import json, sys, numpy as np, torch
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl
shapes = [tuple(x) for x in json.loads(sys.argv[2])]
ns_steps = int(sys.argv[3])
numels = [r * c for r, c in shapes]
offsets = list(np.cumsum([0] + numels[:-1]))
plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
P = wl.draw(shapes, 0.02, 31).cuda()
G = wl.draw(shapes, 1.0, 32).cuda()
M = torch.zeros_like(P)
cz.cz_profile_enable(True)
for _ in range(2):
    cz.cz_muon_step(plan, 0, P, G, M, cz.StepArgs(offsets, shapes), 0.02, 0.95, ns_steps)
torch.cuda.synchronize()
prof = cz.cz_profile_read()
assert cz.cz_device_status(None, None) == cz.CZ_OK
torch.save({"P": P.cpu(), "M": M.cpu(), "launches": {k: v[1] for k, v in prof.items()}}, sys.argv[1])
"""


def _run_child(tmp_path, env_name, env_value, shapes, ns_steps=5, extra_env=None):
    import json
    import os
    import subprocess
    import sys
    f = tmp_path / f"out_{env_name}_{env_value}.pt"
    e = dict(os.environ, **{env_name: env_value}, **(extra_env or {}))
    r = subprocess.run([sys.executable, "-c", _CHILD, str(f), json.dumps(shapes), str(ns_steps)], env=e,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return torch.load(f)


def test_fused_and_per_product_launches_are_bit_identical(tmp_path):
    """One persistent launch for all Newton-Schulz products and one launch per product
    compute every output tile with the same K order and epilogue: bit-identical
    results after two steps.  Each variant runs in its own process (the choice is
    read once per process)."""
    shapes = [(384, 1024), (1024, 384), (256, 256), (128, 640)]
    on = _run_child(tmp_path, "CZ_NS_FUSED", "1", shapes)
    off = _run_child(tmp_path, "CZ_NS_FUSED", "0", shapes)
    assert on["launches"]["ns_fused"] == 2 and on["launches"]["ns_gram"] == 0   # small shard: fused launch
    assert off["launches"]["ns_fused"] == 0 and off["launches"]["ns_gram"] >= 10  # >= one Gram launch per step
    assert torch.equal(on["P"], off["P"])
    assert torch.equal(on["M"], off["M"])
    # the same launch without the cooperative attribute (the form profilers replay)
    plain = _run_child(tmp_path, "CZ_NS_COOPERATIVE", "0", shapes)
    assert plain["launches"]["ns_fused"] == 2
    assert torch.equal(on["P"], plain["P"])


@pytest.mark.parametrize("fused", ["1", "0"])
def test_single_cta_tiles_and_cta_pair_tiles_are_bit_identical(tmp_path, fused):
    """CZ_NS_PAIR=0: the tiled products on single CTAs (128 x 256 tiles, cta_group::1) instead of CTA pairs
    (256 x 256, cta_group::2), in the fused launch and in one launch per product.  Each output element is
    accumulated over the same K sequence and rounded at the same points, so the bits agree; the shard also
    holds on-chip matrices of both kinds (their kernels do not depend on the switch)."""
    shapes = [(384, 1024), (1024, 384), (640, 640), (300, 520), (64, 96), (200, 240)]
    single = _run_child(tmp_path, "CZ_NS_PAIR", "0", shapes, extra_env={"CZ_NS_FUSED": fused})
    pair = _run_child(tmp_path, "CZ_NS_PAIR", "1", shapes, extra_env={"CZ_NS_FUSED": fused})
    if fused == "1":
        assert single["launches"]["ns_fused"] == 2 and pair["launches"]["ns_fused"] == 2
    else:
        assert single["launches"]["ns_gram"] >= 10 and pair["launches"]["ns_gram"] >= 10
    assert torch.equal(single["M"], pair["M"])
    assert torch.equal(single["P"], pair["P"])


@pytest.mark.parametrize("ns_steps", [5, 2])
def test_paced_per_product_launches_are_bit_identical(tmp_path, ns_steps):
    """One launch per product, waves of tiles started together or not (CZ_NS_PACE=0): the same tiles on
    the same units in the same order, so the same bits.  The Gram launch holds 120 tiles of two K values
    (5120 and 4096, 80 and 64 k-blocks): more than the GPU has units, so its second wave waits for the
    first (the paced prefix every unit has); the Poly and Update tiles (K = 1024) are not paced."""
    shapes = [(1024, 4096)] * 4 + [(4096, 1024)] * 4 + [(1024, 5120)] * 2 + [(5120, 1024)] * 2
    paced = _run_child(tmp_path, "CZ_NS_PACE", "1", shapes, ns_steps=ns_steps, extra_env={"CZ_NS_FUSED": "0"})
    plain = _run_child(tmp_path, "CZ_NS_PACE", "0", shapes, ns_steps=ns_steps, extra_env={"CZ_NS_FUSED": "0"})
    assert paced["launches"]["ns_fused"] == 0 and paced["launches"]["ns_gram"] == 2 * ns_steps
    assert torch.equal(paced["P"], plain["P"])
    assert torch.equal(paced["M"], plain["M"])


@pytest.mark.parametrize("ns_steps", [5, 2])
def test_latency_bound_fused_launch_is_bit_identical(tmp_path, ns_steps):
    """A shard whose products all have fewer tiles than the GPU has units runs the fused launch with
    twice the epilogue warps (its stage chains are the whole launch); the same tiles and epilogue math
    as one launch per product, so the same bits."""
    shapes = [(256, 256), (256, 512), (384, 640), (512, 256)]
    on = _run_child(tmp_path, "CZ_NS_FUSED", "1", shapes, ns_steps=ns_steps)
    off = _run_child(tmp_path, "CZ_NS_FUSED", "0", shapes, ns_steps=ns_steps)
    assert on["launches"]["ns_fused"] == 2 and off["launches"]["ns_fused"] == 0
    assert torch.equal(on["P"], off["P"])
    assert torch.equal(on["M"], off["M"])


@pytest.mark.parametrize("ns_steps", [5, 2])
def test_fused_schedule_and_list_walk_are_bit_identical(tmp_path, ns_steps):
    """The fused launch walks the host's dependency-aware schedule (each unit's tiles of every step in
    one sequence) or, with CZ_NS_SCHED=0, the per-(step, product) lists: the same tiles with the same
    K order and epilogues in another order across units, so the same bits, and one launch per step."""
    shapes = [(384, 1024), (1024, 384), (256, 256), (128, 640), (640, 640)]
    on = _run_child(tmp_path, "CZ_NS_SCHED", "1", shapes, ns_steps=ns_steps)
    off = _run_child(tmp_path, "CZ_NS_SCHED", "0", shapes, ns_steps=ns_steps)
    assert on["launches"]["ns_fused"] == 2 and off["launches"]["ns_fused"] == 2
    assert torch.equal(on["P"], off["P"])
    assert torch.equal(on["M"], off["M"])


_STEPS_CHILD = r"""
import json, sys, numpy as np, torch
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl
shapes = [tuple(x) for x in json.loads(sys.argv[2])]
counts = json.loads(sys.argv[3])
numels = [r * c for r, c in shapes]
offsets = list(np.cumsum([0] + numels[:-1]))
plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
P = wl.draw(shapes, 0.02, 41).cuda()
M = torch.zeros_like(P)
for k, n in enumerate(counts):
    G = wl.draw(shapes, 1.0, 42 + k).cuda()
    cz.cz_muon_step(plan, 0, P, G, M, cz.StepArgs(offsets, shapes), 0.02, 0.95, n)
torch.cuda.synchronize()
assert cz.cz_device_status(None, None) == cz.CZ_OK
torch.save({"P": P.cpu(), "M": M.cpu()}, sys.argv[1])
"""


def test_schedule_built_for_the_first_step_count_only(tmp_path):
    """The fused launch's schedule is built for the step count of the first call on a set of buffers;
    later calls with another count walk the lists.  Five calls of 5, 3, 5, 17 and 2 steps on the same
    buffers give the same bits with the schedule as with the lists alone (CZ_NS_SCHED=0)."""
    import json
    import os
    import subprocess
    import sys
    shapes = [(384, 1024), (1024, 384), (256, 256), (640, 640)]
    counts = [5, 3, 5, 17, 2]
    out = {}
    for sched in ("1", "0"):
        f = tmp_path / f"steps_{sched}.pt"
        r = subprocess.run([sys.executable, "-c", _STEPS_CHILD, str(f), json.dumps(shapes), json.dumps(counts)],
                           env=dict(os.environ, CZ_NS_SCHED=sched), capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        out[sched] = torch.load(f)
    assert torch.equal(out["1"]["P"], out["0"]["P"])
    assert torch.equal(out["1"]["M"], out["0"]["M"])


_SCHED_CHILD = r"""
import json, sys, numpy as np, torch
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl
shapes = [tuple(x) for x in json.loads(sys.argv[2])]
sched = json.loads(sys.argv[3])
numels = [r * c for r, c in shapes]
offsets = list(np.cumsum([0] + numels[:-1]))
args = cz.StepArgs(offsets, shapes)
plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
p0 = wl.draw(shapes, 0.02, 41)
g = wl.draw(shapes, 1.0, 42)
m0 = wl.draw(shapes, 0.5, 43)


def bufs():
    return {"P": p0.cuda(), "G": g.cuda(), "M": m0.cuda(),
            "PB": torch.zeros(p0.numel(), dtype=torch.bfloat16, device="cuda"),
            "D": torch.zeros(p0.numel(), device="cuda")}


def call(b, sc):
    o = cz.make_opts(param_bf16=b["PB"], debug_update_out=b["D"], nesterov=sc["nesterov"], eps=sc["eps"],
                     coeffs=tuple(sc["coeffs"]))
    cz.cz_muon_step_ex(plan, 0, b["P"], b["G"], b["M"], args, sc["lr"], sc["mu"], 5, None, o)
    torch.cuda.synchronize()
    assert cz.cz_device_status(None, None) == cz.CZ_OK


n0 = cz.cz_step_programs_built()
a = bufs()
call(a, sched[0])                     # builds a's program with the first scalars
n1 = cz.cz_step_programs_built()
for k in ("P", "M"):
    a[k].copy_({"P": p0, "M": m0}[k])
a["PB"].zero_()
a["D"].zero_()
call(a, sched[1])                     # the same program with the second scalars
n2 = cz.cz_step_programs_built()
b = bufs()
call(b, sched[1])                     # other buffers: a program built with the second scalars
n3 = cz.cz_step_programs_built()
torch.save({"a": {k: v.cpu() for k, v in a.items()}, "b": {k: v.cpu() for k, v in b.items()},
            "built": [n1 - n0, n2 - n1, n3 - n2]}, sys.argv[1])
"""


def test_step_scalars_are_launch_parameters(tmp_path):
    """lr, mu, eps, Nesterov and the Newton-Schulz coefficients can change from call to
    call (a learning-rate schedule) without a new step program, and a cached program
    called with new scalars gives, bit for bit, what a program built with them gives;
    on-chip small, tiled tall and wide, and ragged tensors; fused and per-product
    launches (one process each), both against the fp64 oracle with the new scalars."""
    import json
    import os
    import subprocess
    import sys
    shapes = [(64, 64), (96, 128), (384, 1024), (1024, 384), (300, 520)]
    sched = [{"lr": 0.02, "mu": 0.95, "eps": 1e-7, "nesterov": True, "coeffs": list(OM.QUINTIC)},
             {"lr": 0.0031, "mu": 0.8, "eps": 1e-5, "nesterov": False, "coeffs": list(OM.CUBIC)}]
    out = {}
    for fused in ("1", "0"):
        f = tmp_path / f"sched_{fused}.pt"
        env = dict(os.environ, CZ_NS_FUSED=fused)
        r = subprocess.run([sys.executable, "-c", _SCHED_CHILD, str(f), json.dumps(shapes), json.dumps(sched)],
                           env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        out[fused] = torch.load(f)
    for fused, d in out.items():
        assert d["built"] == [1, 0, 1], (fused, d["built"])
        for k in ("P", "M", "PB", "D"):
            assert torch.equal(d["a"][k], d["b"][k]), (fused, k)
    for k in ("P", "M", "PB", "D"):
        assert torch.equal(out["1"]["a"][k], out["0"]["a"][k]), k
    # the second scalars took effect: the fp64 oracle with them
    sc = sched[1]
    numels = [r * c for r, c in shapes]
    offsets = list(np.cumsum([0] + numels[:-1]))
    g = wl.draw(shapes, 1.0, 42)
    m0 = wl.draw(shapes, 0.5, 43)
    D, M = out["1"]["a"]["D"], out["1"]["a"]["M"]
    for (r, c), o in zip(shapes, offsets):
        gi = g[o:o + r * c].reshape(r, c).numpy()
        mi = m0[o:o + r * c].reshape(r, c).numpy()
        m_new, _ = OM.momentum(gi, mi, sc["mu"])
        assert rel_fro(M[o:o + r * c].reshape(r, c).numpy(), m_new) <= MOM_TOL
        X = OM.orthogonalise(m_new.astype(np.float64), 5, tuple(sc["coeffs"]), eps=sc["eps"])
        delta = sc["lr"] * OM.shape_scale(r, c) * X
        assert rel_fro(D[o:o + r * c].reshape(r, c).numpy(), delta) <= UPDATE_TOL, (r, c)


_EVICT_CHILD = r"""
import sys, numpy as np, torch
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl
w = wl.tiny()
plan = cz.cz_plan_partition(w.numels, [len(w.shapes)], 1, 1.0)
args = cz.StepArgs(w.offsets, w.shapes)
p0 = wl.draw(w.shapes, 0.02, 5).cuda()
G = wl.draw(w.shapes, 1.0, 6).cuda()
P, M = p0.clone(), torch.zeros_like(p0)
n = int(sys.argv[2])
D = [torch.zeros_like(p0) for _ in range(n)]
n0 = cz.cz_step_programs_built()
for k in list(range(n)) + [0]:          # n distinct programs, then the first (evicted) again
    P.copy_(p0)
    M.zero_()
    cz.cz_muon_step_ex(plan, 0, P, G, M, args, 0.02, 0.95, 5, None, cz.make_opts(debug_update_out=D[k]))
torch.cuda.synchronize()
assert cz.cz_device_status(None, None) == cz.CZ_OK
built = cz.cz_step_programs_built() - n0
same = all(torch.equal(D[0], d) for d in D)
torch.save({"built": built, "same": same, "D0": D[0].cpu(), "P": P.cpu()}, sys.argv[1])
"""


def test_program_cache_eviction_frees_page_locked_tables(tmp_path):
    """More distinct step programs than the cache keeps (64): the cache is cleared,
    each evicted program waits for its last table copy before its page-locked image
    is freed, an evicted program is rebuilt when its key returns, every call gives
    the same delta bit for bit, and the process exits cleanly with programs alive."""
    import subprocess
    import sys
    n = 70
    f = tmp_path / "evict.pt"
    r = subprocess.run([sys.executable, "-c", _EVICT_CHILD, str(f), str(n)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = torch.load(f)
    assert d["built"] == n + 1
    assert d["same"]
    w = wl.tiny()
    p0 = wl.draw(w.shapes, 0.02, 5)
    assert torch.equal(d["P"], p0 - d["D0"])      # the last call (a rebuilt program) applied that delta
    assert float(d["D0"].abs().max()) > 0


def test_two_caller_streams_with_small_and_tiled_matrices():
    """Two shards stepped at the same time on two caller streams (own workspaces), each with
    small matrices (on chip, one CTA and a CTA pair, on a side stream beside the tiled products) and
    tiled ones: every result equals that shard stepped alone on the default stream, bit for bit."""
    shapes = [(64, 64), (96, 128), (384, 1024), (300, 520), (200, 240)]
    runs = {k: Run(shapes, R=1, seed=s_) for k, s_ in (("a", 71), ("b", 72), ("ra", 71), ("rb", 72))}
    runs["ra"].step()
    runs["rb"].step()
    streams = {"a": torch.cuda.Stream(), "b": torch.cuda.Stream()}
    for k in ("a", "b"):
        r = runs[k]
        nb = cz.cz_workspace_size(r.plan, 0, shapes)
        r.WS = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        r.opts = cz.make_opts(param_bf16=r.PB, debug_update_out=r.D, workspace=r.WS, workspace_bytes=nb)
    torch.cuda.synchronize()
    for _ in range(3):       # the first call builds each program; later ones overlap on the GPU
        for k in ("a", "b"):
            r = runs[k]
            r.P.copy_(r.p0.cuda())
            r.M.zero_()
        torch.cuda.synchronize()
        for k in ("a", "b"):
            r = runs[k]
            cz.cz_muon_step_ex(r.plan, 0, r.P, r.G, r.M, r.args, LR, MU, 5, streams[k], r.opts)
        torch.cuda.synchronize()
        for k, ref in (("a", "ra"), ("b", "rb")):
            assert cz.cz_device_status(None, runs[k].WS) == cz.CZ_OK
            for buf in ("P", "M", "PB", "D"):
                assert torch.equal(getattr(runs[k], buf), getattr(runs[ref], buf)), (k, buf)


SMALL_SHAPES = [(1, 5), (7, 1), (3, 256), (256, 128), (128, 256), (100, 130), (130, 100), (64, 64),
                (128, 128), (17, 255), (33, 65), (96, 192)]


@pytest.mark.parametrize("ns_steps", [1, 2, 5])
def test_small_matrices_on_chip(ns_steps):
    """m <= 128 and n <= 256: every Newton-Schulz step in one CTA with the operands in
    shared memory (one ns_small launch for all of them), against the fp64 oracle;
    ragged m and n, vectors, tall and wide, the largest admitted shape, bf16 copy.
    A tensor whose bf16 storage alone moves it past 2e-2 (the rounding model of
    tests/bf16_model.py) is held to 1.5x the model's own error instead, and every
    tensor must also sit within 1e-2 of the rounding model."""
    from tests.bf16_model import orthogonalise_bf16
    run = Run(SMALL_SHAPES, R=1, seed=5)
    cz.cz_profile_enable(True)
    try:
        run.step(ns_steps=ns_steps)
        prof = cz.cz_profile_read()
    finally:
        cz.cz_profile_enable(False)
    assert prof["ns_small"][1] == 1
    assert all(prof[k][1] == 0 for k in ("ns_gram", "ns_poly", "ns_update", "ns_update_apply", "ns_fused"))
    tols = []
    D = run.D.cpu()
    for i, (r, c) in enumerate(SMALL_SHAPES):
        _, u = OM.momentum(run.tensor(run.g, i).numpy(), np.zeros((r, c), np.float32), MU)
        ref = OM.orthogonalise(u, ns_steps)
        model = orthogonalise_bf16(u, ns_steps)
        tols.append(max(UPDATE_TOL, 1.5 * rel_fro(model, ref)))
        got = run.tensor(D, i).numpy() / (LR * OM.shape_scale(r, c))
        assert rel_fro(got, model) <= 1e-2, ("vs rounding model", (r, c), rel_fro(got, model))
    check_against_oracle(run, [True] * len(SMALL_SHAPES), run.p0, run.m0, ns_steps=ns_steps, tol=tols)


PAIR_SHAPES = [(256, 256), (129, 256), (256, 129), (200, 240), (240, 200), (136, 136), (255, 256), (256, 255),
               (129, 129)]


@pytest.mark.parametrize("ns_steps", [1, 2, 5])
def test_small_pair_matrices_on_chip(ns_steps):
    """128 < m <= 256 and n <= 256: every Newton-Schulz step on a CTA pair with each CTA holding half of
    every iterate's rows in shared memory (one ns_small_pair launch for all of them), against the fp64
    oracle: ragged m and n on both CTAs' halves, tall and wide, the largest admitted shape, the
    smallest m the pair takes.  The single-CTA matrices of the shard run beside them."""
    from tests.bf16_model import orthogonalise_bf16
    shapes = PAIR_SHAPES + [(64, 64), (96, 200)]
    run = Run(shapes, R=1, seed=7)
    cz.cz_profile_enable(True)
    try:
        run.step(ns_steps=ns_steps)
        prof = cz.cz_profile_read()
    finally:
        cz.cz_profile_enable(False)
    assert prof["ns_small"][1] == 2                 # the single-CTA launch and the CTA-pair launch
    assert all(prof[k][1] == 0 for k in ("ns_gram", "ns_poly", "ns_update", "ns_update_apply", "ns_fused"))
    tols = []
    D = run.D.cpu()
    for i, (r, c) in enumerate(shapes):
        _, u = OM.momentum(run.tensor(run.g, i).numpy(), np.zeros((r, c), np.float32), MU)
        ref = OM.orthogonalise(u, ns_steps)
        model = orthogonalise_bf16(u, ns_steps)
        tols.append(max(UPDATE_TOL, 1.5 * rel_fro(model, ref)))
        got = run.tensor(D, i).numpy() / (LR * OM.shape_scale(r, c))
        assert rel_fro(got, model) <= 1e-2, ("vs rounding model", (r, c), rel_fro(got, model))
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0, ns_steps=ns_steps, tol=tols)


def test_more_small_matrices_than_the_gpu_holds_at_once():
    """90 CTA-pair matrices (180 CTAs of 193 KB shared memory, one per SM: more than the GPU's SMs, so the
    clusters run in waves) and 170 single-CTA ones in one shard: both on-chip launches cannot be resident
    together, so they run one after the other on the caller's stream; every tensor against the fp64
    oracle."""
    from tests.bf16_model import orthogonalise_bf16
    shapes = [(200, 240)] * 45 + [(240, 200)] * 45 + [(64, 96)] * 85 + [(96, 64)] * 85
    run = Run(shapes, R=1, seed=9)
    cz.cz_profile_enable(True)
    try:
        run.step()
        prof = cz.cz_profile_read()
    finally:
        cz.cz_profile_enable(False)
    assert prof["ns_small"][1] == 2
    assert all(prof[k][1] == 0 for k in ("ns_gram", "ns_poly", "ns_update", "ns_update_apply", "ns_fused"))
    tols = []
    for i, (r, c) in enumerate(shapes):
        _, u = OM.momentum(run.tensor(run.g, i).numpy(), np.zeros((r, c), np.float32), MU)
        tols.append(max(UPDATE_TOL, 1.5 * rel_fro(orthogonalise_bf16(u, 5), OM.orthogonalise(u, 5))))
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0, tol=tols)


def test_small_on_chip_and_tiled_paths_are_bit_identical(tmp_path):
    """The on-chip kernels (one CTA, or a CTA pair) keep the tiled kernels' arithmetic
    (same K order of the products, same folding, same bf16 rounding points), so
    sending the small matrices through the tiled GEMMs instead gives the same bits;
    the shard mixes small matrices of both kinds with one the tiled path must take
    (m = 384), so both on-chip launches run on the side stream, one after the other."""
    shapes = SMALL_SHAPES + PAIR_SHAPES + [(384, 512)]
    on = _run_child(tmp_path, "CZ_NS_SMALL", "1", shapes)
    off = _run_child(tmp_path, "CZ_NS_SMALL", "0", shapes)
    assert on["launches"]["ns_small"] == 4 and off["launches"]["ns_small"] == 0
    assert torch.equal(on["M"], off["M"])
    assert torch.equal(on["P"], off["P"])
    # no tiled matrix: the CTA-pair launch runs on the caller's stream beside the single-CTA one
    shapes = SMALL_SHAPES[:4] + PAIR_SHAPES[:4]
    on = _run_child(tmp_path, "CZ_NS_SMALL", "1", shapes)
    off = _run_child(tmp_path, "CZ_NS_SMALL", "0", shapes)
    assert on["launches"]["ns_small"] == 4 and off["launches"]["ns_small"] == 0
    assert torch.equal(on["M"], off["M"])
    assert torch.equal(on["P"], off["P"])


def test_low_rank_plus_noise_gradients_track_the_rounding_model():
    """Rank-8 gradients plus 5% noise, through the tiled path (wide, tall, and a larger wide one): bf16
    storage alone moves such tensors far past the 2e-2 bar (the quintic map scales the noise directions
    by up to a^5 ~ 485 along with the rounding of the dominant ones), so each tensor is held to 1.5x the
    rounding model's own distance from the fp64 oracle: the kernels lose no more than bf16 storage does."""
    from tests.bf16_model import orthogonalise_bf16
    shapes = [(128, 640), (640, 128), (256, 1024)]
    run = Run(shapes, R=1, seed=9)
    rng = np.random.default_rng(9)
    g = torch.zeros_like(run.g)
    for i, (r, c) in enumerate(shapes):
        lr_part = rng.standard_normal((r, 8)) @ rng.standard_normal((8, c))
        noise = 0.05 * np.linalg.norm(lr_part) / np.sqrt(r * c) * rng.standard_normal((r, c))
        o = run.offsets[i]
        g[o:o + r * c] = torch.from_numpy((lr_part + noise).astype(np.float32).reshape(-1))
    run.g = g
    run.G = g.cuda()
    run.step()
    tols = []
    for i, (r, c) in enumerate(shapes):
        _, u = OM.momentum(run.tensor(run.g, i).numpy(), np.zeros((r, c), np.float32), MU)
        e_model = rel_fro(orthogonalise_bf16(u, 5), OM.orthogonalise(u, 5))
        assert e_model > UPDATE_TOL          # the case this test is about
        tols.append(1.5 * e_model)
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0, tol=tols)


def test_degenerate_gradients_zero_and_rank_one():
    """A zero gradient (with zero momentum) leaves its tensor exactly unchanged: u = 0, X0 = 0 / (0 + eps) = 0,
    and the iteration keeps X = 0. An exactly rank-one gradient s u v^T: in exact arithmetic the update is
    lr * scale * f^5(1) u v^T (f^5(1) = 0.6964364). In bf16 the rounding of X0 puts singular values of order
    2^-9 beside the rank-one direction, which f^5 amplifies by up to a^5 ~ 485, so the update lands far from
    the closed form in Frobenius norm: the NumPy rounding model lands about 1.17 away. Held to: the component
    along u v^T within 1e-2 of f^5(1), every singular value of update / (lr * scale) in f's range (<= 1.3),
    and the Frobenius distance within 1.5x the rounding model's. Tiled wide, tall and square tensors, plus
    small ones on chip."""
    from tests.bf16_model import orthogonalise_bf16
    shapes = [(256, 640), (640, 256), (384, 384), (64, 96), (96, 64), (128, 256)]
    zero = {2, 5}
    run = Run(shapes, R=1, seed=29)
    rng = np.random.default_rng(29)
    g = torch.zeros_like(run.g)
    uv = {}
    for i, (r, c) in enumerate(shapes):
        if i in zero:
            continue
        u = rng.standard_normal(r); u /= np.linalg.norm(u)
        v = rng.standard_normal(c); v /= np.linalg.norm(v)
        uv[i] = np.outer(u, v)
        o = run.offsets[i]
        g[o:o + r * c] = torch.from_numpy((2.5 * uv[i]).astype(np.float32).reshape(-1))
    run.g = g
    run.G = g.cuda()
    run.step()
    P, M, D, PB = run.P.cpu(), run.M.cpu(), run.D.cpu(), run.PB.cpu()
    f5 = OM.ns_poly_scalar(1.0)
    for i, (r, c) in enumerate(shapes):
        if i in zero:
            assert torch.equal(run.tensor(P, i), run.tensor(run.p0, i))
            assert not bool(run.tensor(M, i).any()) and not bool(run.tensor(D, i).any())
            assert torch.equal(run.tensor(PB, i), run.tensor(run.p0, i).to(torch.bfloat16))
            continue
        x = run.tensor(D, i).numpy().astype(np.float64) / (LR * OM.shape_scale(r, c))
        assert abs(float(np.sum(x * uv[i])) - f5) <= 1e-2, (r, c)
        assert np.linalg.svd(x, compute_uv=False).max() <= 1.3, (r, c)
        _, u_in = OM.momentum(run.tensor(run.g, i).numpy(), np.zeros((r, c), np.float32), MU)
        exact = OM.orthogonalise(u_in, 5)
        e_model = rel_fro(orthogonalise_bf16(u_in, 5), exact)
        assert rel_fro(x, exact) <= 1.5 * e_model, (r, c)
        # the master moved by exactly the reported delta
        assert torch.equal(run.tensor(P, i), run.tensor(run.p0, i) - run.tensor(D, i))


def test_more_shape_groups_than_one_launch_holds():
    """40 distinct tiled shapes (a launch's problem table holds 32 groups): every Newton-Schulz product runs as
    two launches over the groups, the fused launch steps aside, and every tensor still matches the oracle."""
    shapes = [(130 + i, 260 + 2 * i) if i % 2 == 0 else (260 + 2 * i, 130 + i) for i in range(40)]
    run = Run(shapes, R=1, seed=17)
    cz.cz_profile_enable(True)
    try:
        run.step()
        prof = cz.cz_profile_read()
    finally:
        cz.cz_profile_enable(False)
    assert prof["ns_fused"][1] == 0
    assert prof["ns_gram"][1] == 2 * 5 and prof["ns_poly"][1] == 2 * 5
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0)


@pytest.mark.parametrize("ns_steps", [63, 64])
def test_largest_step_counts(tmp_path, ns_steps):
    """The largest accepted step counts (the fused launch's counters hold 64 steps): fused and
    per-product launches bit for bit, results finite, and every update's singular values,
    divided by lr * scale, inside the quintic map's band [0.5, 1.3].  After this many steps
    the fp64 oracle is no reference: the band's fixed points repel (|f'| = 1.58 at 0.868 and
    6.5 at 1.264), so rounding differences grow along each singular value's orbit."""
    shapes = [(384, 1024), (1024, 384), (256, 256)]
    run = Run(shapes, R=1, seed=23)
    run.step(ns_steps=ns_steps)
    D = run.D.cpu()
    assert bool(torch.isfinite(D).all())
    for i, (r, c) in enumerate(shapes):
        sv = np.linalg.svd(run.tensor(D, i).numpy().astype(np.float64) / (LR * OM.shape_scale(r, c)),
                           compute_uv=False)
        assert 0.5 <= sv.min() and sv.max() <= 1.3, ((r, c), sv.min(), sv.max())
    on = _run_child(tmp_path, "CZ_NS_FUSED", "1", shapes, ns_steps=ns_steps)
    off = _run_child(tmp_path, "CZ_NS_FUSED", "0", shapes, ns_steps=ns_steps)
    assert on["launches"]["ns_fused"] == 2 and off["launches"]["ns_fused"] == 0
    assert torch.equal(on["P"], off["P"])
    assert torch.equal(on["M"], off["M"])


@pytest.mark.parametrize("ns_steps", [2, 6])
def test_even_step_counts_end_in_the_other_x_buffer(tmp_path, ns_steps):
    """With an even number of Newton-Schulz steps the last Update (the apply) reads the second X ping-pong
    buffer: against the oracle, and the fused and per-product launches bit for bit."""
    shapes = [(384, 1024), (1024, 384), (256, 256)]
    run = Run(shapes, R=1, seed=21)
    run.step(ns_steps=ns_steps)
    check_against_oracle(run, [True] * len(shapes), run.p0, run.m0, ns_steps=ns_steps)
    on = _run_child(tmp_path, "CZ_NS_FUSED", "1", shapes, ns_steps=ns_steps)
    off = _run_child(tmp_path, "CZ_NS_FUSED", "0", shapes, ns_steps=ns_steps)
    assert on["launches"]["ns_fused"] == 2 and off["launches"]["ns_fused"] == 0
    assert torch.equal(on["P"], off["P"])
