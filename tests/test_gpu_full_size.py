"""Full-size GPU checks: the largest workloads in the bench's launch configuration,
failure detection on the device, and checkpoint/resume.

At full size the fp64 oracle cannot run every tensor in a test, so each workload
checks every tensor against properties that hold at any size (momentum, the
fp32 master moving by exactly the reported delta, the bf16 copy = RNE(master))
and compares a sample of tensors, one per distinct shape where affordable,
against the CPU oracle.
"""

import numpy as np
import pytest
import torch

from oracle import muon as OM
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

UPDATE_TOL = 2e-2
LR, MU = 0.02, 0.95


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _run_full(w, sample_idx):
    dev = torch.device("cuda")
    gdt = torch.bfloat16 if w.grad_bf16 else torch.float32
    P0 = wl.draw(w.shapes, w.param_std, 0, device=dev)
    G = wl.draw(w.shapes, w.grad_std, 1, device=dev, dtype=gdt)
    M = torch.zeros_like(P0)
    P = P0.clone()
    PB = torch.zeros(P.numel(), dtype=torch.bfloat16, device=dev)
    D = torch.zeros_like(P0)
    plan = cz.cz_plan_partition(w.numels, [len(w.numels)], 1, 1.0)
    ws = cz.cz_workspace_size(plan, 0, w.shapes)
    WS = torch.zeros(ws, dtype=torch.uint8, device=dev)
    opts = cz.make_opts(param_bf16=PB, workspace=WS, workspace_bytes=ws, debug_update_out=D,
                        grad_is_bf16=w.grad_bf16)
    cz.cz_muon_step_ex(plan, 0, P, G, M, cz.StepArgs(w.offsets, w.shapes), LR, MU, 5, None, opts)
    assert cz.cz_device_status(None, WS) == cz.CZ_OK
    torch.cuda.synchronize()
    # properties of every tensor, on the device
    Gf = G.float()
    assert torch.equal(M, Gf)                                   # first step from zero: m = g
    assert torch.equal(P, P0 - D)                               # master moved by exactly the reported delta
    assert torch.equal(PB, P.to(torch.bfloat16))                # bf16 copy = RNE(master)
    assert bool(torch.isfinite(D).all())
    worst = 0.0
    for i in sample_idx:
        r, c = w.shapes[i]
        o = w.offsets[i]
        g = Gf[o:o + r * c].reshape(r, c).cpu().numpy()
        m0 = np.zeros((r, c), np.float32)
        _, u = OM.momentum(g, m0, MU)
        delta = LR * OM.shape_scale(r, c) * OM.orthogonalise(u, 5)
        e = rel_fro(D[o:o + r * c].reshape(r, c).cpu().numpy(), delta)
        worst = max(worst, e)
        assert e <= UPDATE_TOL, (w.names[i], (r, c), e)
    del P0, G, M, P, PB, D, WS
    torch.cuda.empty_cache()
    return worst


def test_qwen3_14b_microgroup_full_size():
    w = wl.qwen3_14b_microgroup(64)
    first = {}
    for i, s in enumerate(w.shapes):
        first.setdefault(s, i)
    # k/v (1024x5120), q/o (5120x5120), down (5120x17408, wide) and gate/up (17408x5120, tall: the
    # transposed apply), each the first of its shape in the draw
    sample = [first[s] for s in [(1024, 5120), (5120, 5120), (5120, 17408), (17408, 5120)] if s in first]
    assert (5120, 17408) in first and (17408, 5120) in first
    _run_full(w, sample)


def test_qwen3_1p7b_28_layers_full_size():
    """28 Qwen3-1.7B layers (196 matrices, 1,409,286,144 elements, byte offsets past
    5 GB) in one flat buffer: every tensor through the device-side properties, the
    oracle on the first tensor of each distinct shape and on the buffer's last tensor."""
    w = wl.qwen3_1p7b_layers(28)
    assert w.total == 1_409_286_144
    first = {}
    for i, s in enumerate(w.shapes):
        first.setdefault(s, i)
    sample = sorted(set(first.values()) | {len(w.shapes) - 1})
    assert len(first) == 4 and w.offsets[-1] * 4 > (5 << 30)
    _run_full(w, sample)


def test_qwen3_32b_heaviest_shard_full_size():
    full = wl.qwen3_32b_reverse()
    b = cz.cz_make_buckets(full.numels, full.bucket_cap)
    plan = cz.cz_plan_partition(full.numels, b, full.R, full.alpha)
    loads = plan.rank_load()
    heavy = max(range(len(loads)), key=lambda r: loads[r])
    own = plan.owner()
    shapes = [s for s, o in zip(full.shapes, own) if o == heavy]
    names = [n for n, o in zip(full.names, own) if o == heavy]
    w = wl.Workload("shard", shapes, names, 0.02, 1e-3)
    tall = [i for i, (r, c) in enumerate(shapes) if r > c]
    wide = [i for i, (r, c) in enumerate(shapes) if r <= c]
    # gate/up (25600x5120) take the transposed apply, down (5120x25600) the direct one: one of each
    assert tall and wide
    _run_full(w, [tall[0], wide[0]])


def test_bounded_wait_times_out_and_context_stays_usable():
    WS = torch.zeros(256, dtype=torch.uint8, device="cuda")
    cz.cz_selftest_bounded_wait(2_000_000, WS)          # 2 ms limit on a barrier nothing completes
    assert cz.cz_device_status(None, WS) == cz.CZ_ERR_TIMEOUT
    assert cz.cz_device_status(None, WS) == cz.CZ_OK    # read clears it
    # the context still runs the step correctly
    w = wl.tiny()
    p, g, m = wl.make_state(w, seed=0)
    P, G, M = p.cuda(), g.cuda(), m.cuda()
    D = torch.zeros_like(P)
    plan = cz.cz_plan_partition(w.numels, [6], 1, 1.0)
    cz.cz_muon_step_ex(plan, 0, P, G, M, cz.StepArgs(w.offsets, w.shapes), LR, MU, 5, None,
                       cz.make_opts(debug_update_out=D))
    assert cz.cz_device_status(None, None) == cz.CZ_OK
    Dh = D.cpu().numpy()
    for off, (r, c) in zip(w.offsets, w.shapes):
        _, u = OM.momentum(g.numpy()[off:off + r * c].reshape(r, c), np.zeros((r, c), np.float32), MU)
        delta = LR * OM.shape_scale(r, c) * OM.orthogonalise(u, 5)
        assert rel_fro(Dh[off:off + r * c].reshape(r, c), delta) <= UPDATE_TOL


def test_checkpoint_resume_is_bit_identical():
    """State = fp32 master + momentum (the plan is recomputed from numels, buckets, R, alpha):
    3 steps, save, reload into fresh buffers, 3 steps == 6 straight steps, bit for bit."""
    shapes = [(256, 768), (768, 256), (384, 384), (128, 640)]
    numels = [r * c for r, c in shapes]
    offsets = list(np.cumsum([0] + numels[:-1]))
    args = cz.StepArgs(offsets, shapes)
    grads = [wl.draw(shapes, 1e-3, 50 + k).cuda() for k in range(6)]

    def fresh():
        plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
        return plan

    p0 = wl.draw(shapes, 0.02, 3).cuda()
    # straight run
    plan = fresh()
    P, M = p0.clone(), torch.zeros_like(p0)
    for k in range(6):
        cz.cz_muon_step(plan, 0, P, grads[k], M, args, LR, MU, 5)
    torch.cuda.synchronize()
    straight = (P.cpu().clone(), M.cpu().clone())
    # run, checkpoint to host, resume with a new plan and new device buffers
    plan = fresh()
    P, M = p0.clone(), torch.zeros_like(p0)
    for k in range(3):
        cz.cz_muon_step(plan, 0, P, grads[k], M, args, LR, MU, 5)
    torch.cuda.synchronize()
    ckpt = (P.cpu().clone(), M.cpu().clone())
    del P, M, plan
    plan = fresh()
    P, M = ckpt[0].cuda(), ckpt[1].cuda()
    for k in range(3, 6):
        cz.cz_muon_step(plan, 0, P, grads[k], M, args, LR, MU, 5)
    torch.cuda.synchronize()
    assert cz.cz_device_status(None, None) == cz.CZ_OK
    assert torch.equal(P.cpu(), straight[0])
    assert torch.equal(M.cpu(), straight[1])
