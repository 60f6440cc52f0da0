"""cz_muon_step_noalloc against cz_muon_step_ex, through the C-ABI.

The no-allocation entry point is for callers that cannot call cudaMalloc when
the optimizer step runs (an allocator that owns all device memory, memory
reserved up front, or code that must not trigger the synchronisation that
cudaMalloc/cudaFree can cause).  It runs the same kernels with its scratch in a
static device array, so its results must match the allocating entry point's,
call after call, even though the array keeps the previous call's contents.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import numpy as np
import pytest
import torch

from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

UPDATE_TOL = 2e-2
MOM_TOL = 1e-6
LR, MU = 0.02, 0.95
SHAPES = [(64, 64), (128, 64), (64, 192), (256, 256), (32, 128), (192, 96), (256, 768), (768, 256), (300, 520)]


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _state(seed):
    dev = torch.device("cuda")
    P = wl.draw(SHAPES, 0.02, seed, device=dev)
    G = wl.draw(SHAPES, 1.0, seed + 1, device=dev)
    M = torch.zeros_like(P)
    PB = torch.zeros(P.numel(), dtype=torch.bfloat16, device=dev)
    return P, G, M, PB


def test_noalloc_matches_allocating_entry_point_two_calls():
    numels = [r * c for r, c in SHAPES]
    offsets = list(np.cumsum([0] + numels[:-1]))
    plan = cz.cz_plan_partition(numels, [len(SHAPES)], 1, 1.0)
    args = cz.StepArgs(offsets, SHAPES)
    assert cz.cz_workspace_size(plan, 0, SHAPES) <= cz.CZ_STATIC_WORKSPACE_BYTES

    P1, G1, M1, PB1 = _state(21)
    P2, G2, M2, PB2 = _state(21)
    ws_bytes = cz.cz_workspace_size(plan, 0, SHAPES)
    WS = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")   # status word starts at zero
    opts_ref = cz.make_opts(param_bf16=PB1, workspace=WS, workspace_bytes=ws_bytes)
    opts_new = cz.make_opts(param_bf16=PB2)

    for call in range(2):
        before = P1.cpu().clone()
        cz.cz_muon_step_ex(plan, 0, P1, G1, M1, args, LR, MU, 5, None, opts_ref)
        cz.cz_muon_step_noalloc(plan, 0, P2, G2, M2, args, LR, MU, 5, None, opts_new)
        torch.cuda.synchronize()
        assert cz.cz_device_status(None, WS) == cz.CZ_OK
        p1, p2 = P1.cpu().numpy(), P2.cpu().numpy()
        for off, (r, c) in zip(offsets, SHAPES):
            sl = slice(off, off + r * c)
            d_ref = before.numpy()[sl].astype(np.float64) - p1[sl]
            d_new = before.numpy()[sl].astype(np.float64) - p2[sl]
            assert rel_fro(d_new, d_ref) <= UPDATE_TOL, (call, r, c)
            assert rel_fro(M2.cpu().numpy()[sl], M1.cpu().numpy()[sl]) <= MOM_TOL, (call, r, c)
        assert torch.equal(PB1.cpu(), PB2.cpu()) or rel_fro(PB2.float().cpu(), PB1.float().cpu()) <= UPDATE_TOL
        # next call: new gradients, same buffers (the static array keeps the last call's contents)
        g = wl.draw(SHAPES, 1.0, 100 + call, device="cuda")
        G1.copy_(g)
        G2.copy_(g)


def test_noalloc_rejects_a_shard_larger_than_the_static_array():
    shapes = [(4096, 4096)]
    plan = cz.cz_plan_partition([4096 * 4096], [1], 1, 1.0)
    assert cz.cz_workspace_size(plan, 0, shapes) > cz.CZ_STATIC_WORKSPACE_BYTES
    args = cz.StepArgs([0], shapes)
    P = torch.zeros(4096 * 4096, device="cuda")
    with pytest.raises(cz.CzError) as e:
        cz.cz_muon_step_noalloc(plan, 0, P, P, P, args, LR, MU, 5)
    assert e.value.status == cz.CZ_ERR_NOMEM
    bad = cz.make_opts(workspace=P, workspace_bytes=16)
    small = cz.cz_plan_partition([64 * 64], [1], 1, 1.0)
    with pytest.raises(cz.CzError) as e:
        cz.cz_muon_step_noalloc(small, 0, P, P, P, cz.StepArgs([0], [(64, 64)]), LR, MU, 5, None, bad)
    assert e.value.status == cz.CZ_ERR_INVALID
