"""cz_muon_step_noalloc against cz_muon_step_ex and the oracle, through the C-ABI.

The no-allocation entry point is for callers that cannot call cudaMalloc when
the optimizer step runs: a framework whose caching allocator owns all of device
memory, a runtime that reserves its memory up front, or code that must not
trigger the synchronisation that cudaMalloc/cudaFree can cause.  It runs the
same kernels with its scratch in a static device array, so for the same inputs
its results must be the allocating entry point's bit for bit, call after call,
even though the array keeps whatever the previous call (here: a call on another
plan and other buffers) left in it.

This file is collected last so that a run stopping at the first failure has
already run every other test.  Each test builds its own state, so the file
passes alone in a fresh process and after the others.
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
# small matrices (on-chip path), tiled ones, tall and wide, and a ragged shape
SHAPES = [(64, 64), (128, 64), (64, 192), (256, 256), (32, 128), (192, 96), (256, 768), (768, 256), (300, 520)]
# another shard, run between the calls compared, so the static array holds foreign tables and iterates
OTHER = [(384, 640), (96, 200), (1024, 512)]


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _layout(shapes):
    numels = [r * c for r, c in shapes]
    offsets = [int(x) for x in np.cumsum([0] + numels[:-1])]
    plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
    return plan, offsets, cz.StepArgs(offsets, shapes)


def _state(shapes, seed):
    dev = torch.device("cuda")
    P = wl.draw(shapes, 0.02, seed, device=dev)
    G = wl.draw(shapes, 1.0, seed + 1, device=dev)
    M = torch.zeros_like(P)
    PB = torch.zeros(P.numel(), dtype=torch.bfloat16, device=dev)
    D = torch.zeros_like(P)
    return P, G, M, PB, D


def test_noalloc_is_bit_identical_to_the_allocating_entry_point():
    plan, offsets, args = _layout(SHAPES)
    ws_bytes = cz.cz_workspace_size(plan, 0, SHAPES)
    assert ws_bytes <= cz.CZ_STATIC_WORKSPACE_BYTES
    P1, G1, M1, PB1, D1 = _state(SHAPES, 21)
    P2, G2, M2, PB2, D2 = _state(SHAPES, 21)
    WS = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")   # status word starts at zero
    opts_ref = cz.make_opts(param_bf16=PB1, workspace=WS, workspace_bytes=ws_bytes, debug_update_out=D1)
    opts_new = cz.make_opts(param_bf16=PB2, debug_update_out=D2)

    o_plan, _, o_args = _layout(OTHER)
    oP, oG, oM, oPB, _ = _state(OTHER, 5)

    free_deltas = []
    for call in range(3):
        g0 = G1.cpu().numpy().copy()
        m0 = M1.cpu().numpy().copy()
        cz.cz_muon_step_ex(plan, 0, P1, G1, M1, args, LR, MU, 5, None, opts_ref)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        cz.cz_muon_step_noalloc(plan, 0, P2, G2, M2, args, LR, MU, 5, None, opts_new)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        if call > 0:
            # the step program and the array exist since the first call: nothing more is allocated
            free_deltas.append(free0 - free1)
        assert cz.cz_device_status(None, WS) == cz.CZ_OK
        assert cz.cz_device_status(None, None) == cz.CZ_OK     # the static array's status word
        # the same kernels on the same inputs: the same bits
        assert torch.equal(P1, P2), call
        assert torch.equal(M1, M2), call
        assert torch.equal(PB1, PB2), call
        assert torch.equal(D1, D2), call
        # and the oracle agrees with the no-alloc step's delta and momentum
        Dh, Mh = D2.cpu().numpy(), M2.cpu().numpy()
        for off, (r, c) in zip(offsets, SHAPES):
            sl = slice(off, off + r * c)
            m_new, u = OM.momentum(g0[sl].reshape(r, c), m0[sl].reshape(r, c), MU)
            delta = LR * OM.shape_scale(r, c) * OM.orthogonalise(u, 5)
            assert rel_fro(Dh[sl].reshape(r, c), delta) <= UPDATE_TOL, (call, r, c)
            assert rel_fro(Mh[sl].reshape(r, c), m_new) <= MOM_TOL, (call, r, c)
        # a step on another plan and other buffers through the same static array
        cz.cz_muon_step_noalloc(o_plan, 0, oP, oG, oM, o_args, LR, MU, 5, None, cz.make_opts(param_bf16=oPB))
        # next call: new gradients, same buffers
        g = wl.draw(SHAPES, 1.0, 100 + call, device="cuda")
        G1.copy_(g)
        G2.copy_(g)
    assert cz.cz_device_status(None, None) == cz.CZ_OK
    assert free_deltas == [0, 0], free_deltas


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
