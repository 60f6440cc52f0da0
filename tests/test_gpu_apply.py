"""GPU parity of the standalone scale-and-apply (cz_apply_update) through the C-ABI.

Against the fp64 oracle (oracle.muon.apply_update, rounded once to fp32): the
kernel rounds twice (fp32(coef * U), then fp32(W - d)) with coef = fp32(lr * scale),
so |W_gpu - W_oracle| <= 2^-23 * (|W_new| + |coef * U|) (one half-ulp per rounding
plus the oracle's own rounding, with margin).  The bf16 copy equals RNE of the
GPU's fp32 result bit for bit; bytes outside the listed tensors are untouched.
Against the fused apply of the Muon step: the same delta gives the same bits.
"""

import numpy as np
import pytest
import torch

from oracle import muon as OM
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


def _layout(shapes, gaps):
    """Offsets with the given gap (elements) before each tensor; returns (offsets, total)."""
    offs, cur = [], 0
    for (r, c), g in zip(shapes, gaps):
        cur += g
        offs.append(cur)
        cur += r * c
    return offs, cur + 5


def _run_apply(shapes, gaps, lr, shape_scale=True, seed=0, with_bf16=True):
    offs, total = _layout(shapes, gaps)
    gen = torch.Generator().manual_seed(seed)
    W = torch.full((total,), SENTINEL, dtype=torch.float32)
    U = torch.full((total,), -SENTINEL, dtype=torch.float32)
    for o, (r, c) in zip(offs, shapes):
        W[o:o + r * c] = 0.02 * torch.randn(r * c, generator=gen)
        U[o:o + r * c] = torch.randn(r * c, generator=gen)
    Wd, Ud = W.cuda(), U.cuda()
    PB = torch.full((total,), 7.0, dtype=torch.bfloat16, device="cuda") if with_bf16 else None
    cz.cz_apply_update(Wd, PB, Ud, offs, shapes, lr, shape_scale)
    torch.cuda.synchronize()
    return W, U, offs, Wd.cpu(), (PB.cpu() if with_bf16 else None)


def _check(W, U, offs, shapes, Wg, PB, lr, shape_scale=True):
    inside = np.zeros(W.numel(), bool)
    for o, (r, c) in zip(offs, shapes):
        sl = slice(o, o + r * c)
        inside[sl] = True
        w0 = W[sl].numpy().reshape(r, c)
        u = U[sl].numpy().reshape(r, c)
        want = OM.apply_update(w0, u, lr, shape_scale)
        got = Wg[sl].numpy().reshape(r, c)
        coef = lr * (OM.shape_scale(r, c) if shape_scale else 1.0)
        bound = 2.0 ** -23 * (np.abs(want).astype(np.float64) + np.abs(coef * u.astype(np.float64))) * 1.001
        err = np.abs(got.astype(np.float64) - want.astype(np.float64))
        assert np.all(err <= bound), ((r, c), float(err.max()))
        if PB is not None:
            bits = PB[sl].view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(bits, OM.bf16_rne(got).reshape(-1)), ("bf16 copy", (r, c))
    assert np.array_equal(Wg.numpy()[~inside], W.numpy()[~inside]), "bytes outside the tensors changed"
    if PB is not None:
        assert bool(torch.all(PB[torch.from_numpy(~inside)] == 7.0)), "bf16 bytes outside the tensors changed"


@pytest.mark.parametrize("gaps", [[0, 0, 0, 0, 0, 0], [4, 8, 3, 1, 7, 2]])
def test_apply_ragged_tall_wide_against_oracle(gaps):
    # a tail below one vector, a chunk boundary (4096) plus a ragged tail, tall and wide;
    # odd gaps put tensors at offsets that are not multiples of 4 (scalar path)
    shapes = [(7, 13), (300, 17), (64, 64), (1, 5), (4097, 1), (33, 129)]
    W, U, offs, Wg, PB = _run_apply(shapes, gaps, lr=0.02)
    _check(W, U, offs, shapes, Wg, PB, 0.02)


def test_apply_without_shape_scale_is_the_local_add():
    """TP lifecycle stage 4, P += Delta W: lr = -1 and no shape scale give the fp32 sum exactly."""
    shapes = [(96, 32), (17, 45)]
    W, U, offs, Wg, PB = _run_apply(shapes, [0, 3], lr=-1.0, shape_scale=False)
    _check(W, U, offs, shapes, Wg, PB, -1.0, shape_scale=False)
    for o, (r, c) in zip(offs, shapes):
        sl = slice(o, o + r * c)
        assert np.array_equal(Wg[sl].numpy(), W[sl].numpy() + U[sl].numpy())


def test_apply_without_bf16_copy():
    shapes = [(40, 24)]
    W, U, offs, Wg, _ = _run_apply(shapes, [0], lr=0.5, with_bf16=False)
    _check(W, U, offs, shapes, Wg, None, 0.5)


def test_apply_more_tensors_than_one_launch_takes():
    """300 small tensors (one launch takes 256): the second launch covers the rest; ragged gaps between."""
    shapes = [(3 + (i % 5), 2 + (i % 7)) for i in range(300)]
    gaps = [i % 3 for i in range(300)]
    W, U, offs, Wg, PB = _run_apply(shapes, gaps, lr=0.02, seed=5)
    _check(W, U, offs, shapes, Wg, PB, 0.02)


def test_apply_full_qwen3_1p7b_layer():
    w = wl.qwen3_1p7b_layers(1)
    W, U, offs, Wg, PB = _run_apply(w.shapes, [0] * len(w.shapes), lr=0.02, seed=3)
    _check(W, U, offs, w.shapes, Wg, PB, 0.02)


def test_standalone_apply_equals_the_fused_apply():
    """The Muon step's fused apply subtracts the delta it reports (debug_update_out); applying
    that delta with the standalone kernel (lr = 1, no scale) from the same weights gives the
    same fp32 master and bf16 copy bit for bit: tiled wide and tall tensors, on-chip small ones."""
    shapes = [(384, 128), (128, 384), (256, 256), (64, 192), (192, 96), (32, 128)]
    numels = [r * c for r, c in shapes]
    offs = list(np.cumsum([0] + numels[:-1]))
    plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
    p = wl.draw(shapes, 0.02, 0).cuda()
    g = wl.draw(shapes, 1.0, 1).cuda()
    m = torch.zeros_like(p)
    p0 = p.clone()
    D = torch.zeros_like(p)
    PB = torch.zeros(p.numel(), dtype=torch.bfloat16, device="cuda")
    opts = cz.make_opts(param_bf16=PB, debug_update_out=D)
    cz.cz_muon_step_ex(plan, 0, p, g, m, cz.StepArgs(offs, shapes), 0.02, 0.95, 5, None, opts)
    assert cz.cz_device_status(None, None) == cz.CZ_OK
    PB2 = torch.zeros_like(PB)
    cz.cz_apply_update(p0, PB2, D, offs, shapes, 1.0, False)
    torch.cuda.synchronize()
    assert torch.equal(p0, p)
    assert torch.equal(PB2.view(torch.int16), PB.view(torch.int16))
