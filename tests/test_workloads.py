"""The seeded synthetic inputs (zero_sharded_gb300/workloads.py), on the CPU.

Both sides of every parity test draw their inputs here, so the recipe is pinned:
the shapes and buffer layout of each workload, the reverse layer order of the
Qwen3-32B layout, the Qwen3-14B micro-group draw, and the determinism of the
seeded Gaussian draws (parameters from seed s, gradients from seed s + 1).
"""

import torch

from zero_sharded_gb300 import workloads as wl


def test_tiny_layout():
    w = wl.tiny()
    assert w.shapes == [(64, 64), (128, 64), (64, 192), (256, 256), (32, 128), (192, 96)]
    assert w.offsets == [0, 4096, 12288, 24576, 90112, 94208]
    assert w.total == 112_640 and w.R == 2 and w.grad_std == 1.0


def test_qwen3_layer_counts():
    one = wl.qwen3_1p7b_layers(1)
    assert [n.split(".")[1] for n in one.names] == ["q", "k", "v", "o", "gate", "up", "down"]
    assert one.total == 50_331_648
    assert wl.qwen3_1p7b_layers(28).total == 28 * 50_331_648 == 1_409_286_144
    big = wl.qwen3_32b_reverse()
    assert len(big.shapes) == 448 and big.total == 31_205_621_760
    assert big.names[:7] == [f"L63.{n}" for n in ("down", "up", "gate", "o", "v", "k", "q")]
    assert big.names[-1] == "L0.q" and big.bucket_cap == 40_000_000 and big.R == 32 and big.alpha == 1.0


def test_qwen3_14b_microgroup_draw():
    w = wl.qwen3_14b_microgroup(64)
    allowed = {s for _, s in wl.QWEN3_14B}
    assert len(w.shapes) == 64 and set(w.shapes) <= allowed and w.grad_bf16
    kinds = {n.split(".")[1] for n in w.names}             # q, k, v, o, gate, up, down: 4 distinct shapes
    assert len(kinds) >= 6 and set(w.shapes) == allowed    # a uniform draw of 64 over 7 kinds covers nearly all
    assert w.shapes == wl.qwen3_14b_microgroup(64).shapes  # seeded
    assert w.total == sum(r * c for r, c in w.shapes)


def test_draws_are_seeded_and_distinct():
    shapes = [(96, 64), (33, 17)]
    a = wl.draw(shapes, 0.02, 7)
    assert torch.equal(a, wl.draw(shapes, 0.02, 7))
    assert not torch.equal(a, wl.draw(shapes, 0.02, 8))
    w = wl.Workload("t", shapes, ["a", "b"], 0.02, 1e-3)
    p, g, m = wl.make_state(w, seed=3)
    assert torch.equal(p, wl.draw(shapes, 0.02, 3)) and torch.equal(g, wl.draw(shapes, 1e-3, 4))
    assert not bool(m.any()) and p.dtype == torch.float32 and g.dtype == torch.float32
    wb = wl.Workload("t", shapes, ["a", "b"], 0.02, 1e-3, grad_bf16=True)
    assert wl.make_state(wb, seed=3)[1].dtype == torch.bfloat16


def test_draw_statistics():
    x = wl.draw([(1024, 1024)], 0.5, 11).double()
    assert abs(float(x.mean())) < 5e-3 and abs(float(x.std()) - 0.5) < 5e-3
