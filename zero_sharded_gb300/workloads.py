"""Seeded synthetic workloads: tensor shapes, buffer layout and random draws.

This module is the only code the CUDA path and the CPU oracle both use, so it
holds no step of the method: it lists Qwen3-shaped matrices, packs them at
consecutive offsets of one flat buffer, and draws Gaussian values with a seeded
``torch.Generator``.  It never loads the CUDA library.

The Canzona pages evaluate on Qwen3 models (1.7B to 32B) trained at sequence
length 4096 (summary page, section 5); no dataset or trained weights are needed
for the optimizer step, so Gaussian matrices of those shapes stand in for them.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence, Tuple

import torch

Shape = Tuple[int, int]

# rows x cols = out x in (PyTorch nn.Linear weight layout)
TINY_SHAPES: List[Shape] = [(64, 64), (128, 64), (64, 192), (256, 256), (32, 128), (192, 96)]


def qwen3_layer(hidden: int, q_out: int, kv_out: int, ffn: int) -> List[Tuple[str, Shape]]:
    """One decoder layer's matrices in forward order: q, k, v, o, gate, up, down."""
    return [("q", (q_out, hidden)), ("k", (kv_out, hidden)), ("v", (kv_out, hidden)),
            ("o", (hidden, q_out)), ("gate", (ffn, hidden)), ("up", (ffn, hidden)),
            ("down", (hidden, ffn))]


QWEN3_1P7B = qwen3_layer(hidden=2048, q_out=2048, kv_out=1024, ffn=6144)
QWEN3_14B = qwen3_layer(hidden=5120, q_out=5120, kv_out=1024, ffn=17408)
QWEN3_32B = qwen3_layer(hidden=5120, q_out=8192, kv_out=1024, ffn=25600)


@dataclass
class Workload:
    name: str
    shapes: List[Shape]
    names: List[str]
    param_std: float
    grad_std: float
    grad_bf16: bool = False
    bucket_cap: int = 0          # 0: one bucket holding every tensor
    R: int = 1
    alpha: float = 1.0

    @property
    def numels(self) -> List[int]:
        return [r * c for r, c in self.shapes]

    @property
    def offsets(self) -> List[int]:
        out, pos = [], 0
        for r, c in self.shapes:
            out.append(pos)
            pos += r * c
        return out

    @property
    def total(self) -> int:
        return sum(self.numels)


def tiny() -> Workload:
    """6 fp32 matrices at consecutive offsets; params N(0, .02), grads N(0, 1); R=2, alpha=1."""
    return Workload("tiny-6", list(TINY_SHAPES), [f"t{i}" for i in range(6)], 0.02, 1.0, R=2)


def qwen3_1p7b_layers(n_layers: int = 1) -> Workload:
    """n Qwen3-1.7B-shaped layers in forward order; params N(0, .02), grads N(0, 1e-3)."""
    shapes, names = [], []
    for layer in range(n_layers):
        for nm, sh in QWEN3_1P7B:
            shapes.append(sh)
            names.append(f"L{layer}.{nm}")
    name = "qwen3-1.7b-layer" if n_layers == 1 else f"qwen3-1.7b-{n_layers}layers"
    return Workload(name, shapes, names, 0.02, 1e-3)


def qwen3_32b_reverse(n_layers: int = 64, R: int = 32, alpha: float = 1.0,
                      bucket_cap: int = 40_000_000) -> Workload:
    """Qwen3-32B matrices laid out in reverse layer order (63 -> 0), each layer's
    forward list reversed (down, up, gate, o, v, k, q), in 40M-element buckets."""
    shapes, names = [], []
    for layer in reversed(range(n_layers)):
        for nm, sh in reversed(QWEN3_32B):
            shapes.append(sh)
            names.append(f"L{layer}.{nm}")
    return Workload("qwen3-32b-64L-reverse", shapes, names, 0.02, 1e-3,
                    bucket_cap=bucket_cap, R=R, alpha=alpha)


def qwen3_14b_microgroup(count: int = 64, seed: int = 0) -> Workload:
    """`count` matrices drawn uniformly over the 7 Qwen3-14B layer matrices (bf16 grads)."""
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, len(QWEN3_14B), (count,), generator=g).tolist()
    shapes = [QWEN3_14B[i][1] for i in idx]
    names = [f"m{j}.{QWEN3_14B[i][0]}" for j, i in enumerate(idx)]
    return Workload("qwen3-14b-microgroup64", shapes, names, 0.02, 1e-3, grad_bf16=True)


def draw(shapes: Sequence[Shape], std: float, seed: int, device="cpu",
         dtype=torch.float32) -> torch.Tensor:
    """One flat buffer of N(0, std^2) values, tensor by tensor in buffer order."""
    total = sum(r * c for r, c in shapes)
    gen = torch.Generator(device=device).manual_seed(seed)
    out = torch.empty(total, dtype=torch.float32, device=device)
    pos = 0
    for r, c in shapes:
        n = r * c
        out[pos:pos + n].normal_(0.0, std, generator=gen)
        pos += n
    return out.to(dtype)


def make_state(w: Workload, seed: int = 0, device="cpu"):
    """(param fp32, grad, momentum fp32 zeros): params from `seed`, grads from `seed + 1`."""
    p = draw(w.shapes, w.param_std, seed, device)
    gdt = torch.bfloat16 if w.grad_bf16 else torch.float32
    g = draw(w.shapes, w.grad_std, seed + 1, device, gdt)
    m = torch.zeros_like(p)
    return p, g, m


def draw_grad(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    gdt = torch.bfloat16 if w.grad_bf16 else torch.float32
    return draw(w.shapes, w.grad_std, seed, device, gdt)


def spectrum_matrix(rows: int, cols: int, sigmas: Sequence[float], seed: int):
    """U diag(sigma) V^T with Haar-random orthonormal factors (float64, numpy-compatible torch)."""
    k = min(rows, cols)
    g = torch.Generator().manual_seed(seed)
    U, _ = torch.linalg.qr(torch.randn(rows, k, generator=g, dtype=torch.float64))
    V, _ = torch.linalg.qr(torch.randn(cols, k, generator=g, dtype=torch.float64))
    s = torch.tensor(list(sigmas), dtype=torch.float64)
    return (U * s) @ V.T, U, s, V
