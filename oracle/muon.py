"""Oracle for the local Muon step one DP rank runs on the tensors it owns.

TEST INFRASTRUCTURE ONLY (see the package header).  Plain fp64 NumPy, one tensor
at a time, no blocking, fusion or reordering.

The Canzona pages fix the shape of the update but not its formulas: the summary
page (paper-graph-ui), sections 2 and 3.4, gives W_{t+1} = W_t - eta *
MatrixOp(W_t, grad W_t) and says Muon orthogonalises the (momentum) gradient with
Newton-Schulz iterations built from matrix products that mix all rows and
columns; section 4.1 ("Asynchronous computation") writes the host-rank step as
Delta W = Muon_step(G, States_local) with the momentum state resident on the
owner.  The concrete step used here is the standard Muon update with the
hyper-parameters this workload fixes:

  1. momentum (SGD form, Nesterov):  m <- mu*m + g  (stored fp32);  u = g + mu*m
  2. Frobenius normalisation:        X0 = u / (||u||_F + eps),  eps = 1e-7
  3. orientation:                    X0 is m x n with m = min(rows, cols); a tall
                                     tensor (rows > cols) is transposed
  4. K Newton-Schulz steps:          A = X X^T;  B = b A + c A A;  X <- a X + B X
                                     quintic (a, b, c) = (3.4445, -4.7750, 2.0315)
  5. back to rows x cols, then apply W <- W - lr * sqrt(max(1, rows/cols)) * X_K
     in fp32; the bf16 parameter copy is RNE(W).

No weight decay.  The EMA ("lerp") momentum form would give the same X_K (the
normalisation removes the (1-mu) factor) but a different stored m; the SGD form
is the one checked.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np

QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)
EPS = 1e-7


def ns_poly_scalar(s: float, coeffs=QUINTIC, steps: int = 5) -> float:
    """The scalar map f^K(s), f(s) = a s + b s^3 + c s^5, that NS applies to each singular value."""
    a, b, c = coeffs
    x = float(s)
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def newton_schulz(X0: np.ndarray, steps: int, coeffs=QUINTIC) -> np.ndarray:
    """K steps of A = X X^T; B = b A + c A A; X <- a X + B X, in fp64 (X already m x n, m <= n)."""
    a, b, c = coeffs
    X = np.asarray(X0, dtype=np.float64)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def momentum(g: np.ndarray, m: np.ndarray, mu: float) -> Tuple[np.ndarray, np.ndarray]:
    """m_new = fp32(mu*m + g) (the stored state) and the Nesterov input u = g + mu*m_new (fp64)."""
    g64 = np.asarray(g, dtype=np.float64)
    m64 = np.asarray(m, dtype=np.float64)
    m_new = (mu * m64 + g64).astype(np.float32)
    u = g64 + mu * m_new.astype(np.float64)
    return m_new, u


def orthogonalise(u: np.ndarray, steps: int, coeffs=QUINTIC, eps: float = EPS) -> np.ndarray:
    """Steps 2-5 up to (not including) the scale: X_K in the tensor's rows x cols layout."""
    u = np.asarray(u, dtype=np.float64)
    rows, cols = u.shape
    X = u / (np.sqrt(np.sum(u * u)) + eps)
    tall = rows > cols
    if tall:
        X = X.T
    X = newton_schulz(X, steps, coeffs)
    if tall:
        X = X.T
    return X


def shape_scale(rows: int, cols: int) -> float:
    return float(np.sqrt(max(1.0, rows / cols)))


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns the uint16 bit patterns."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    out = (rounded & 0xFFFF).astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def apply_update(W: np.ndarray, X: np.ndarray, lr: float, shape_scale_on: bool = True) -> np.ndarray:
    """Step 5 alone: fp32(W - lr * sqrt(max(1, rows/cols)) * X), computed in fp64 and rounded once.

    W is the fp32 rows x cols tensor, X the update in the same layout; with
    shape_scale_on False the coefficient is lr alone (the TP lifecycle's local
    add P += Delta W is lr = -1)."""
    W = np.asarray(W, dtype=np.float32)
    rows, cols = W.shape
    coef = lr * (shape_scale(rows, cols) if shape_scale_on else 1.0)
    return (W.astype(np.float64) - coef * np.asarray(X, dtype=np.float64)).astype(np.float32)


def muon_step_tensor(W: np.ndarray, g: np.ndarray, m: np.ndarray, lr: float, mu: float,
                     steps: int = 5, coeffs=QUINTIC, eps: float = EPS):
    """One Muon step on one whole tensor (rows x cols).

    Returns (W_new fp32, m_new fp32, W_new as bf16 bits, delta fp64) where
    delta = lr * sqrt(max(1, rows/cols)) * X_K is what is subtracted.
    """
    W = np.asarray(W, dtype=np.float32)
    rows, cols = W.shape
    m_new, u = momentum(g, m, mu)
    X = orthogonalise(u, steps, coeffs, eps)
    delta = lr * shape_scale(rows, cols) * X
    W_new = apply_update(W, X, lr)
    return W_new, m_new, bf16_rne(W_new), delta


def muon_step_flat(flat_param, flat_grad, flat_mom, offsets, shapes, owned, lr, mu,
                   steps: int = 5, coeffs=QUINTIC, eps: float = EPS):
    """Apply muon_step_tensor to every owned tensor of flat fp32 buffers (copies returned).

    ``owned`` is a boolean per tensor; other elements are left untouched.
    Returns (param, mom, bf16 bits of param (owned tensors only meaningful), deltas dict).
    """
    P = np.array(flat_param, dtype=np.float32, copy=True)
    M = np.array(flat_mom, dtype=np.float32, copy=True)
    B = bf16_rne(P)
    deltas = {}
    for i, (off, (r, c)) in enumerate(zip(offsets, shapes)):
        if not owned[i]:
            continue
        n = r * c
        sl = slice(off, off + n)
        Wn, mn, bn, d = muon_step_tensor(P[sl].reshape(r, c), np.asarray(flat_grad[sl]).reshape(r, c),
                                         M[sl].reshape(r, c), lr, mu, steps, coeffs, eps)
        P[sl] = Wn.reshape(-1)
        M[sl] = mn.reshape(-1)
        B[sl] = bn.reshape(-1)
        deltas[i] = d
    return P, M, B, deltas


def ns_flops(rows: int, cols: int, steps: int = 5) -> int:
    """Dense flop count of the three products per step: 2m^2 n + 2m^3 + 2m^2 n."""
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4 * m * m * n + 2 * m * m * m)
