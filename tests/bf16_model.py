"""A NumPy model of where the GPU path rounds to bf16 (test helper, no CUDA).

The fp64 oracle (oracle/muon.py) is what the method computes; this model is the
same Newton-Schulz iteration with the design's storage precisions applied at
the same points as the kernels:

* X~ = bf16(u) in the m x n orientation; s = 1 / (||u||_F + eps) in fp32;
* per step: A = bf16(s^2 * fp32(X X^T)) (s^2 in step 1 only),
  B' = bf16(b*A + c*fp32(A A) + a*I), X = bf16(s * fp32(B' X)) (s in step 1 only);
  the last X stays fp32 (the apply epilogue consumes the accumulator).

Products are formed in fp64 and rounded to fp32, which stands in for the tensor
cores' fp32 accumulation (the summation order differs, so agreement with the
GPU is close but not bitwise).  Its use: for inputs where bf16 storage alone
moves the result by more than the 2e-2 bar (the quintic map amplifies rounding
where a singular value passes near 1.2, f'(1.2) ~ 3.9), the tests bound the GPU
by the model's own distance from the fp64 oracle instead of by the bar.
"""

from __future__ import annotations

import numpy as np

from oracle import muon as OM


def _bf(x, rounding=True):
    if not rounding:
        return np.asarray(x, np.float64)
    return OM.bf16_to_f32(OM.bf16_rne(np.asarray(x, np.float32))).astype(np.float32)


def orthogonalise_bf16(u, steps, coeffs=OM.QUINTIC, eps=OM.EPS, rounding=True):
    """X_K in the tensor's rows x cols layout, as the GPU path stores it (fp32 values)."""
    a, b, c = (np.float32(v) for v in coeffs)
    u = np.asarray(u, np.float64)
    tall = u.shape[0] > u.shape[1]
    u32 = u.astype(np.float32)
    if rounding:
        sg = np.float32(1.0) / (np.float32(np.sqrt(np.sum(u32.astype(np.float64) ** 2))) + np.float32(eps))
    else:
        sg = 1.0 / (np.sqrt(np.sum(u * u)) + eps)
    X = _bf((u32.T if tall else u32) if rounding else (u.T if tall else u), rounding)
    f = (lambda y: y.astype(np.float32)) if rounding else (lambda y: y)
    one = np.float32(1.0) if rounding else 1.0
    for t in range(steps):
        s2 = sg * sg if t == 0 else one
        A = _bf(f(X.astype(np.float64) @ X.T.astype(np.float64)) * s2, rounding)
        P = f(A.astype(np.float64) @ A.astype(np.float64))
        B = _bf(b * A + c * P + a * np.eye(A.shape[0], dtype=np.float32), rounding) if rounding else \
            float(coeffs[1]) * A + float(coeffs[2]) * P + float(coeffs[0]) * np.eye(A.shape[0])
        s = sg if t == 0 else one
        Y = f(B.astype(np.float64) @ X.astype(np.float64)) * s
        X = Y if (t + 1 == steps or not rounding) else _bf(Y)
    return np.asarray(X.T if tall else X, np.float64)
