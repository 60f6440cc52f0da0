"""Oracle for the variable-size collectives around the step (test infrastructure only).

Summary page "Canzona: ...", section 3.4, "Runtime Static-Layout Enforcement":
bucket B_i is reduce-scattered and all-gathered with per-rank sizes
S_{i,r} = s_{i,r} - s_{i,r-1} (element cuts of the partition map).  Written as the
plain definitions: the padded layout (R blocks of `block` elements), and the
reduce-scatter result as a sum of slices.
"""

from __future__ import annotations

import numpy as np


def pack(bucket, elem_cuts, block):
    R = len(elem_cuts) - 1
    out = np.zeros(R * block, dtype=np.asarray(bucket).dtype)
    for r in range(R):
        lo, hi = int(elem_cuts[r]), int(elem_cuts[r + 1])
        out[r * block:r * block + (hi - lo)] = bucket[lo:hi]
    return out


def unpack(padded, elem_cuts, block, bucket):
    out = np.array(bucket, copy=True)
    for r in range(len(elem_cuts) - 1):
        lo, hi = int(elem_cuts[r]), int(elem_cuts[r + 1])
        out[lo:hi] = padded[r * block:r * block + (hi - lo)]
    return out


def reduce_scatter(buckets, elem_cuts, rank):
    """Rank `rank`'s interval of the element-wise sum of every rank's bucket."""
    lo, hi = int(elem_cuts[rank]), int(elem_cuts[rank + 1])
    acc = np.zeros(hi - lo, dtype=np.float64)
    for b in buckets:
        acc += np.asarray(b[lo:hi], dtype=np.float64)
    return acc
