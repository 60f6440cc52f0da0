"""Pins of the variable-size collective oracle (oracle/comm.py), on the CPU.

Summary page "Canzona: ...", section 3.4, "Runtime Static-Layout Enforcement": a
bucket is reduce-scattered and all-gathered with per-rank sizes S_r = s_r - s_{r-1}
taken from the partition map's element cuts.  With equal-count collectives the
bucket travels as R blocks of max_r S_r elements; the pins below fix that layout
by hand-worked values and by the identity the padded collectives rely on.
"""

import numpy as np
import pytest

from oracle import comm as OC


def test_pack_unpack_hand_worked():
    bucket = np.arange(10, 20, dtype=np.float32)          # 10 elements
    cuts = [0, 3, 7, 10]                                  # S = 3, 4, 3
    block = 4                                             # max_r S_r
    packed = OC.pack(bucket, cuts, block)
    assert packed.tolist() == [10, 11, 12, 0, 13, 14, 15, 16, 17, 18, 19, 0]
    back = OC.unpack(packed, cuts, block, np.full(10, -1.0, np.float32))
    assert back.tolist() == bucket.tolist()


def test_reduce_scatter_hand_worked():
    b0 = np.array([1, 2, 3, 4], np.float32)
    b1 = np.array([10, 20, 30, 40], np.float32)
    cuts = [0, 1, 4]
    assert OC.reduce_scatter([b0, b1], cuts, 0).tolist() == [11]
    assert OC.reduce_scatter([b0, b1], cuts, 1).tolist() == [22, 33, 44]


def test_empty_shard_and_padding_stay_zero():
    bucket = np.array([5, 6, 7], np.int64)
    cuts = [0, 0, 3, 3]                                   # ranks 0 and 2 own nothing
    packed = OC.pack(bucket, cuts, 3)
    assert packed.tolist() == [0, 0, 0, 5, 6, 7, 0, 0, 0]
    assert OC.reduce_scatter([bucket], cuts, 0).size == 0
    assert OC.unpack(packed, cuts, 3, np.zeros(3, np.int64)).tolist() == [5, 6, 7]


@pytest.mark.parametrize("seed", range(20))
def test_padded_collectives_equal_the_variable_size_ones(seed):
    """Summing every rank's packed bucket and reading block r gives rank r's
    reduce-scatter result; unpacking every rank's block restores the whole bucket
    (the all-gather).  Brute force over random cuts, including empty shards."""
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 7))
    n = int(rng.integers(0, 60))
    cuts = [0] + sorted(int(x) for x in rng.integers(0, n + 1, R - 1)) + [n]
    block = max(1, max(cuts[r + 1] - cuts[r] for r in range(R)))
    buckets = [rng.standard_normal(n) for _ in range(R)]
    summed = sum(OC.pack(b, cuts, block) for b in buckets)
    for r in range(R):
        S = cuts[r + 1] - cuts[r]
        assert np.allclose(summed[r * block:r * block + S], OC.reduce_scatter(buckets, cuts, r), rtol=0, atol=1e-12)
        assert not np.any(summed[r * block + S:(r + 1) * block])          # padding stays zero
    gathered = OC.unpack(summed, cuts, block, np.zeros(n))
    assert np.allclose(gathered, sum(buckets), rtol=0, atol=1e-12)
