"""Bucket pack/unpack kernels (variable-size collectives around the step) against the oracle.

Pure data movement: bit-exact for every element width; plus the NCCL helper on a
single-rank process group.
"""

import numpy as np
import pytest
import torch

from oracle import comm as OC
from zero_sharded_gb300 import cz

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.uint8, torch.int64])
def test_pack_unpack_bit_exact(dtype):
    rng = np.random.default_rng(0)
    for R in (1, 2, 3, 8, 33):
        sizes = rng.integers(0, 5000, size=R)
        cuts = [0] + np.cumsum(sizes).tolist()
        block = int(max(sizes.max(), 1)) + int(rng.integers(0, 3))
        n = cuts[-1]
        if dtype.is_floating_point:
            bucket = torch.randn(max(n, 1), generator=torch.Generator().manual_seed(R)).to(dtype)[:n]
        else:
            bucket = torch.randint(0, 120, (n,), generator=torch.Generator().manual_seed(R)).to(dtype)
        raw = bucket.view(torch.uint8 if dtype == torch.uint8 else {2: torch.int16, 4: torch.int32, 8: torch.int64}[bucket.element_size()])
        bd = bucket.cuda()
        padded = torch.full((R * block,), 7, dtype=dtype, device="cuda")
        cz.cz_bucket_pack(bd, cuts, block, padded)
        torch.cuda.synchronize()
        want = OC.pack(raw.numpy(), cuts, block)
        got = padded.cpu().view(raw.dtype).numpy()
        assert np.array_equal(got, want)
        out = torch.zeros_like(bd)
        cz.cz_bucket_unpack(padded, cuts, block, out)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(raw.dtype), raw)


def test_pack_rejects_bad_layouts():
    b = torch.zeros(10, device="cuda")
    p = torch.zeros(20, device="cuda")
    for cuts, block in (([1, 10], 10), ([0, 6, 4], 10), ([0, 6, 10], 5)):
        with pytest.raises(cz.CzError):
            cz.cz_bucket_pack(b, cuts, block, p)


def test_nccl_single_rank_reduce_scatter_all_gather(tmp_path):
    import torch.distributed as dist

    from zero_sharded_gb300 import comm

    dist.init_process_group("nccl", init_method=f"file://{tmp_path}/store", rank=0, world_size=1)
    try:
        bucket = torch.randn(4321, device="cuda")
        cuts = [0, 4321]
        shard = comm.reduce_scatter_bucket(bucket, cuts, 0)
        assert torch.equal(shard, bucket)
        out = torch.zeros_like(bucket)
        comm.all_gather_bucket(shard * 2, cuts, 0, out)
        assert torch.equal(out, bucket * 2)
    finally:
        dist.destroy_process_group()
