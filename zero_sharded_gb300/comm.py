"""Variable-size Reduce-Scatter / All-Gather of a bucket under a partition map.

Canzona summary page, section 3.4, "Runtime Static-Layout Enforcement": gradients
of bucket B_i are reduce-scattered so that rank r receives exactly its interval
[s_{i,r-1}, s_{i,r}) (S_{i,r} elements), and after the step the updated shards are
all-gathered back into the full bucket.  Collectives with equal counts per rank
(NCCL ReduceScatter / AllGather) are used on R blocks of max_r S_{i,r} elements;
the libcz kernels cz_bucket_pack / cz_bucket_unpack move the bucket into and out
of that padded layout.

`pack` / `unpack` default to those device kernels; they are parameters only so
that a test can run the same collective sequence with another implementation of
the same copy contract.
"""

from __future__ import annotations

from typing import Callable, Optional, Sequence

import torch
import torch.distributed as dist

from . import cz


def _block(elem_cuts: Sequence[int], elem_bytes: int) -> int:
    """max_r S_r rounded up to 16 bytes, so every block starts 16-byte aligned."""
    m = max(int(elem_cuts[r + 1]) - int(elem_cuts[r]) for r in range(len(elem_cuts) - 1))
    q = max(1, 16 // elem_bytes)
    return max(q, (m + q - 1) // q * q)


def reduce_scatter_bucket(bucket: torch.Tensor, elem_cuts: Sequence[int], rank: int, group=None,
                          pack: Optional[Callable] = None) -> torch.Tensor:
    """Sum of every rank's `bucket` restricted to this rank's interval (S_r elements)."""
    pack = pack or cz.cz_bucket_pack
    R = len(elem_cuts) - 1
    block = _block(elem_cuts, bucket.element_size())
    padded = torch.empty(R * block, dtype=bucket.dtype, device=bucket.device)
    pack(bucket, elem_cuts, block, padded)
    out = torch.empty(block, dtype=bucket.dtype, device=bucket.device)
    dist.reduce_scatter_tensor(out, padded, op=dist.ReduceOp.SUM, group=group)
    return out[: int(elem_cuts[rank + 1]) - int(elem_cuts[rank])]


def all_gather_bucket(shard: torch.Tensor, elem_cuts: Sequence[int], rank: int, bucket_out: torch.Tensor,
                      group=None, unpack: Optional[Callable] = None) -> None:
    """Writes every rank's shard into its interval of `bucket_out`."""
    unpack = unpack or cz.cz_bucket_unpack
    R = len(elem_cuts) - 1
    block = _block(elem_cuts, shard.element_size())
    n = int(elem_cuts[rank + 1]) - int(elem_cuts[rank])
    if shard.numel() != n:
        raise ValueError(f"shard has {shard.numel()} elements, the plan gives rank {rank} {n}")
    mine = torch.zeros(block, dtype=shard.dtype, device=shard.device)
    mine[:n] = shard
    gathered = torch.empty(R * block, dtype=shard.dtype, device=shard.device)
    dist.all_gather_into_tensor(gathered, mine, group=group)
    unpack(gathered, elem_cuts, block, bucket_out)
