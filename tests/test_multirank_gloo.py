"""The bench's multi-rank path on CPU: two processes over gloo (world size 2).

Each rank builds the workload, plans it with R = world (alpha-Balanced LPT), selects
its shard, and steps it; the Canzona optimizer step needs no collective (summary
page, section 3.4, "Runtime Static-Layout Enforcement": zero communication), so
the only collectives are the plan-agreement check and the bench's max-over-ranks
timing reduction.  On CPU the fp64 oracle stands in for the GPU step.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from oracle import muon as OM
    from zero_sharded_gb300 import cz
    from zero_sharded_gb300 import workloads as wl

    w, buckets, R, alpha, my_rank, _ = bench.build_workload("tiny", world, rank)
    assert R == world and my_rank == rank
    plan = cz.cz_plan_partition(w.numels, buckets, R, alpha)
    owner = torch.tensor(plan.owner(), dtype=torch.int32)
    gathered = [torch.zeros_like(owner) for _ in range(world)]
    dist.all_gather(gathered, owner)
    assert all(torch.equal(g, owner) for g in gathered), "ranks disagree on the plan"
    p, g, m = wl.make_state(w, seed=0)
    owned = [int(o) == rank for o in owner.tolist()]
    P, M, _, _ = OM.muon_step_flat(p.numpy(), g.numpy(), m.numpy(), w.offsets, w.shapes, owned, 0.02, 0.95)
    np.save(os.path.join(out_dir, f"P{rank}.npy"), P)
    np.save(os.path.join(out_dir, f"owner{rank}.npy"), owner.numpy())
    t = torch.tensor([float(rank + 1)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)            # the bench's max-over-ranks timing
    assert t.item() == float(world)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_over_gloo(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from oracle import muon as OM
    from zero_sharded_gb300 import workloads as wl

    w, buckets, R, alpha, _, _ = bench.build_workload("tiny", world, 0)
    owner = np.load(tmp_path / "owner0.npy")
    assert set(owner.tolist()) == {0, 1}                  # both ranks own tensors
    p, g, m = wl.make_state(w, seed=0)
    single, _, _, _ = OM.muon_step_flat(p.numpy(), g.numpy(), m.numpy(), w.offsets, w.shapes,
                                        [True] * len(w.shapes), 0.02, 0.95)
    per_rank = [np.load(tmp_path / f"P{r}.npy") for r in range(world)]
    for i, (off, (r, c)) in enumerate(zip(w.offsets, w.shapes)):
        sl = slice(off, off + r * c)
        o = int(owner[i])
        # the owner's result equals the single-rank result; the other rank left the tensor untouched
        assert np.array_equal(per_rank[o][sl], single[sl])
        assert np.array_equal(per_rank[1 - o][sl], p.numpy()[sl])


def _rsag_worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import comm as OC
    from zero_sharded_gb300 import comm
    from zero_sharded_gb300 import cz

    # one bucket of 5 tensors partitioned by Algorithm 1 over `world` ranks
    numels = [300, 1200, 64, 800, 16]
    plan = cz.cz_plan_partition(numels, [5], world, 1.0)
    _, ecuts = plan.cuts()
    cuts = ecuts[0]

    def pack(bucket, c, block, padded):
        padded.copy_(torch.from_numpy(OC.pack(bucket.numpy(), c, block)))

    def unpack(padded, c, block, bucket):
        bucket.copy_(torch.from_numpy(OC.unpack(padded.numpy(), c, block, bucket.numpy())))

    g = torch.Generator().manual_seed(100 + rank)
    grad = torch.randn(sum(numels), generator=g, dtype=torch.float64)
    shard = comm.reduce_scatter_bucket(grad, cuts, rank, pack=pack)
    np.save(os.path.join(out_dir, f"grad{rank}.npy"), grad.numpy())
    np.save(os.path.join(out_dir, f"shard{rank}.npy"), shard.numpy())
    # "updated" shard -> all-gather into the full bucket on every rank
    updated = shard * 2.0 + rank
    full = torch.full((sum(numels),), -1.0, dtype=torch.float64)
    comm.all_gather_bucket(updated, cuts, rank, full, unpack=unpack)
    np.save(os.path.join(out_dir, f"full{rank}.npy"), full.numpy())
    np.save(os.path.join(out_dir, "cuts.npy"), np.array(cuts))
    dist.barrier()
    dist.destroy_process_group()


def test_variable_size_reduce_scatter_all_gather_over_gloo(tmp_path):
    """The padded collective sequence reproduces the definitions: rank r receives the
    sum of all ranks' gradients over its interval, and the gathered bucket holds every
    rank's shard at its interval (shard sizes S_r differ per rank)."""
    from oracle import comm as OC

    world = 2
    mp.start_processes(_rsag_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    cuts = np.load(tmp_path / "cuts.npy").tolist()
    sizes = [cuts[r + 1] - cuts[r] for r in range(world)]
    assert len(set(sizes)) > 1                      # really variable-size
    grads = [np.load(tmp_path / f"grad{r}.npy") for r in range(world)]
    expect_full = np.empty(cuts[-1])
    for r in range(world):
        shard = np.load(tmp_path / f"shard{r}.npy")
        want = OC.reduce_scatter(grads, cuts, r)
        assert np.allclose(shard, want, rtol=0, atol=1e-12)
        expect_full[cuts[r]:cuts[r + 1]] = shard * 2.0 + r
    for r in range(world):
        assert np.array_equal(np.load(tmp_path / f"full{r}.npy"), expect_full)
