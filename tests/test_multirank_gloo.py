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

    w, buckets, R, alpha, my_rank = bench.build_workload("tiny", world, rank)
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

    w, buckets, R, alpha, _ = bench.build_workload("tiny", world, 0)
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
