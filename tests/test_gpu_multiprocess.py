"""Two ranks as two processes, each stepping its own shard through the CUDA path.

Each process plans the same tensors with R = 2 (alpha-Balanced LPT), checks over a
gloo process group that both ranks hold the same partition, and runs
cz_muon_step_ex for its rank on the one GPU; the ranks' kernels never wait on one
another (the step needs no communication: summary page, section 3.4, "Runtime
Static-Layout Enforcement"), so sharing the GPU is safe.  Merging each tensor
from its owner must give, bit for bit, what one process stepping every tensor
(R = 1) gives, and a rank must leave the tensors it does not own untouched.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from zero_sharded_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPES = [(384, 1024), (1024, 384), (256, 256), (128, 640), (640, 640), (64, 192), (300, 520)]
LR, MU = 0.02, 0.95


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layout():
    numels = [r * c for r, c in SHAPES]
    offsets = [int(x) for x in np.cumsum([0] + numels[:-1])]
    return numels, offsets


def _state():
    P = wl.draw(SHAPES, 0.02, 61)
    G = wl.draw(SHAPES, 1.0, 62)
    return P, G


def _rank(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from zero_sharded_gb300 import cz

    numels, offsets = _layout()
    plan = cz.cz_plan_partition(numels, [len(SHAPES)], world, 1.0)
    owner = torch.tensor(plan.owner(), dtype=torch.int32)
    got = [torch.zeros_like(owner) for _ in range(world)]
    dist.all_gather(got, owner)
    assert all(torch.equal(g, owner) for g in got), "ranks disagree on the plan"
    torch.cuda.set_device(0)
    P0, G0 = _state()
    P, G = P0.cuda(), G0.cuda()
    M = torch.zeros_like(P)
    PB = torch.zeros(P.numel(), dtype=torch.bfloat16, device="cuda")
    args = cz.StepArgs(offsets, SHAPES)
    for _ in range(2):
        cz.cz_muon_step_ex(plan, rank, P, G, M, args, LR, MU, 5, None, cz.make_opts(param_bf16=PB))
    assert cz.cz_device_status(None, None) == cz.CZ_OK
    torch.save({"P": P.cpu(), "M": M.cpu(), "PB": PB.cpu(), "owner": owner}, os.path.join(out_dir, f"r{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


def test_two_processes_step_their_shards_like_one():
    import tempfile

    from zero_sharded_gb300 import cz

    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank, args=(world, _free_port(), d), nprocs=world, start_method="spawn")
        parts = [torch.load(os.path.join(d, f"r{r}.pt")) for r in range(world)]
    owner = parts[0]["owner"].tolist()
    assert set(owner) == {0, 1}                         # both ranks own tensors
    numels, offsets = _layout()
    plan = cz.cz_plan_partition(numels, [len(SHAPES)], 1, 1.0)
    P0, G0 = _state()
    P, G = P0.cuda(), G0.cuda()
    M = torch.zeros_like(P)
    PB = torch.zeros(P.numel(), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        cz.cz_muon_step_ex(plan, 0, P, G, M, cz.StepArgs(offsets, SHAPES), LR, MU, 5, None,
                           cz.make_opts(param_bf16=PB))
    assert cz.cz_device_status(None, None) == cz.CZ_OK
    P, M, PB = P.cpu(), M.cpu(), PB.cpu()
    for i, (off, n) in enumerate(zip(offsets, numels)):
        sl = slice(off, off + n)
        own, other = parts[owner[i]], parts[1 - owner[i]]
        assert torch.equal(own["P"][sl], P[sl]), i
        assert torch.equal(own["M"][sl], M[sl]), i
        assert torch.equal(own["PB"][sl], PB[sl]), i
        assert torch.equal(other["P"][sl], P0[sl]), i          # the other rank left it untouched
        assert torch.equal(other["M"][sl], torch.zeros(n)), i
