"""The Muon step inside a CUDA graph, through the C-ABI.

A call enqueued into a capturing stream records the same kernels with the same
launch parameters as an eager call (the step's tables are copied from the
program's page-locked image by a kernel, which a graph can replay), so replays
must give, step after step, what eager calls give, bit for bit.  What cannot be
captured (building a program, growing a workspace, a pageable upload) is refused
with CZ_ERR_INVALID before anything is enqueued.
"""

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

_CHILD = r"""
import json, sys, numpy as np, torch
from zero_sharded_gb300 import cz
from zero_sharded_gb300 import workloads as wl
shapes = [tuple(x) for x in json.loads(sys.argv[2])]
numels = [r * c for r, c in shapes]
offsets = list(np.cumsum([0] + numels[:-1]))
args = cz.StepArgs(offsets, shapes)
plan = cz.cz_plan_partition(numels, [len(shapes)], 1, 1.0)
ws_bytes = cz.cz_workspace_size(plan, 0, shapes)
p0 = wl.draw(shapes, 0.02, 61).cuda()
grads = [wl.draw(shapes, 1.0, 62 + k).cuda() for k in range(3)]
LR, MU = 0.02, 0.95


def state():
    return {"P": p0.clone(), "G": torch.zeros_like(p0), "M": torch.zeros_like(p0),
            "PB": torch.zeros(p0.numel(), dtype=torch.bfloat16, device="cuda"),
            "WS": torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")}


def call(st, stream):
    o = cz.make_opts(param_bf16=st["PB"], workspace=st["WS"], workspace_bytes=ws_bytes)
    cz.cz_muon_step_ex(plan, 0, st["P"], st["G"], st["M"], args, LR, MU, 5, stream, o)


# eager: three steps
e = state()
eager = []
s0 = torch.cuda.current_stream()
for k in range(3):
    e["G"].copy_(grads[k])
    call(e, s0)
    torch.cuda.synchronize()
    eager.append((e["P"].clone(), e["M"].clone(), e["PB"].clone()))

# graph: one call outside the capture builds the program, then the state is reset
g = state()
call(g, s0)
torch.cuda.synchronize()
g["P"].copy_(p0)
g["M"].zero_()
g["PB"].zero_()
built = cz.cz_step_programs_built()
graph = torch.cuda.CUDAGraph()
cap = torch.cuda.Stream()
cap.wait_stream(s0)
with torch.cuda.graph(graph, stream=cap):
    call(g, torch.cuda.current_stream())
same = []
for k in range(3):
    g["G"].copy_(grads[k])
    graph.replay()
    torch.cuda.synchronize()
    same.append([torch.equal(a, b) for a, b in zip((g["P"], g["M"], g["PB"]), eager[k])])
assert cz.cz_device_status(None, g["WS"]) == cz.CZ_OK
rebuilt = cz.cz_step_programs_built() - built

# a schedule through lr_device: eager calls with lr = 0.02, 0.01, 0.005 against replays of one capture
# that reads lr from device memory written before each replay
sched = [0.02, 0.01, 0.005]
e2 = state()
eager2 = []
for k, lr in enumerate(sched):
    e2["G"].copy_(grads[k])
    o = cz.make_opts(param_bf16=e2["PB"], workspace=e2["WS"], workspace_bytes=ws_bytes)
    cz.cz_muon_step_ex(plan, 0, e2["P"], e2["G"], e2["M"], args, lr, MU, 5, s0, o)
    torch.cuda.synchronize()
    eager2.append((e2["P"].clone(), e2["M"].clone(), e2["PB"].clone()))
lr_t = torch.full((1,), 123.0, device="cuda")     # the lr argument below is never used
h = state()
oh = cz.make_opts(param_bf16=h["PB"], workspace=h["WS"], workspace_bytes=ws_bytes, lr_device=lr_t)
cz.cz_muon_step_ex(plan, 0, h["P"], h["G"], h["M"], args, 9.0, MU, 5, s0, oh)
torch.cuda.synchronize()
h["P"].copy_(p0)
h["M"].zero_()
h["PB"].zero_()
graph3 = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph3, stream=cap):
    cz.cz_muon_step_ex(plan, 0, h["P"], h["G"], h["M"], args, 9.0, MU, 5, torch.cuda.current_stream(), oh)
same_sched = []
for k, lr in enumerate(sched):
    h["G"].copy_(grads[k])
    lr_t.fill_(lr)
    graph3.replay()
    torch.cuda.synchronize()
    same_sched.append([torch.equal(a, b) for a, b in zip((h["P"], h["M"], h["PB"]), eager2[k])])

# refused inside a capture: buffers without an eager call first
f = state()
refused = []
graph2 = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph2, stream=cap):
    try:
        call(f, torch.cuda.current_stream())
        refused.append(None)
    except cz.CzError as err:
        refused.append(err.status)
    f["P"].add_(0.0)      # keeps the captured graph non-empty
torch.cuda.synchronize()
json.dump({"same": same, "same_sched": same_sched, "rebuilt": rebuilt, "refused": refused,
           "invalid": cz.CZ_ERR_INVALID}, open(sys.argv[1], "w"))
"""


@pytest.mark.parametrize("fused", ["1", "0"])
def test_step_replayed_from_a_cuda_graph(tmp_path, fused):
    """Three replays of a captured step (new gradients copied in before each) equal three
    eager steps bit for bit (fp32 master, momentum, bf16 copy), with the fused launch and
    with one launch per product; a capture that reads lr from device memory follows a
    schedule written there before each replay, bit for bit as eager calls with those lr;
    capturing builds nothing; a first call for new buffers is refused inside a capture.  The
    shard mixes tiled matrices with on-chip ones of both kinds (one CTA, a CTA pair)."""
    shapes = [(64, 64), (96, 128), (384, 1024), (1024, 384), (300, 520), (200, 240)]
    f = tmp_path / f"graph_{fused}.json"
    env = dict(os.environ, CZ_NS_FUSED=fused)
    r = subprocess.run([sys.executable, "-c", _CHILD, str(f), json.dumps(shapes)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    d = json.loads(f.read_text())
    assert d["same"] == [[True, True, True]] * 3, d["same"]
    assert d["same_sched"] == [[True, True, True]] * 3, d["same_sched"]
    assert d["rebuilt"] == 0
    assert d["refused"] == [d["invalid"]], d["refused"]
