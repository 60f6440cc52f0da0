#!/usr/bin/env python
"""Bench of the local Muon step one data-parallel rank runs on its shard.

Default workload: the heaviest rank's shard of a Qwen3-32B-shaped model (64
layers laid out in reverse layer order in 40,000,000-element buckets, planned by
the alpha-Balanced Greedy LPT planner with R = 32, alpha = 1, cost = numel): 8
FFN matrices of 5120 x 25600 (gate/up 25600 x 5120, down 5120 x 25600),
1,048,576,000 elements, fp32 master/momentum/gradients, bf16 parameter copy,
mu = 0.95 Nesterov, lr = 0.02, 5 quintic Newton-Schulz steps.  Other workloads:
`--workload` (the tiny six-matrix case, one Qwen3-1.7B-shaped layer, 28 such
layers, the 64-matrix Qwen3-14B micro-group, and the shards of the FLOPs-cost
comparison).  Under torchrun with N ranks each GPU steps its own shard (the k-th
heaviest of the R = 32 plan for the Qwen3-32B shard; a layer of N layers planned
with R = N otherwise) with no collective inside the step (weak scaling).

Prints ONE JSON line (rank 0).  `value` is the slowest rank's mean step time in
milliseconds (weak scaling: a flat value over N is perfect scaling);
`ms_per_shard_job` divides it by the number of shards.

`--compare-cost` instead times every distinct shard of the Qwen3-32B layout under
the numel-cost plan and under the Newton-Schulz-FLOPs-cost plan and prints one
JSON line with each plan's slowest shard (the step is communication-free, so the
slowest shard sets the distributed optimizer step).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon step ms per shard; Newton-Schulz TFLOP/s and % of GB300 bf16 peak"
LR, MU, NS_STEPS = 0.02, 0.95, 5
BUCKET_CAP = 40_000_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def ns_flops(shapes, steps=NS_STEPS):
    """Dense flops of the three products per Newton-Schulz step: 2m^2n + 2m^3 + 2m^2n."""
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        tot += steps * (4 * m * m * n + 2 * m * m * m)
    return tot


SMALL_M, SMALL_N = 128, 256     # matrices whose Newton-Schulz steps run on chip in one CTA (ns_small)
SMALL_PAIR_M = 256              # ... and on a CTA pair, m up to this (the ns_small kind too)


def _is_small(r, c):
    return min(r, c) <= SMALL_PAIR_M and max(r, c) <= SMALL_N


def ns_flops_by_kind(shapes, steps=NS_STEPS):
    """Algorithmic flops per step of each GEMM kernel kind (the product each launch computes)."""
    tiled = [s for s in shapes if not _is_small(*s)]
    small = [s for s in shapes if _is_small(*s)]
    g = sum(2 * min(r, c) ** 2 * max(r, c) for r, c in tiled)
    p = sum(2 * min(r, c) ** 3 for r, c in tiled)
    gs = sum(2 * min(r, c) ** 2 * max(r, c) for r, c in small)
    ps = sum(2 * min(r, c) ** 3 for r, c in small)
    return {"ns_gram": steps * g, "ns_poly": steps * p, "ns_update": (steps - 1) * g, "ns_update_apply": g,
            "ns_fused": steps * (2 * g + p), "ns_small": steps * (2 * gs + ps)}


def ns_flops_executed(shapes, steps=NS_STEPS, bn=256):
    """Flops the tensor cores execute: 256x256 tiles on CTA pairs (128x256 with CZ_NS_PAIR=0), symmetric
    products on the tiles touching the upper triangle only; on-chip small matrices as 128-row products
    with n padded to 64 (one CTA, m <= 128) or as 256 x 256 x 256 products (a CTA pair)."""
    bm = 128 if os.environ.get("CZ_NS_PAIR", "1") == "0" else 256

    def cdiv(a, b):
        return (a + b - 1) // b
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        if _is_small(r, c) and m <= SMALL_M:
            n_pad = cdiv(n, 64) * 64
            tot += steps * (2 * 128 * 128 * n_pad + 2 * 128 * 128 * 128 + 2 * 128 * n_pad * 128)
            continue
        if _is_small(r, c):
            tot += steps * 3 * 2 * SMALL_PAIR_M ** 3
            continue
        sym = sum(1 for a in range(cdiv(m, bm)) for b in range(cdiv(m, bn)) if a * bm <= b * bn + bn - 1)
        kpad_n, kpad_m = cdiv(n, 64) * 64, cdiv(m, 64) * 64
        gram = sym * 2 * bm * bn * kpad_n
        poly = sym * 2 * bm * bn * kpad_m
        upd = cdiv(m, bm) * cdiv(n, bn) * 2 * bm * bn * kpad_m
        tot += steps * (gram + poly + upd)
    return tot


def ns_flops_executed_by_kind(shapes, steps=NS_STEPS, bn=256):
    """Executed flops per step of each GEMM kernel kind, counted as ns_flops_executed counts them."""
    bm = 128 if os.environ.get("CZ_NS_PAIR", "1") == "0" else 256

    def cdiv(a, b):
        return (a + b - 1) // b
    g = p = u = 0
    for r, c in shapes:
        if _is_small(r, c):
            continue
        m, n = min(r, c), max(r, c)
        sym = sum(1 for a in range(cdiv(m, bm)) for b in range(cdiv(m, bn)) if a * bm <= b * bn + bn - 1)
        g += sym * 2 * bm * bn * cdiv(n, 64) * 64
        p += sym * 2 * bm * bn * cdiv(m, 64) * 64
        u += cdiv(m, bm) * cdiv(n, bn) * 2 * bm * bn * cdiv(m, 64) * 64
    small = ns_flops_executed([s for s in shapes if _is_small(*s)], steps)
    return {"ns_gram": steps * g, "ns_poly": steps * p, "ns_update": (steps - 1) * u, "ns_update_apply": u,
            "ns_fused": steps * (g + p + u), "ns_small": small}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu captures summarised
# under profiles/, per kernel kind, keyed by a hash of the sources that kernel is built and launched from:
# once one of them changes the figure no longer describes the kernel and the bench reports null.
STEP_SOURCES = ["muon_step.cpp", "fused_schedule.h", "ptx.cuh", "step_kernels.h", "cz_internal.h"]
KERNEL_SOURCES = {
    "ns_gemm": ["ns_gemm.cu"] + STEP_SOURCES,
    "momentum": ["momentum.cu"] + STEP_SOURCES,
    "ns_small": ["ns_small.cu", "ns_small_pair.cu"] + STEP_SOURCES,
    "apply": ["apply.cu"],
}
KIND_SOURCE = {"ns_fused": "ns_gemm", "ns_gram": "ns_gemm", "ns_poly": "ns_gemm", "ns_update": "ns_gemm",
               "ns_update_apply": "ns_gemm", "momentum": "momentum", "ns_small": "ns_small", "apply": "apply"}
NCU_TRAFFIC = {
    # kernel source group: (source hash, {workload: {kind: bytes per launch}})
    "ns_gemm": ("ed6e332a2132d77b", {"qwen3-1.7b-layer": {"ns_fused": 2609.48e6},
                                     "qwen3-32b-R32-shard4": {"ns_gram": 5905.45e6, "ns_poly": 993.78e6,
                                                              "ns_update": 11097.07e6, "ns_update_apply": 24284.40e6}}),
    "momentum": ("abb7cc086cbae0af", {"qwen3-1.7b-layer": {"momentum": 648.84e6},
                                      "qwen3-32b-R32-shard4": {"momentum": 14626.10e6}}),
    # the tiny workload's two on-chip launches per step (one CTA: 0.342 MB, CTA pair: 0.448 MB), averaged
    "ns_small": ("b100f296afbd2642", {"tiny": {"ns_small": 0.3950e6}}),
    "apply": ("a6d9356fa7fabfff", {"qwen3-1.7b-layer": {"apply": 649.76e6}}),
}


def kernel_source_hash(group: str) -> str:
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES[group]:
        h.update(name.encode())
        with open(os.path.join(ROOT, "zero_sharded_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kind: str):
    """Bytes per launch from the committed ncu captures, or None if the kernel changed since."""
    group = KIND_SOURCE.get(kind)
    if group is None:
        return None
    digest, table = NCU_TRAFFIC[group]
    if digest != kernel_source_hash(group):
        return None
    return table.get(workload, {}).get(kind)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ workloads
WORKLOADS = ["qwen3-32b-shard", "qwen3-1.7b-layer", "tiny", "qwen3-1.7b-28L", "qwen3-14b-microgroup",
             "qwen3-32b-shard-flops", "qwen3-32b-shard-numel-maxflops", "qwen3-32b-ffn-pair", "qwen3-14b-ffn-pair"]
DEFAULT_WORKLOAD = "qwen3-32b-shard"
QWEN32_LAYOUT = "qwen3-32b 64 layers in reverse layer order, 448 tensors, 320 buckets of >= 40M elements"


def plan_owner_load(numels, buckets, R, alpha, costs=None, planner="cz"):
    """Algorithm 1's owner per tensor and load per rank.  The GPU arm plans through libcz; the reference
    arm, which runs no code of the CUDA library, through the oracle's planner (bit-exact with libcz's)."""
    if planner == "oracle":
        from oracle import planner as OP

        p = OP.plan_partition(numels, buckets, R, alpha, costs)
        return list(p.owner), list(p.rank_load)
    from zero_sharded_gb300 import cz

    if costs is None:
        p = cz.cz_plan_partition(numels, buckets, R, alpha)
    else:
        p = cz.cz_plan_partition_cost(numels, costs, buckets, R, alpha)
    return p.owner(), p.rank_load()


def make_buckets(numels, cap, planner="cz"):
    if planner == "oracle":
        from oracle import planner as OP

        return OP.make_buckets(numels, cap)
    from zero_sharded_gb300 import cz

    return cz.cz_make_buckets(numels, cap)


def qwen32_plan(cost: str, planner="cz"):
    """The 64-layer Qwen3-32B layout planned by Algorithm 1 (R = 32, alpha = 1) with W(p) = numel ("numel")
    or W(p) = the tensor's Newton-Schulz flops K(4m^2n + 2m^3) ("flops").  Returns (layout, owner, load)."""
    from zero_sharded_gb300 import workloads as wl

    full = wl.qwen3_32b_reverse()
    b = make_buckets(full.numels, full.bucket_cap, planner)
    costs = None if cost == "numel" else [ns_flops([s]) for s in full.shapes]
    own, load = plan_owner_load(full.numels, b, full.R, full.alpha, costs, planner)
    return full, own, load


def shard_of(full, owner, r: int, name: str):
    """Plan rank r's tensors of the layout, in buffer order, as a workload of their own."""
    from zero_sharded_gb300 import workloads as wl

    shapes = [s for s, o in zip(full.shapes, owner) if o == r]
    names = [n for n, o in zip(full.names, owner) if o == r]
    return wl.Workload(name, shapes, names, full.param_std, full.grad_std)


def build_workload(name: str, world: int, rank: int, planner="cz"):
    """Returns (workload, buckets, R, alpha, plan rank this GPU runs, config extras)."""
    from zero_sharded_gb300 import workloads as wl

    if name == "qwen3-1.7b-layer":
        w = wl.qwen3_1p7b_layers(world)
        buckets = make_buckets(w.numels, BUCKET_CAP, planner) if world > 1 else [len(w.numels)]
        return w, buckets, world, 1.0, rank, {"R": world, "alpha": 1.0}
    if name == "tiny":
        # one copy of the six tiny matrices per rank, one bucket per copy, planned with R = world
        base = wl.tiny()
        w = wl.Workload("tiny-6" if world == 1 else f"tiny-6x{world}", base.shapes * world,
                        [f"r{k}.{n}" for k in range(world) for n in base.names], base.param_std, base.grad_std)
        return w, [len(base.shapes)] * world, world, 1.0, rank, {"R": world, "alpha": 1.0}
    if name == "qwen3-32b-ffn-pair":
        # one up (25600 x 5120, tall) and one down (5120 x 25600, wide) matrix of the Qwen3-32B shard: the
        # headline shard's kernels at its shapes on a few GB of device memory (profiling captures)
        w = wl.Workload("qwen3-32b-ffn-pair", [(25600, 5120), (5120, 25600)], ["up", "down"], 0.02, 1e-3)
        return w, [2], 1, 1.0, 0, {"R": 1, "alpha": 1.0}
    if name == "qwen3-14b-ffn-pair":
        # one gate/up (17408 x 5120, tall) and one down (5120 x 17408, wide) matrix of the Qwen3-14B shapes, bf16
        # gradients as in the micro-group: its FFN kernels at their shapes on a few GB (profiling captures)
        w = wl.Workload("qwen3-14b-ffn-pair", [(17408, 5120), (5120, 17408)], ["up", "down"], 0.02, 1e-3,
                        grad_bf16=True)
        return w, [2], 1, 1.0, 0, {"R": 1, "alpha": 1.0}
    if name == "qwen3-1.7b-28L":
        w = wl.qwen3_1p7b_layers(28)
        return w, [len(w.numels)], 1, 1.0, 0, {"R": 1, "alpha": 1.0}
    if name == "qwen3-14b-microgroup":
        w = wl.qwen3_14b_microgroup(64)
        return w, [len(w.numels)], 1, 1.0, 0, {"R": 1, "alpha": 1.0}
    if name in ("qwen3-32b-shard", "qwen3-32b-shard-flops", "qwen3-32b-shard-numel-maxflops"):
        # plan the whole 64-layer model with R = 32, then run one rank's tensors on this GPU
        cost = "flops" if name == "qwen3-32b-shard-flops" else "numel"
        full, own, plan_load = qwen32_plan(cost, planner)
        if name == "qwen3-32b-shard-numel-maxflops":
            # the numel plan's rank with the most Newton-Schulz flops (its slowest rank)
            fl = [0] * full.R
            for s, o in zip(full.shapes, own):
                fl[o] += ns_flops([s])
            load, what = fl, "the most Newton-Schulz flops under the numel plan"
        else:
            load = plan_load
            what = "the heaviest planned load" + (" (cost = Newton-Schulz flops)" if cost == "flops" else "")
        order = sorted(range(full.R), key=lambda r: (-load[r], r))
        r = order[rank % full.R]        # GPU rank k runs the k-th heaviest plan rank
        tag = {"qwen3-32b-shard": "", "qwen3-32b-shard-flops": "flopscost-",
               "qwen3-32b-shard-numel-maxflops": "numel-maxflops-"}[name]
        w = shard_of(full, own, r, f"qwen3-32b-R32-{tag}shard{r}")
        extras = {"R": full.R, "alpha": full.alpha, "cost": cost, "plan_rank": r,
                  "planned_from": f"{QWEN32_LAYOUT}; Algorithm 1 with R = 32, alpha = 1, W(p) = {cost}; "
                                  f"plan rank {r}" + (f", {what}" if rank == 0 else f", the {rank + 1}-th by load")}
        return w, [len(w.shapes)], 1, 1.0, 0, extras
    raise SystemExit(f"unknown workload {name}")


# ------------------------------------------------------------------ clocks
REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock and clock-event reasons, read (never set) while the bench runs.

    Preferred: NVML through ctypes, polled every 2 ms in a thread, so that the samples fall inside the
    timed region (mark_begin / mark_end bracket it; the summary keeps the samples between the marks).
    Fallback when NVML cannot be loaded: `nvidia-smi -lms 200` for the whole sampler lifetime."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        self.samples = []              # (time, sm MHz, reason bits)
        self.t_begin = self.t_end = None
        self.nvml = None
        self.thread = None
        self.stop_flag = False
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                raise OSError("handle")
            mx = ctypes.c_uint(0)
            lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx))   # NVML_CLOCK_SM
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nvml = (ctypes, lib, h, reasons)
            self.max_mhz = float(mx.value)
        except Exception:
            self.nvml = None

    def _poll(self):
        ctypes, lib, h, reasons = self.nvml
        mhz = ctypes.c_uint(0)
        bits = ctypes.c_ulonglong(0)
        while not self.stop_flag:
            ok = lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(1), ctypes.byref(mhz)) == 0
            ok = ok and reasons(h, ctypes.byref(bits)) == 0
            if ok:
                self.samples.append((time.perf_counter(), float(mhz.value), int(bits.value)))
            time.sleep(0.002)

    def start(self):
        if self.nvml is not None:
            import threading
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark_begin(self):
        self.t_begin = time.perf_counter()

    def mark_end(self):
        self.t_end = time.perf_counter()

    def stop(self):
        if self.nvml is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            rows = self.samples
            if self.t_begin is not None and self.t_end is not None:
                inside = [r for r in rows if self.t_begin <= r[0] <= self.t_end]
                if inside:
                    rows = inside
            if not rows:
                return None
            reasons = sorted({nm for _, _, b in rows for bit, nm in REASON_BITS.items() if b & bit})
            return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(rows), "source": "nvml, 2 ms polls inside the timed region"}
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for _, _, flags in rows:
            for nm, fl in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), flags):
                if fl.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "source": "nvidia-smi -lms 200"}


# ------------------------------------------------------------------ CPU oracle timing
def torch_library_step(P, G, M, shapes, offsets, lr=LR, mu=MU, steps=NS_STEPS, coeffs=(3.4445, -4.7750, 2.0315),
                       eps=1e-7):
    """The same Muon step written with PyTorch library calls, for comparison only (never the product
    path): fp32 momentum as elementwise ops, the Frobenius norm with torch.linalg, Newton-Schulz in bf16
    with batched torch.matmul (cuBLAS) per shape group, the apply in fp32."""
    import torch

    a, b, c = coeffs
    groups = {}
    for off, (r, cc) in zip(offsets, shapes):
        groups.setdefault((min(r, cc), max(r, cc)), []).append((off, r, cc))
    M.mul_(mu).add_(G)
    U = G + mu * M
    for (m, n), items in groups.items():
        xs = []
        for off, r, cc in items:
            u = U[off:off + r * cc].view(r, cc)
            xs.append(u.t() if r > cc else u)
        X32 = torch.stack(xs)
        X = (X32 / (torch.linalg.vector_norm(X32, dim=(1, 2), keepdim=True) + eps)).to(torch.bfloat16)
        for _ in range(steps):
            A = X @ X.mT
            B = b * A + c * (A @ A)
            X = a * X + B @ X
        for k, (off, r, cc) in enumerate(items):
            xk = X[k].float()
            P[off:off + r * cc].view(r, cc).sub_((xk.t() if r > cc else xk), alpha=lr * max(1.0, r / cc) ** 0.5)


ORACLE_WHOLE_FLOPS = 3e12   # shards up to this much Newton-Schulz work are timed whole (about 10 s of fp64)


def time_oracle_sample(shapes, grad_std, seed=0):
    """Times the fp64 oracle, as it stands, on the shard or on a bounded sample of it.

    A shard with at most ORACLE_WHOLE_FLOPS of Newton-Schulz work (the tiny workload, the Qwen3-1.7B layer) is
    timed whole, every tensor through `muon_step_tensor`.  A larger one is sampled per Newton-Schulz shape class
    (m = min, n = max of rows/cols; a tall tensor costs the oracle what its transpose does): one tensor of the
    class runs `muon_step_tensor` with one Newton-Schulz step (momentum, normalisation, one step, scale, apply,
    bf16 copy) and then one more `newton_schulz` step on an m x n iterate, so that the tensor's time is the first
    plus (K - 1) times the second, extrapolated by the class's multiplicity.
    Returns (ms_per_step, sample_desc, cores)."""
    import numpy as np

    from oracle import muon as OM

    flops = sum(ns_flops([s]) for s in shapes)
    rng = np.random.default_rng(seed)
    if flops <= ORACLE_WHOLE_FLOPS:
        total_ms = 0.0
        for r, c in shapes:
            W = (0.02 * rng.standard_normal((r, c))).astype(np.float32)
            g = (grad_std * rng.standard_normal((r, c))).astype(np.float32)
            m = np.zeros((r, c), np.float32)
            t0 = time.perf_counter()
            OM.muon_step_tensor(W, g, m, LR, MU, NS_STEPS)
            total_ms += (time.perf_counter() - t0) * 1e3
        desc = f"oracle (fp64 NumPy) on every tensor of the shard ({len(shapes)} tensors), timed whole"
        return total_ms, desc, os.cpu_count() or 1
    classes = {}
    for r, c in shapes:
        key = (min(r, c), max(r, c))
        first, mult = classes.get(key, ((r, c), 0))
        classes[key] = (first, mult + 1)
    total_ms = 0.0
    parts = []
    for (mm, nn), ((r, c), mult) in classes.items():
        W = (0.02 * rng.standard_normal((r, c))).astype(np.float32)
        g = (grad_std * rng.standard_normal((r, c))).astype(np.float32)
        m = np.zeros((r, c), np.float32)
        t0 = time.perf_counter()
        OM.muon_step_tensor(W, g, m, LR, MU, 1)
        t_one = time.perf_counter() - t0
        X = rng.standard_normal((mm, nn)) / np.sqrt(mm * nn)
        t0 = time.perf_counter()
        OM.newton_schulz(X, 1)
        t_ns = time.perf_counter() - t0
        total_ms += mult * (t_one + (NS_STEPS - 1) * t_ns) * 1e3
        parts.append(f"{mm}x{nn} x{mult}")
    desc = (f"oracle (fp64 NumPy), extrapolated: per Newton-Schulz shape class ({', '.join(parts)}; "
            f"{len(shapes)} tensors) one tensor through muon_step_tensor with 1 Newton-Schulz step plus "
            f"{NS_STEPS - 1} x one timed newton_schulz step, times the class's multiplicity")
    return total_ms, desc, os.cpu_count() or 1


def step_config(w, my_shapes, extras, world):
    """The `config` object of the JSON line (the same for both arms)."""
    cfg = {"workload": w.name, "matrices": len(my_shapes), "elements": sum(r * c for r, c in my_shapes),
           "ns_steps": NS_STEPS, "R": extras.get("R", 1), "alpha": extras.get("alpha", 1.0),
           "l2": "flushed between timed steps: 256 MiB write, then 256 MiB read of another buffer",
           "grad": "bf16" if w.grad_bf16 else "fp32", "parallelism": f"dp{world}"}
    for k in ("cost", "plan_rank", "planned_from"):
        if k in extras:
            cfg[k] = extras[k]
    return cfg


def run_reference(args):
    """The reference arm: the oracle, as it stands, on this run's rank-0 shard, timed on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w, buckets, R, alpha, my_rank, extras = build_workload(args.workload, world, 0, planner="oracle")
    owner, _ = plan_owner_load(w.numels, buckets, R, alpha, planner="oracle")
    my_shapes = [s for s, o in zip(w.shapes, owner) if o == my_rank]
    for _ in range(args.warmup):
        time_oracle_sample(my_shapes, w.grad_std)
    vals = []
    desc, cores = "", 1
    for _ in range(args.steps):
        ms, desc, cores = time_oracle_sample(my_shapes, w.grad_std)
        vals.append(ms)
    v = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": v, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(w, my_shapes, extras, world),
            "cpu_baseline": {"value": v, "unit": "ms", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_cost_compare(args):
    """Both cost models of Algorithm 1 on the Qwen3-32B layout (R = 32, alpha = 1), measured on the GPU: every
    distinct shard (the multiset of its tensor shapes) of the numel plan and of the Newton-Schulz-flops plan is
    stepped `--steps` times after `--warmup` (L2 flushed before each step, CUDA events on the stream), and each
    plan's slowest rank is reported.  The step is communication-free, so that rank sets the distributed
    optimizer step time of the plan.  One GPU; prints one JSON line."""
    from collections import Counter

    import torch

    from zero_sharded_gb300 import build as zbuild
    from zero_sharded_gb300 import cz
    from zero_sharded_gb300 import workloads as wl

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if not os.path.exists(zbuild.LIB):
        zbuild.build()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    flush_rd = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        torch.sum(flush_rd)

    plans = {}
    for cost in ("numel", "flops"):
        full, own, load = qwen32_plan(cost)
        ranks = []
        for r in range(full.R):
            shapes = [s for s, o in zip(full.shapes, own) if o == r]
            ranks.append((r, tuple(sorted(Counter(shapes).items())), shapes))
        plans[cost] = (load, ranks)
    distinct = {}
    for cost in plans:
        for r, key, shapes in plans[cost][1]:
            distinct.setdefault(key, shapes)

    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    clocks.mark_begin()
    comp_ms = {}
    for key, shapes in distinct.items():
        if not shapes:
            comp_ms[key] = 0.0
            continue
        w = wl.Workload("shard", list(shapes), [f"t{i}" for i in range(len(shapes))], 0.02, 1e-3)
        plan = cz.cz_plan_partition(w.numels, [len(shapes)], 1, 1.0)
        P = wl.draw(w.shapes, w.param_std, 0, device=dev)
        G = wl.draw(w.shapes, w.grad_std, 1, device=dev)
        M = torch.zeros_like(P)
        PB = P.to(torch.bfloat16)
        ws_bytes = cz.cz_workspace_size(plan, 0, w.shapes)
        WS = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        sargs = cz.StepArgs(w.offsets, w.shapes)
        opts = cz.make_opts(param_bf16=PB, workspace=WS, workspace_bytes=ws_bytes)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush_l2()
                if i >= args.warmup:
                    ev[i - args.warmup][0].record(stream)
                cz.cz_muon_step_ex(plan, 0, P, G, M, sargs, LR, MU, NS_STEPS, stream, opts)
                if i >= args.warmup:
                    ev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        st = cz.cz_device_status(stream, WS)
        if st != cz.CZ_OK:
            raise SystemExit(f"device status: {cz.cz_status_string(st)}")
        comp_ms[key] = statistics.mean(a.elapsed_time(b) for a, b in ev)
        del P, G, M, PB, WS
        torch.cuda.empty_cache()
    clocks.mark_end()
    clk = clocks.stop()

    out = {}
    for cost, (load, ranks) in plans.items():
        ms = [comp_ms[key] for _, key, _ in ranks]
        tf = [ns_flops(shapes) / 1e12 for _, _, shapes in ranks]
        slow = max(range(len(ranks)), key=lambda r: (ms[r], -r))
        heavy = max(range(len(ranks)), key=lambda r: (load[r], -r))
        out[cost] = {"slowest_rank": slow, "slowest_ms": ms[slow], "slowest_ns_tflop": tf[slow],
                     "slowest_shard": {f"{a}x{b}": n for (a, b), n in ranks[slow][1]},
                     "heaviest_load_rank": heavy, "heaviest_load_ms": ms[heavy],
                     "max_rank_ns_tflop": max(tf), "mean_rank_ms": statistics.mean(ms),
                     "rank_ms": ms, "rank_ns_tflop": tf}
    line = {"mode": "plan-cost-compare", "metric": "Muon step ms of each plan's slowest shard", "unit": "ms",
            "higher_is_better": False, "layout": QWEN32_LAYOUT + "; Algorithm 1, R = 32, alpha = 1",
            "steps": args.steps, "warmup": args.warmup, "distinct_shards_timed": len(distinct),
            "numel": out["numel"], "flops": out["flops"],
            "slowest_ms_flops_over_numel": out["flops"]["slowest_ms"] / out["numel"]["slowest_ms"],
            "max_ns_tflop_flops_over_numel": out["flops"]["max_rank_ns_tflop"] / out["numel"]["max_rank_ns_tflop"],
            "clocks": clk, "data": "synthetic", "dtype": "bf16"}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["cz", "reference"], default="cz")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=WORKLOADS)
    ap.add_argument("--compare-cost", action="store_true",
                    help="time every distinct shard of the Qwen3-32B layout under the numel and the flops plans")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-torch-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.compare_cost:
        return run_cost_compare(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from zero_sharded_gb300 import build as zbuild
    from zero_sharded_gb300 import cz
    from zero_sharded_gb300 import workloads as wl

    if not os.path.exists(zbuild.LIB):
        zbuild.build()
    w, buckets, R, alpha, my_rank, extras = build_workload(args.workload, world, rank)
    plan = cz.cz_plan_partition(w.numels, buckets, R, alpha)
    owner = plan.owner()
    my_shapes = [s for s, o in zip(w.shapes, owner) if o == my_rank]
    stream = torch.cuda.Stream(device=dev)

    # synthetic inputs, generated on the device from fixed seeds
    gdt = torch.bfloat16 if w.grad_bf16 else torch.float32
    P = wl.draw(w.shapes, w.param_std, 0, device=dev)
    G = wl.draw(w.shapes, w.grad_std, 1, device=dev, dtype=gdt)
    M = torch.zeros_like(P)
    PB = P.to(torch.bfloat16)
    ws_bytes = cz.cz_workspace_size(plan, my_rank, w.shapes)
    WS = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)   # status word starts at zero
    # L2 flush between timed steps: write 256 MiB (> the 129 MB L2), then read another 256 MiB, so that no input
    # of the step stays in L2 and no dirty line of the flush is left for the step to write back
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    flush_rd = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        torch.sum(flush_rd)
    sargs = cz.StepArgs(w.offsets, w.shapes)
    opts = cz.make_opts(param_bf16=PB, workspace=WS, workspace_bytes=ws_bytes, grad_is_bf16=w.grad_bf16)

    def step():
        cz.cz_muon_step_ex(plan, my_rank, P, G, M, sargs, LR, MU, NS_STEPS, stream, opts)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step()
    st = cz.cz_device_status(stream, WS)
    if st != cz.CZ_OK:
        raise SystemExit(f"device status after warm-up: {cz.cz_status_string(st)}")

    # ---------------- timed region: K steps, L2 flushed between steps (outside the events)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    clocks.mark_begin()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    st = cz.cz_device_status(stream, WS)
    if st != cz.CZ_OK:
        raise SystemExit(f"device status after timed steps: {cz.cz_status_string(st)}")
    my_ms = statistics.mean(step_ms)
    t = torch.tensor([my_ms], device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    max_ms = float(t.item())

    # ---------------- per-kernel times (library event tracing), same steps again
    cz.cz_profile_enable(True)
    cz.cz_profile_read()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2()
            step()
    torch.cuda.synchronize()
    prof = cz.cz_profile_read()
    cz.cz_profile_enable(False)
    launches_per_step = sum(c for _, c in prof.values()) / args.steps
    ns_kinds = ("ns_gram", "ns_poly", "ns_update", "ns_update_apply", "ns_fused", "ns_small")
    ns_ms = sum(prof[k][0] for k in ns_kinds) / args.steps
    ns_launch = sum(prof[k][1] for k in ns_kinds) / args.steps
    mom_ms = prof["momentum"][0] / args.steps

    peaks, peak_src = load_peaks()
    F = ns_flops(my_shapes)
    F_exec = ns_flops_executed(my_shapes)
    ns_tflops = F / (ns_ms * 1e-3) / 1e12 if ns_ms > 0 else 0.0
    ns_exec_tflops = F_exec / (ns_ms * 1e-3) / 1e12 if ns_ms > 0 else 0.0
    el = sum(r * c for r, c in my_shapes)
    # algorithmic bytes of the momentum pass: read g and m, write m and one bf16 copy of u
    mom_bytes = el * (10 + (2 if w.grad_bf16 else 4))
    mom_moved = mom_bytes                                      # X is written once, in its m x n orientation
    mom_gbs = mom_bytes / (mom_ms * 1e-3) / 1e9 if mom_ms > 0 else 0.0
    hbm = float(peaks.get("hbm_gbs", 6800.0))

    # ---------------- end to end: host gradients in, bf16 parameters out, every step.
    # Every step copies its fp32 (or bf16) gradients from pinned host memory and reads its bf16 parameters
    # back; the copies run on two copy streams and overlap the neighbouring steps' compute (device gradient
    # and bf16-parameter buffers are double-buffered; momentum and the fp32 master are shared, so steps stay
    # ordered). Inputs (4.19 GB of gradients, 4.19 GB master, 4.19 GB momentum on the Qwen3-32B shard) exceed
    # the L2, so no flush is inserted. The warm-up steps are drained before the timed ones, so the window holds
    # exactly the K timed steps: value = (end of the last read-back - start of the first gradient copy) / K,
    # with the first copy and the last read-back exposed (nothing of the warm-up left to overlap them).
    e2e = None
    if not args.no_e2e:
        Gh = G.to("cpu").pin_memory()
        # the rank's own tensors only (after a reduce-scatter a ZeRO-1 rank holds just its shard's
        # gradients): contiguous owned element ranges, one copy each way per range
        own_rng = []
        for o_, (r_, c_), ow in sorted(zip(w.offsets, w.shapes, owner)):
            if ow != my_rank:
                continue
            if own_rng and own_rng[-1][1] == o_:
                own_rng[-1][1] = o_ + r_ * c_
            else:
                own_rng.append([o_, o_ + r_ * c_])
        PBh = [torch.empty(PB.shape, dtype=PB.dtype).pin_memory() for _ in range(2)]
        Gd = [G, torch.empty_like(G)]
        PBd = [PB, torch.empty_like(PB)]
        optsd = [cz.make_opts(param_bf16=PBd[i], workspace=WS, workspace_bytes=ws_bytes, grad_is_bf16=w.grad_bf16)
                 for i in range(2)]
        h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        n = args.warmup + args.steps
        ev_h2d = [torch.cuda.Event() for _ in range(n)]
        ev_step = [torch.cuda.Event() for _ in range(n)]
        ev_d2h = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # diagnostics: each timed step's compute and each timed gradient copy, on their own streams
        tse = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        tce = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(ev_step[i - 2])             # the device buffer's previous user is done
                if i == args.warmup:
                    # the warm-up steps are drained first (a copy that overlapped a warm-up step would put
                    # that step's compute inside the window); the region opens where the first timed step's
                    # gradient copy starts and closes when the last timed step's read-back ends
                    torch.cuda.synchronize()
                    t0.record(h2d)
                tce[i][0].record(h2d)
                for lo, hi in own_rng:
                    Gd[b][lo:hi].copy_(Gh[lo:hi], non_blocking=True)
                tce[i][1].record(h2d)
                ev_h2d[i].record(h2d)
            stream.wait_event(ev_h2d[i])
            if i >= 2:
                stream.wait_event(ev_d2h[i - 2])             # bf16 buffer read back before it is rewritten
            tse[i][0].record(stream)
            cz.cz_muon_step_ex(plan, my_rank, P, Gd[b], M, sargs, LR, MU, NS_STEPS, stream, optsd[b])
            tse[i][1].record(stream)
            ev_step[i].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_step[i])
                for lo, hi in own_rng:
                    PBh[b][lo:hi].copy_(PBd[b][lo:hi], non_blocking=True)
                ev_d2h[i].record(d2h)
        t1.record(d2h)
        torch.cuda.synchronize()
        e_ms = t0.elapsed_time(t1) / args.steps
        timed = range(args.warmup, n)
        e2e_step_ms = statistics.mean(tse[i][0].elapsed_time(tse[i][1]) for i in timed)
        e2e_h2d_ms = statistics.mean(tce[i][0].elapsed_time(tce[i][1]) for i in timed)
        te = torch.tensor([e_ms], device=dev)
        if world > 1:
            dist.all_reduce(te, op=dist.ReduceOp.MAX)
        e2e = {"value": float(te.item()), "unit": "ms",
               "h2d_bytes_per_step": int(sum(hi - lo for lo, hi in own_rng) * G.element_size()),
               "d2h_bytes_per_step": int(sum(hi - lo for lo, hi in own_rng) * PB.element_size()),
               "overlap": "two copy streams; step j+1's gradient copy and step j's read-back overlap compute",
               "step_ms_inside": e2e_step_ms, "h2d_ms_per_step": e2e_h2d_ms,
               "timing": "(end of the last timed read-back - start of the first timed gradient copy) / steps; "
                         "warm-up drained before the first timed copy, copies of later steps overlap compute"}

    # roofline of the dominant kernel (largest share of the step's device time).  The tensor cores execute the
    # symmetric products' upper-triangle tiles only (and K padded to 64), so the rate held against the peak is the
    # executed one; the dense count of the three products (K * sum(4m^2n + 2m^3)) is reported beside it.  The peak
    # is the measured cuBLAS bf16 rate for the clock state sampled in the timed region: the sustained rate when
    # the power cap was active, the burst rate otherwise.
    reasons = (clk or {}).get("reasons", [])
    capped = "sw_power_cap" in reasons
    peak_key = "bf16_tflops_sustained" if capped else "bf16_tflops"
    peak_t = float(peaks.get(peak_key, FALLBACK_PEAKS[peak_key]))
    peak_note = (f"{peak_key} of {peak_src} (" + ("sw_power_cap active in the timed region" if capped else
                 "no clock-event reason active in the timed region") + ")")
    dom = max(prof, key=lambda k: prof[k][0])
    dom_ms, dom_n = prof[dom][0], prof[dom][1]
    avg_ms = dom_ms / max(dom_n, 1)
    traffic = ncu_traffic(w.name, dom) if world == 1 else None
    if dom.startswith("ns_"):
        ex_per_launch = ns_flops_executed_by_kind(my_shapes)[dom] * args.steps / max(dom_n, 1)
        alg_per_launch = ns_flops_by_kind(my_shapes)[dom] * args.steps / max(dom_n, 1)
        ach = ex_per_launch / (avg_ms * 1e-3) / 1e12
        kname = ("ns_small_kernel, ns_small_pair_kernel" if dom == "ns_small" else "ns_gemm_kernel") + f" ({dom})"
        roof = {"bound": "tensor", "kernel": kname, "achieved": ach, "peak": peak_t,
                "unit": "TFLOP/s", "frac": ach / peak_t if peak_t else None, "traffic": traffic,
                "flops": "executed", "executed_per_launch": ex_per_launch, "launch_ms": avg_ms,
                "launches_per_step": dom_n / args.steps, "peak_source": peak_note,
                "algorithmic_per_launch": alg_per_launch,
                "algorithmic_achieved": alg_per_launch / (avg_ms * 1e-3) / 1e12}
    else:
        per_launch = mom_bytes
        ach = per_launch / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm if hbm else None, "traffic": traffic, "algorithmic_per_launch": per_launch,
                "launch_ms": avg_ms, "peak_source": f"hbm_gbs of {peak_src}"}

    # variable-size collective support: pack + unpack of the gradient buffer as one bucket whose shards are
    # whole tensors (cuts at tensor boundaries, as a partition map gives), blocks rounded to 16 bytes
    el_all = G.numel()
    cuts8 = list(w.offsets) + [el_all]
    nsh = len(cuts8) - 1
    blk = max(cuts8[i + 1] - cuts8[i] for i in range(nsh))
    blk = (blk + 7) // 8 * 8
    padded = torch.empty(nsh * blk, dtype=G.dtype, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with torch.cuda.stream(stream):
        cz.cz_bucket_pack(G, cuts8, blk, padded, stream)
        cz.cz_bucket_unpack(padded, cuts8, blk, G, stream)
        ev[0].record(stream)
        cz.cz_bucket_pack(G, cuts8, blk, padded, stream)
        ev[1].record(stream)
        cz.cz_bucket_unpack(padded, cuts8, blk, G, stream)
        ev[2].record(stream)
    torch.cuda.synchronize()
    esz = G.element_size()
    pack_ms, unpack_ms = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
    comm_pack = {"bucket_elements": el_all, "ranks": nsh, "block": blk,
                 "pack_gbs": (el_all + nsh * blk) * esz / (pack_ms * 1e-3) / 1e9,
                 "unpack_gbs": 2 * el_all * esz / (unpack_ms * 1e-3) / 1e9}
    del padded

    # standalone scale-and-apply (the apply the step fuses into its last Newton-Schulz epilogue) on the
    # shard's tensors: reads W and U (fp32), writes W and the bf16 copy; L2 flushed before each launch
    my_offs = [o for o, ow in zip(w.offsets, owner) if ow == my_rank]
    U = torch.empty_like(P).normal_(generator=torch.Generator(device=dev).manual_seed(7))
    n_ap = max(3, min(args.steps, 10))
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_ap)]
    with torch.cuda.stream(stream):
        cz.cz_apply_update(P, PB, U, my_offs, my_shapes, 1e-6, True, stream)
        for i in range(n_ap):
            flush_l2()
            ev_a[2 * i].record(stream)
            cz.cz_apply_update(P, PB, U, my_offs, my_shapes, 1e-6, True, stream)
            ev_a[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    ap_ms = statistics.mean(ev_a[2 * i].elapsed_time(ev_a[2 * i + 1]) for i in range(n_ap))
    ap_bytes = el * 14
    apply_standalone = {"bound": "hbm", "kernel": "apply_kernel", "achieved": ap_bytes / (ap_ms * 1e-3) / 1e9,
                        "peak": hbm, "unit": "GB/s", "frac": ap_bytes / (ap_ms * 1e-3) / 1e9 / hbm,
                        "bytes_per_element": 14, "launch_ms": ap_ms, "launches_timed": n_ap,
                        "traffic": ncu_traffic(w.name, "apply") if world == 1 else None,
                        "peak_source": f"hbm_gbs of {peak_src}"}
    del U

    # the same step through PyTorch library calls (cuBLAS bf16 matmuls per shape group), timed like the
    # step itself (L2 flushed before each step, CUDA events on the stream): context for what the kernels buy
    torch_base = None
    if not args.no_torch_baseline and world == 1:
        n_tb = max(3, min(args.steps, 5))
        ev_t = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_tb)]
        with torch.cuda.stream(stream):
            torch_library_step(P, G, M, my_shapes, my_offs)
            for i in range(n_tb):
                flush_l2()
                ev_t[2 * i].record(stream)
                torch_library_step(P, G, M, my_shapes, my_offs)
                ev_t[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        tb_ms = statistics.mean(ev_t[2 * i].elapsed_time(ev_t[2 * i + 1]) for i in range(n_tb))
        torch_base = {"ms_per_step": tb_ms, "steps_timed": n_tb, "speedup_of_this_path": tb_ms / max_ms,
                      "what": "PyTorch library calls: fp32 momentum elementwise, torch.linalg norm, bf16 batched "
                              "torch.matmul (cuBLAS) per shape group for Newton-Schulz, fp32 apply; no bf16 copy"}

    # planner timing on the 64-layer Qwen3-32B layout (host work, as the pages' "milliseconds" claim)
    full = wl.qwen3_32b_reverse()
    fb = cz.cz_make_buckets(full.numels, full.bucket_cap)
    t0 = time.perf_counter()
    p32 = cz.cz_plan_partition(full.numels, fb, full.R, full.alpha)
    plan_ms = (time.perf_counter() - t0) * 1e3
    planner = {"layout": "qwen3-32b 64 layers, 448 tensors, 320 buckets, R=32, alpha=1", "alg1_ms": plan_ms,
               "r_lb": p32.metrics()["r_lb"], "naive_r_lb": cz.cz_plan_naive(full.numels, fb, full.R).metrics()["r_lb"],
               "shard_plan": plan.metrics()}

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cms, desc, cores = time_oracle_sample(my_shapes, w.grad_std)
            cpu = {"value": cms, "unit": "ms", "cores": cores, "kind": "oracle", "sample": desc}
        line = {
            "metric": METRIC, "value": max_ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": step_config(w, my_shapes, extras, world),
            "value_definition": "the slowest rank's mean step time over the timed steps (each GPU steps one shard)",
            "ms_per_shard_job": max_ms / world,
            "roofline": roof,
            "ns_all_phases": {"executed_tflops": ns_exec_tflops, "unit": "TFLOP/s", "peak": peak_t,
                              "executed_frac": ns_exec_tflops / peak_t if peak_t else None,
                              "peak_source": peak_note, "executed_flops_per_step": F_exec,
                              "algorithmic_flops_per_step": F, "algorithmic_tflops": ns_tflops,
                              "launches_per_step": ns_launch, "ms_per_step": ns_ms},
            "momentum_pass": {"bound": "hbm", "achieved": mom_gbs, "peak": hbm, "unit": "GB/s",
                              "frac": mom_gbs / hbm if hbm else None, "bytes_per_element": mom_bytes / max(el, 1),
                              "moved_bytes_per_element": mom_moved / max(el, 1),
                              "traffic": ncu_traffic(w.name, "momentum") if world == 1 else None,
                              "ms_per_step": mom_ms, "peak_source": f"hbm_gbs of {peak_src}"},
            "step_ms_stats": {"median": statistics.median(step_ms),
                              "p90": sorted(step_ms)[min(len(step_ms) - 1, int(round(0.9 * (len(step_ms) - 1))))],
                              "min": min(step_ms), "max": max(step_ms), "rank": rank},
            "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clk, "wall_s_timed_region": wall,
            "planner": planner, "comm_pack": comm_pack, "apply_standalone": apply_standalone,
            "torch_library_baseline": torch_base,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
