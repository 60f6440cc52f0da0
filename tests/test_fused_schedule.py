"""The fused launch's dependency-aware schedule, checked on the CPU.

tests/cpp/fused_schedule_check.cpp includes the library's scheduler
(zero_sharded_gb300/csrc/fused_schedule.h, host code with no CUDA types), builds the
seven tile lists of a shard, and checks that every (step, product, matrix) gets
exactly its tiles from the right list, and that replaying the units' sequences with
random tile durations and hand-offs never blocks for good (the launch's waits cannot
form a cycle).
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("no g++")
    out = str(tmp_path_factory.mktemp("sched") / "fused_schedule_check")
    src = os.path.join(ROOT, "tests", "cpp", "fused_schedule_check.cpp")
    inc = os.path.join(ROOT, "zero_sharded_gb300", "csrc")
    r = subprocess.run(["g++", "-O2", "-std=c++17", "-Wall", "-I", inc, src, "-o", out], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
    return out


SHARDS = {
    # the Qwen3-1.7B layer's shape groups (m = min, n = max)
    "layer": "2048x2048,2048x2048,1024x2048,1024x2048,2048x6144,2048x6144,2048x6144",
    # one tile per product: a chain of stages
    "single": "256x256",
    # ragged sizes
    "ragged": "384x1024,384x1024,256x256,128x640,640x640,300x520",
}


@pytest.mark.parametrize("shard", sorted(SHARDS))
@pytest.mark.parametrize("steps", [1, 2, 5, 6, 16])
def test_schedule_covers_every_tile_and_cannot_deadlock(checker, shard, steps):
    units = 1 if shard == "single" else 76
    r = subprocess.run([checker, str(units), str(steps), SHARDS[shard]], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok:")


def test_schedule_with_more_units_than_tiles(checker):
    r = subprocess.run([checker, "76", "5", SHARDS["single"]], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
