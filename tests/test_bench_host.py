"""bench.py's host-side bookkeeping on the CPU: algorithmic bytes, launch
counts and the committed profile of every benchmarked workload."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_algorithmic_bytes_of_the_worked_configs():
    """The per-call byte counts of the decode configs (planes + x + signs + fp32 y)."""
    w = synth.WORKLOADS
    assert bench.algorithmic_bytes(w["gateup"], 1)["total"] == 23_764_992
    assert bench.algorithmic_bytes(w["down"], 1)["total"] == 19_587_072
    assert bench.algorithmic_bytes(w["down_m8"], 8)["total"] == 19_974_144
    assert bench.algorithmic_bytes(w["head"], 1)["total"] == 338_728_960
    assert bench.algorithmic_bytes(w["tiny"], 1)["total"] == 76_800
    assert bench.algorithmic_bytes(w["embed"], 1)["total"] == 87_040 + 256 + 10_240 + 1_310_720
    assert bench.algorithmic_bytes(w["ffn_gate_up"], 1)["weights"] == 2 * 23_674_880


def test_every_benchmarked_workload_has_a_profile():
    """Each workload bench.py can time (the tiny parity case aside) has an ncu
    summary under profiles/ naming its kernel, the source hash and the commands."""
    for name, w in synth.WORKLOADS.items():
        if name == "tiny":
            continue
        tag, files = bench.dominant_kernel(w)
        path = os.path.join(ROOT, "profiles", f"{tag}_{name}.md")
        assert os.path.exists(path), path
        text = open(path, encoding="utf-8").read()
        assert re.search(r"^source_sha256: [0-9a-f]{64}$", text, re.M), path
        assert "ncu --metrics gpu__time_duration.sum --clock-control none" in text, path
        assert f"python bench.py --workload {name}" in text, path
        assert all(os.path.exists(os.path.join(ROOT, f)) for f in files)
        assert bench.kernels_per_step(w) >= 1


def test_launch_counts():
    import dataclasses

    w = synth.WORKLOADS
    assert bench.kernels_per_step(w["gateup"]) == 1
    assert bench.kernels_per_step(w["ffn_gate_up"]) == 1
    assert bench.kernels_per_step(w["down"]) == 1           # rotation fused into the decode kernel
    assert bench.kernels_per_step(w["prefill"]) == 2
    assert bench.kernels_per_step(w["prefill_down"]) == 3
    # the general gate/up path: two projections and the SwiGLU kernel
    assert bench.kernels_per_step(dataclasses.replace(w["down"], mats=2)) == 3
    assert bench.kernels_per_step(dataclasses.replace(w["gateup"], mats=2, M=4)) == 5
