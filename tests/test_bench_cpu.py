"""bench.py without a GPU: the workload tables are consistent, and the reference arm (the oracle on
the host cores) prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from int4_routed_expert_05_b300 import moe, synth  # noqa: E402
from int4_routed_expert_05_b300.resident import moe_shape  # noqa: E402


def test_workload_tables():
    assert "stack80" in bench.CONFIGS
    from int4_routed_expert_05_b300 import synth_hybrid
    for name, (shape, layers, bits, desc) in bench.CONFIGS.items():
        if name in bench.HYBRID:
            kind, L, ctx = bench.HYBRID[name]
            assert hasattr(synth_hybrid, shape) and L == layers and desc
            continue
        assert hasattr(synth, shape) and bits in (4, 8) and layers >= 1 and desc
    # the hybrid workloads' layer counts are the pages' 36 + 12 = 48
    assert bench.HYBRID["gdn80"][1] + bench.HYBRID["gqa80_8k"][1] == 48
    for name, t in bench.BATCHED.items():
        assert name in bench.CONFIGS and bench.CONFIGS[name][1] == 1 and t in (8, 64, 512, 4096)
    stride = moe.expert_stride(moe_shape(synth.S80))
    for name, slots in bench.POOL_SLOTS.items():
        assert slots == (2 << 30) // stride == 1213


def _reference_line(config):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", config,
                          "--steps", "1", "--warmup", "0", "--ref-budget", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _reference_line("prefill80_t8")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "prefill80_t8"
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == ncores
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_hybrid_lines():
    for cfg in ("gdn80", "gqa80_8k"):
        d = _reference_line(cfg)
        assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == cfg
        assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
