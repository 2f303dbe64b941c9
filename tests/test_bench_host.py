"""Host logic of the benchmark that needs no GPU: the DRAM-traffic figures a
bench line reports come from the committed ncu summaries only while the
kernel's source is the one they were taken on, and the per-kernel
algorithmic work follows the layer's definition."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from nvfp4_mixture_experts_router_gb300 import synth  # noqa: E402


def test_traffic_entries_name_existing_sources():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    csrc = os.path.join(ROOT, "nvfp4_mixture_experts_router_gb300", "csrc")
    entries = {k: v for k, v in d.items() if not k.startswith("_")}
    assert entries
    for key, e in entries.items():
        workload, kernel = key.rsplit(":", 1)
        assert kernel in ("fc1", "fc2"), key
        assert os.path.exists(os.path.join(csrc, e["source"])), key
        assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0, key
        assert len(e["source_sha"]) == 16 and e["command"].startswith("ncu "), key
        assert "--clock-control none" in e["command"], key


def test_traffic_is_null_once_the_source_changes(tmp_path, monkeypatch):
    """traffic_for reports an entry while its source hash matches, else None."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.source_sha("gemm_swap.cu")
    (prof / "traffic.json").write_text(json.dumps({
        "w:fc1": {"source": "gemm_swap.cu", "source_sha": sha, "dram_bytes_per_launch": 123},
        "w:fc2": {"source": "gemm_swap.cu", "source_sha": "0" * 16, "dram_bytes_per_launch": 456},
    }))
    real_join = os.path.join

    def join(*parts):
        if len(parts) >= 2 and parts[0] == bench.ROOT and parts[1] == "profiles":
            return real_join(str(tmp_path), *parts[1:])
        return real_join(*parts)

    monkeypatch.setattr(bench.os.path, "join", join)
    assert bench.traffic_for("fc1", "w") == 123
    assert bench.traffic_for("fc2", "w") is None
    assert bench.traffic_for("fc1", "other") is None


def test_source_hash_follows_included_headers():
    """A translation unit's hash covers the headers it includes (the swapped
    GEMM includes common.cuh and kernels.h), so it differs from a hash of
    the unit's own text alone, and it is deterministic."""
    import hashlib
    csrc = os.path.join(ROOT, "nvfp4_mixture_experts_router_gb300", "csrc")
    own = hashlib.sha256(open(os.path.join(csrc, "gemm_swap.cu"), "rb").read()).hexdigest()[:16]
    assert bench.source_sha("gemm_swap.cu") != own
    assert bench.source_sha("gemm_swap.cu") == bench.source_sha("gemm_swap.cu")


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_flops_follow_the_layer_definition(idx):
    """2 R (N1 H + I H): N1 = 2I with SwiGLU, I with ReLU2."""
    c = synth.config(idx)
    n1 = 2 * c.I if c.act == 0 else c.I
    assert bench.flops_per_step(c) == pytest.approx(2.0 * c.T * c.K * (n1 * c.H + c.I * c.H))


def test_forward_times_quantiles():
    """The per-forward summary takes the median, p10 and p90 of the sorted
    times (checked with a stand-in for the CUDA events)."""
    import types

    class Ev:
        t = 0.0

        def __init__(self, enable_timing=True):
            self.at = None

        def record(self):
            self.at = Ev.t

        def elapsed_time(self, other):
            return other.at - self.at

    durations = iter([5.0, 1.0, 3.0, 2.0, 4.0, 9.0, 7.0, 6.0, 8.0, 10.0, 0.5])

    def call():
        Ev.t += next(durations)

    fake = types.SimpleNamespace(cuda=types.SimpleNamespace(Event=Ev, synchronize=lambda: None))
    saved = sys.modules.get("torch")
    sys.modules["torch"] = fake
    try:
        r = bench.forward_times(call, 11)
    finally:
        sys.modules["torch"] = saved
    s = sorted([5.0, 1.0, 3.0, 2.0, 4.0, 9.0, 7.0, 6.0, 8.0, 10.0, 0.5])
    assert r["median_ms"] == s[5] and r["p10_ms"] == s[1] and r["p90_ms"] == s[9] and r["n"] == 11
