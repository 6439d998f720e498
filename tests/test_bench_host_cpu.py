"""bench.py's host-side helpers on the CPU: the clock record parsed from nvidia-smi samples
(a stand-in process returns canned lines), the measured-peaks fallback, and the traffic record
lookup keyed by the kernel sources' hash."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _FakeProc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_record_median_max_and_reasons(monkeypatch):
    lines = "\n".join([
        "2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1200.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1210.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ])
    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: _FakeProc(lines))
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    c = bench.Clocks("GPU-0")
    r = c.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_record_flags_thermal_slowdown(monkeypatch):
    lines = "1500, 2070, 1300, 0x20, Not Active, Active, Not Active, Not Active"
    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: _FakeProc(lines))
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    r = bench.Clocks(None).stop()
    assert r["reasons"] == ["hw_thermal_slowdown"] and r["sm_mhz"] == 1500.0


def test_peaks_fallback_and_measured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, 1900.0, 1700.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6787.2, "bf16_tflops": 1919.3, "bf16_tflops_sustained": 1700.0}))
    assert bench.peaks() == (6787.2, 1919.3, 1700.0, "measured")


def test_recorded_traffic_needs_the_current_sources(tmp_path, monkeypatch):
    import rpa_inputs as ri

    src = bench.kernel_sources(ri.workload("tiny"), "decode_attention")
    sha = bench.sources_sha(src)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "kernel_traffic.txt").write_text(
        "# comment\n"
        f"decode_attention decode {sha} 123456\n"
        "decode_attention mixed 0000000000000000 999\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # sources_sha reads the kernel files relative to ROOT: keep them readable from the repo
    monkeypatch.setattr(bench, "sources_sha", lambda names: sha)
    assert bench.recorded_traffic("decode_attention", "decode", src) == 123456.0
    assert bench.recorded_traffic("decode_attention", "fp8_window", src) is None
    assert bench.recorded_traffic("combine", "decode", src) is None


def test_kernel_sources_follow_the_routing():
    """Each workload's dominant kernel is charged to its own source file."""
    import rpa_inputs as ri

    want = {("decode", "decode_attention"): "rpa_decode.cu", ("long_prefill", "prefill_attention"): "rpa_prefill_tc.cu",
            ("fp8_window", "prefill_attention"): "rpa_prefill_tc8.cu",
            ("long_prefill_d256", "prefill_attention"): "rpa_prefill_tc8.cu",
            ("mla_decode", "prefill_attention"): "rpa_mla.cu"}
    for (w, k), f in want.items():
        src = bench.kernel_sources(_shape_only(w), k)
        assert src[0].endswith(f) and src[1].endswith("rpa_internal.cuh"), (w, src)
    # every 8-bit cache takes the 64-key-tile kernel, D 64 included; 2-byte K/V at D 64 / 128 the
    # 128-key-tile kernel; every named file exists
    import os
    import types

    for kv, d, f in (("fp8_e4m3", 64, "rpa_prefill_tc8.cu"), ("int8", 128, "rpa_prefill_tc8.cu"),
                     ("fp8_e5m2", 256, "rpa_prefill_tc8.cu"), ("f16", 64, "rpa_prefill_tc.cu"),
                     ("bf16", 128, "rpa_prefill_tc.cu"), ("f16", 256, "rpa_prefill_tc8.cu")):
        src = bench.kernel_sources(types.SimpleNamespace(kv_dtype=kv, head_dim=d, kv_layout="split"),
                                   "prefill_attention")
        assert src[0].endswith(f), (kv, d, src)
        assert all(os.path.isfile(os.path.join(bench.ROOT, x)) for x in src), src


def _shape_only(name):
    """The configuration fields of a named workload without drawing its tensors."""
    import types

    import rpa_inputs as ri

    shapes = {"decode": ("bf16", 128, "split"), "long_prefill": ("bf16", 128, "split"),
              "fp8_window": ("fp8_e4m3", 256, "split"), "long_prefill_d256": ("bf16", 256, "split"),
              "mla_decode": ("bf16", 576, "latent")}
    kv, d, layout = shapes[name]
    assert name in ri.WORKLOADS
    return types.SimpleNamespace(kv_dtype=kv, head_dim=d, kv_layout=layout)


def test_output_shape_follows_the_value_width():
    """The bench allocates o with the value width: head_dim, or 512 for the latent workload."""
    import torch

    import bench
    import rpa_inputs as ri

    for name, width in (("tiny", 64), ("mla_decode", 512)):
        p = ri.workload(name)
        q = torch.zeros(p.q.shape, dtype=torch.bfloat16)
        o = bench.out_for(p, q)
        assert tuple(o.shape) == (p.num_q_tokens, p.num_q_heads, width) and o.dtype == torch.bfloat16
