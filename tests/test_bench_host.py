"""Host-side pieces of bench.py: algorithmic work accounting and the profiled-traffic lookup."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def bench():
    saved = sys.argv
    sys.argv = ["bench.py"]
    try:
        import bench as b
    finally:
        sys.argv = saved
    return b


def test_layer_work_counts_the_shared_expert_only_when_merged(bench):
    import workloads as wl
    cfg = wl.QWEN
    T = 64
    a = bench.layer_work(cfg, T, 30, shared_merged=False)
    b = bench.layer_work(cfg, T, 30, shared_merged=True)
    assert b["gu"][0] - a["gu"][0] == pytest.approx(4.0 * T * cfg.H * cfg.Is)
    assert b["dn"][0] - a["dn"][0] == pytest.approx(2.0 * T * cfg.Is * cfg.H)
    # the layer totals do not depend on how the launches are grouped
    assert a["flops"] == b["flops"] and a["bytes"] == b["bytes"]
    # Mixtral-shaped (no shared expert): unchanged either way
    m0, m1 = bench.layer_work(wl.MIXTRAL, T, 8, False), bench.layer_work(wl.MIXTRAL, T, 8, True)
    assert m0 == m1


def test_profiled_traffic_follows_the_kernel_sources(bench, tmp_path, monkeypatch):
    # the committed summary matches the committed sources
    assert isinstance(bench.profiled_traffic("mixtral", 4096, 8, "gate_up_gemm"), int)
    # no summary for this workload / size / expert count
    assert bench.profiled_traffic("deepseek", 8192, 256, "gate_up_gemm") is None
    assert bench.profiled_traffic("mixtral", 512, 8, "gate_up_gemm") is None
    assert bench.profiled_traffic("mixtral", 4096, 4, "gate_up_gemm") is None
    # a changed kernel source invalidates the stored counters
    changed = tmp_path / "tc_gemm.cu"
    changed.write_text("// changed\n")
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(changed)] + bench.KERNEL_SOURCES[1:])
    assert bench.profiled_traffic("mixtral", 4096, 8, "gate_up_gemm") is None
