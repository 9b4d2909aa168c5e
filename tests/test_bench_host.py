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
    import hashlib
    import json
    # a repository copy with two kernel sources and one traffic entry
    srcs = []
    for i, rel in enumerate(bench.KERNEL_SOURCES):
        f = tmp_path / rel
        f.parent.mkdir(parents=True, exist_ok=True)
        f.write_text(f"// kernel source {i}\n")
        srcs.append(f)
    h = hashlib.sha256()
    for f in srcs:
        h.update(f.read_bytes())
    side = tmp_path / "profiles" / "traffic.json"
    side.parent.mkdir(parents=True, exist_ok=True)
    side.write_text(json.dumps({"entries": [
        {"workload": "mixtral", "T": 4096, "kernel": "gate_up_gemm", "summary": "x.md",
         "traffic_bytes_per_launch": 123456, "kernel_source_sha256": h.hexdigest()}]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(side))
    assert bench.profiled_traffic("mixtral", 4096, 8, "gate_up_gemm") == 123456
    # no entry for this workload / size / expert count
    assert bench.profiled_traffic("deepseek", 8192, 256, "gate_up_gemm") is None
    assert bench.profiled_traffic("mixtral", 512, 8, "gate_up_gemm") is None
    assert bench.profiled_traffic("mixtral", 4096, 4, "gate_up_gemm") is None
    assert bench.profiled_traffic("mixtral", 4096, 8, "down_gemm") is None
    # a changed kernel source invalidates the stored counters
    srcs[0].write_text("// changed\n")
    assert bench.profiled_traffic("mixtral", 4096, 8, "gate_up_gemm") is None


@pytest.mark.parametrize("name", ["qwen", "deepseek", "qwen_nvfp4"])
def test_weight_bytes_follow_the_bundle_size(bench, name):
    """The bytes per weight that the roofline counts match the packed bundle size of the
    workload's storage format (within the 256-byte section padding and the 12 bytes of NVFP4
    matrix scales)."""
    import expert_dispatch_streaming_gb300 as moe
    cfg = bench.WORKLOADS[name]
    nb = moe.moe_bundle_bytes(cfg.H, cfg.I, cfg.wdtype)
    w = bench.layer_work(cfg, 1, 1)
    w0 = bench.layer_work(cfg, 1, 0)
    per_expert = w["bytes"] - w0["bytes"]                 # one more unique routed expert
    assert abs(per_expert - nb) <= 3 * 256 + 12


def test_committed_traffic_entries_are_readable(bench):
    """Every entry of the traffic sidecar names a committed summary and carries its figures."""
    import json
    entries = json.load(open(bench.TRAFFIC_FILE))["entries"]
    assert entries
    for e in entries:
        assert os.path.exists(os.path.join(ROOT, "profiles", e["summary"])), e["summary"]
        assert int(e["traffic_bytes_per_launch"]) > 0
        assert len(e["kernel_source_sha256"]) == 64


def test_tier_bound_is_the_slower_tier(bench):
    # 5.09 GB of misses per step over a 205.5 GB/s link: 24.77 ms, above 2.7 ms of compute
    assert bench.tier_bound_ms(2.7, 5.09e9, 205.5) == pytest.approx(24.769, rel=1e-4)
    # few misses: the resident compute bounds the step
    assert bench.tier_bound_ms(1.6, 91e6, 205.5) == 1.6
    assert bench.tier_bound_ms(1.6, 0.0, 205.5) == 1.6
