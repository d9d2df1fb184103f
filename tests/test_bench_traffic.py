"""bench.py's recorded DRAM traffic (roofline.traffic) belongs to the source it
was captured on: the figure is reported while kvq.cu and common.cuh hash to
the recorded value, scaled by tokens, and is null as soon as they differ.
No GPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_recorded_traffic_matches_committed_source():
    """A recorded figure carries the hash of the source it was captured on and
    must match the committed source; an entry without a hash (the kernel
    changed and was not recaptured yet) reports no traffic."""
    for name, ent in bench.TRAFFIC.items():
        if ent["sha256"] is None:
            for sh in ent["shapes"]:
                assert bench.kernel_traffic(name, 4096, sh) is None
            continue
        assert bench._source_hash(ent["sources"]) == ent["sha256"], f"{name} changed since its ncu capture: recapture"
        for sh in ent["shapes"]:
            assert bench.kernel_traffic(name, 4096, sh) == sh["bytes_per_token"] * 4096


def test_traffic_only_for_the_captured_shape(monkeypatch):
    """Another head count, index count, block size or mode has another
    per-token traffic: no figure is reported for it."""
    sh = dict(bench.TRAFFIC["kvq"]["shapes"][0])
    for k, v in (("N1", 64), ("K", 8192), ("bs", 64)):
        assert bench.kernel_traffic("kvq", 4096, dict(sh, **{k: v})) is None
    ent = dict(bench.TRAFFIC["kvq"], sha256="0" * 64)
    monkeypatch.setitem(bench.TRAFFIC, "kvq", ent)
    assert bench.kernel_traffic("kvq", 4096, sh) is None
    assert bench.kernel_traffic("sdp", 4096, sh) is None


def test_l2_red_microbenchmark_compiles(tmp_path):
    """bench.py --l2-red-ceiling builds bench_l2_red.cu for sm_103a; the
    source must compile (nvcc cross-compiles without a GPU)."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench_l2_red.cu")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", str(tmp_path / "b"), src],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_roofline_arithmetic():
    """The bench's roofline object: algorithmic flops (or bytes) per unit of
    the dominant kernel over its time, against the measured peak."""
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0}
    qhk, pairs, ms = 1 << 30, (1 << 30) // 128, 7.5
    r = bench.roofline("kvq", [], qhk, pairs, ms, peaks, False)
    assert r["bound"] == "tensor" and r["flops_per_query_head_key"] == 3328
    assert abs(r["achieved"] - qhk * 3328 / 7.5e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 2000.0) < 1e-12
    # the key-side scatter's rate against the reduction ceiling, atomic mode only
    assert abs(r["l2_red"]["achieved_gbs"] - pairs * 4352 / 7.5e-3 / 1e9) < 1e-6
    assert "l2_red" not in bench.roofline("kvq", [], qhk, pairs, ms, peaks, True)
    for name, per in (("sdp", 2176), ("sdpb", 2176), ("kvb", 2176), ("dqb", 1152)):
        assert bench.roofline(name, [], qhk, pairs, ms, peaks, False)["flops_per_query_head_key"] == per
    d = bench.roofline("det_reduce", [], qhk, pairs, ms, peaks, True)
    assert d["bound"] == "hbm" and d["bytes_per_pair"] == 2176
    assert abs(d["frac"] - pairs * 2176 / 7.5e-3 / 1e9 / 7000.0) < 1e-12
