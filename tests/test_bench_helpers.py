"""Host logic of bench.py that its JSON line rests on: the roofline object, the
source hash that keys recorded DRAM traffic, and the traffic lookup."""
import json
import os

import pytest


def test_roofline_picks_the_larger_floor_and_scales_the_peak():
    import bench
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    # 2 TFLOP, 1 GB: tensor floor 1 ms, HBM floor 0.17 ms -> tensor
    r = bench.roofline(2e12, 1e9, 2e-3, peaks)
    assert r["bound"] == "tensor" and r["achieved"] == 1000.0 and r["frac"] == 0.5 and r["unit"] == "TFLOP/s"
    # 1 GFLOP, 6 GB: HBM floor 1 ms -> hbm
    r = bench.roofline(1e9, 6e9, 2e-3, peaks)
    assert r["bound"] == "hbm" and r["achieved"] == 3000.0 and r["frac"] == 0.5 and r["unit"] == "GB/s"
    # an fp8 peak is the bf16 figure times the stated ratio
    r = bench.roofline(2e12, 1e9, 1e-3, peaks, peak_scale=bench.FP8_OVER_BF16)
    assert r["peak"] == 2000.0 * bench.FP8_OVER_BF16 and r["frac"] == pytest.approx(2000.0 / r["peak"], abs=1e-4)


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    import bench
    a = 'int f(int x) {\n  // a comment\n  return x + 1; /* block\n comment */\n}\nconst char* s = "//not a comment";\n'
    b = 'int f(int x) {\n\n  return x + 1;\n}\n// appended\nconst char* s = "//not a comment";\n'
    c = a.replace("x + 1", "x + 2")
    d = a.replace('"//not a comment"', '"//not a Comment"')
    for name, text in (("a.cu", a), ("b.cu", b), ("c.cu", c), ("d.cu", d)):
        (tmp_path / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.source_sha("a.cu") == bench.source_sha("b.cu")
    assert bench.source_sha("a.cu") != bench.source_sha("c.cu")
    assert bench.source_sha("a.cu") != bench.source_sha("d.cu")   # text inside a string literal is code


def test_recorded_traffic_matches_the_current_sources():
    """Every figure in profiles/traffic.json names a profile that exists and was
    taken on the kernel's current code, so bench.py reports it."""
    import bench
    path = os.path.join(bench.ROOT, "profiles", "traffic.json")
    with open(path) as f:
        d = json.load(f)
    for key, e in d.items():
        kernel, workload = key.split("|")
        assert kernel in bench.KERNEL_SOURCES
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", e["profile"])), e["profile"]
        assert bench.measured_traffic(kernel, workload) == e["bytes_per_launch"], key
