"""bench.py's host-side measurement logic, on the CPU: the reference arm's JSON
line (the fp64 oracle timed on a bounded sample), the DRAM-traffic record that
is valid only for the source it was taken on, and the roofline arithmetic
(achieved = algorithmic bytes or FLOP / kernel time; frac = achieved / peak;
the dominant kernel class decides which roof)."""
from __future__ import annotations

import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mixed", "--steps", "2", "--warmup", "1",
                        "--ref-seconds", "1.5"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["higher_is_better"] is True
    # at least 3 warm-up steps whatever --warmup asks (the timing rules)
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["dtype"] == "f64" and d["config"]["workload"].startswith("tiny_mixed")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "units" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_traffic_record_needs_the_same_source(tmp_path, monkeypatch):
    src_dir = tmp_path / "paged_prefix_shared_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    kernel = src_dir / "k.cu"
    kernel.write_text("// kernel v1\n")
    sha = hashlib.sha256(kernel.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"k.cu:decode_heavy": {"source_sha256": sha, "dram_bytes_per_launch": 123.0}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k.cu", "decode_heavy") == 123.0
    assert bench.traffic_record("k.cu", "radix_sharing") is None       # no record
    kernel.write_text("// kernel v2\n")
    assert bench.traffic_record("k.cu", "decode_heavy") is None        # source changed


class _Pps:
    KERNEL_BANDWIDTH, KERNEL_TENSOR, KERNEL_MERGE = 0, 1, 2


def _info(kv_unique, kv_read, kv_bw, flops, tt=True):
    return {"kv_bytes_unique": kv_unique, "kv_bytes_read": kv_read, "kv_bytes_bw": kv_bw,
            "flops_mma": flops, "small_rows_on_tensor": 1 if tt else 0}


def test_roofline_bandwidth_class(monkeypatch):
    monkeypatch.setattr(bench, "load_peaks", lambda: ({"hbm_gbs": 6000.0, "bf16_tflops": 2000.0,
                                                      "bf16_tflops_sustained": 1500.0},
                                                     "measured"))
    monkeypatch.setattr(bench, "traffic_record", lambda f, w: None)
    # 2.4e9 B of K/V for the bandwidth tasks + 1e6 B of Q/O in 0.4 ms: 6002.5 GB/s
    roof = bench.roofline(_Pps, [0.4, 0.01, 0.01], [_info(2.4e9, 2.4e9, 2.4e9, 0.0)], 1e6,
                          "decode_heavy", sustained=False)
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx((2.4e9 + 1e6) / 0.4e-3 / 1e9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 6000.0)
    assert roof["kernel"].startswith("key-tile")
    roof = bench.roofline(_Pps, [0.4, 0.01, 0.01], [_info(2.4e9, 2.4e9, 2.4e9, 0.0, tt=False)],
                          1e6, "decode_heavy", sustained=False)
    assert roof["kernel"].startswith("split-KV bandwidth")


def test_roofline_tensor_class_picks_the_closer_roof(monkeypatch):
    monkeypatch.setattr(bench, "load_peaks", lambda: ({"hbm_gbs": 6000.0, "bf16_tflops": 2000.0,
                                                      "bf16_tflops_sustained": 1500.0},
                                                     "measured"))
    monkeypatch.setattr(bench, "traffic_record", lambda f, w: None)
    # compute-heavy: 3e13 FLOP in 30 ms = 1000 TFLOP/s (0.667 of sustained); bytes tiny
    roof = bench.roofline(_Pps, [0.0, 30.0, 0.0], [_info(1e9, 4e9, 0.0, 3e13)], 1e9,
                          "long_prefill", sustained=True)
    assert roof["bound"] == "tensor" and roof["peak"] == 1500.0
    assert roof["achieved"] == pytest.approx(1000.0)
    # the K/V the tensor tasks read counts each byte once: at most the unique bytes
    # 1e9 unique + 2e8 Q/O in 0.3 ms = 4000 GB/s (0.667) against 3e11 FLOP = 1000 TFLOP/s
    # of the 2000 burst (0.5): the HBM roof is the closer one
    roof = bench.roofline(_Pps, [0.0, 0.3, 0.0], [_info(1e9, 4e9, 0.0, 3e11)], 2e8,
                          "tree_verify", sustained=False)
    assert roof["bound"] == "hbm"
    assert roof["achieved"] == pytest.approx((1e9 + 2e8) / 0.3e-3 / 1e9)
