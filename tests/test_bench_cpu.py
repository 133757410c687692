"""Host-side accounting of bench.py (CPU): algorithmic bytes, the
comment-insensitive source digest and the ncu traffic table lookup.

The expected byte counts below are worked out by hand from the layer's
definition: every touched expert's weights (codes + block scales) are read
once per launch; GEMM1 reads each routed row's activation in its quantised
format and writes the row's I activated features in GEMM2's input format;
GEMM2 reads those and writes H bf16 values per routed row.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_bf16_headline_bytes():
    # T=512, H=2048, I=1024, E=64, top-6: 3072 routed rows, all 64 experts
    s = workloads.spec("bf16")
    counts = np.full(64, 48)
    got, touched = bench.algorithmic_bytes(s, counts)
    assert touched == 64
    # GEMM1: 64 x (2048 x 2048 x 2 B) of W13 + 3072 x 4096 B in + 3072 x 2048 B out
    assert got["gemm1_swiglu"] == 64 * 8388608 + 3072 * 4096 + 3072 * 2048 == 555745280
    # GEMM2: 64 x (2048 x 1024 x 2 B) of W2 + 3072 x 2048 B in + 3072 x 4096 B out
    assert got["gemm2"] == 64 * 4194304 + 3072 * 2048 + 3072 * 4096 == 287309824


def test_nvfp4_single_token_bytes():
    # one token, top-8 of 384 experts, H=7168, I=2048: e2m1 codes are half a
    # byte per element, one e4m3 scale byte per 16 elements
    s = workloads.spec("nvfp4_decode", T=1)
    counts = np.zeros(384, np.int64)
    counts[[3, 50, 77, 100, 200, 256, 300, 383]] = 1
    got, touched = bench.algorithmic_bytes(s, counts)
    assert touched == 8
    w13 = 4096 * 7168 // 2 + 4096 * 7168 // 16     # 2I x H weight codes + scales
    w2 = 7168 * 2048 // 2 + 7168 * 2048 // 16
    assert got["gemm1_swiglu"] == 8 * w13 + 8 * (3584 + 448) + 8 * (1024 + 128)
    assert got["gemm2"] == 8 * w2 + 8 * (1024 + 128) + 8 * 2 * 7168


def test_relu2_w13_has_one_projection():
    s = workloads.spec("nvfp4_decode", T=1, act="relu2", clamp=0.0)
    counts = np.zeros(384, np.int64)
    counts[0] = 1
    got, _ = bench.algorithmic_bytes(s, counts)
    # W13 holds I rows (no gate half)
    assert got["gemm1_swiglu"] == 2048 * 7168 * 9 // 16 + (3584 + 448) + (1024 + 128)


def test_mxfp8_bytes_count_one_scale_per_32():
    s = workloads.spec("mxfp8_decode")
    counts = np.zeros(256, np.int64)
    counts[:2] = [3, 5]
    got, touched = bench.algorithmic_bytes(s, counts)
    assert touched == 2
    assert got["gemm2"] == 2 * (7168 * 2048 + 7168 * 64) + 8 * (2048 + 64) + 8 * 2 * 7168


def test_source_digest_ignores_comments_and_spacing(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one\n}\n")
    b.write_text("/* block\n comment */ int f(int x)\n{ return x + 1; }\n")
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_digest(str(a)) == bench.source_digest(str(b))
    assert bench.source_digest(str(a)) != bench.source_digest(str(c))


def _recorded_digests(monkeypatch):
    # the lookup as it behaves while the kernel sources hash as recorded
    import json
    tab = json.load(open(os.path.join(ROOT, "profiles", "gemm_traffic.json")))
    rec = {os.path.join(ROOT, k): v for k, v in tab["sources_sha1"].items()}
    monkeypatch.setattr(bench, "source_digest", lambda path: rec[path])
    return tab


def test_traffic_scaled_by_touched_experts(monkeypatch):
    tab = _recorded_digests(monkeypatch)
    per = tab["per_touched_expert_bytes"]["bf16"]["gemm1_swiglu"]
    v, src = bench.ncu_traffic(workloads.spec("bf16"), 64, "gemm1_swiglu", 1)
    assert v == int(per * 64) and "touched experts" in src
    assert 500e6 < v < 700e6          # close to the 556 MB the kernel must move
    v, src = bench.ncu_traffic(workloads.spec("tiny_bf16"), 8, "gemm1_swiglu", 1)
    assert v is None and "no ncu capture" in src


def test_traffic_scaled_by_algorithmic_bytes(monkeypatch, tmp_path):
    # a reduced-E prefill capture: DRAM bytes per algorithmic byte of the
    # captured case times the run's algorithmic bytes
    import json
    tab = _recorded_digests(monkeypatch)
    tab = dict(tab, traffic_per_algorithmic_byte={"nvfp4_prefill": {"gemm1_swiglu": 1.05}},
               captures=dict(tab["captures"], nvfp4_prefill="T=4096, E=48"))
    root = tmp_path / "r"
    (root / "profiles").mkdir(parents=True)
    (root / "profiles" / "gemm_traffic.json").write_text(json.dumps(tab))
    monkeypatch.setattr(bench, "ROOT", str(root))
    rec = {str(root / k): v for k, v in tab["sources_sha1"].items()}
    monkeypatch.setattr(bench, "source_digest", lambda path: rec[path])
    v, src = bench.ncu_traffic(workloads.spec("nvfp4_prefill"), 192, "gemm1_swiglu", 3.5e9)
    assert v == int(1.05 * 3.5e9) and "algorithmic" in src


def test_traffic_is_dropped_once_a_source_changes(monkeypatch):
    monkeypatch.setattr(bench, "source_digest", lambda path: "0" * 40)
    v, src = bench.ncu_traffic(workloads.spec("bf16"), 64, "gemm1_swiglu", 1)
    assert v is None and "changed" in src


@pytest.mark.parametrize("units,world,secs,rate", [(5120, 1, 2.0, 2560.0),
                                                   (5120, 2, 4.0, 2560.0)])
def test_whole_job_rate(units, world, secs, rate):
    assert bench.whole_job_rate(units, world, secs) == pytest.approx(rate)
