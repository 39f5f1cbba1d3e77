"""Host logic of bench.py, on the CPU: which measured peak a roofline fraction
uses, which resource binds the dominant GEMM, how the fused permute changes
the kernel table and GEMM1's algorithmic bytes, and how a traffic record is
found (by kernel and workload, and only while its kernel's sources are
unchanged)."""
import hashlib
import json
import os

import pytest
import torch

import bench
from workloads import shape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _kmean(g1_ms, g2_ms):
    return {"router_logits": 0.05, "route": 0.02, "permute": 0.03, "grouped_gemm1_swiglu": g1_ms,
            "grouped_gemm2": g2_ms, "unpermute": 0.03}


def _peaks(monkeypatch, burst=2000.0, sustained=1600.0, hbm=7000.0):
    monkeypatch.setattr(bench, "_peaks", lambda: ({"bf16_tflops": burst, "bf16_tflops_sustained": sustained,
                                                    "hbm_gbs": hbm}, "measured"))


def test_short_region_takes_the_burst_peak_long_region_the_sustained(monkeypatch):
    _peaks(monkeypatch)
    s = shape("mixtral")
    counts = torch.full((s.E,), s.T * s.K // s.E)
    flop = 4.0 * s.T * s.K * s.d * s.f
    r = bench._dominant_roofline(s, "mixtral", _kmean(2.0, 1.0), counts, False, region_s=0.07)
    assert r["bound"] == "tensor" and r["kernel"] == "grouped_gemm1_swiglu"
    assert r["achieved"] == pytest.approx(flop / 2.0e-3 / 1e12)
    assert r["peak"] == 2000.0 and "burst" in r["peak_source"]
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["frac_of_bf16_sustained"] == pytest.approx(r["achieved"] / 1600.0)
    r = bench._dominant_roofline(s, "mixtral", _kmean(2.0, 1.0), counts, False, region_s=3.0)
    assert r["peak"] == 1600.0 and "sustained" in r["peak_source"]
    # MXFP8: twice the bf16 figure (the nominal fp8 / bf16 dense ratio)
    r = bench._dominant_roofline(s, "mixtral", _kmean(2.0, 1.0), counts, True, region_s=0.07)
    assert r["peak"] == 4000.0


def test_weight_streaming_shape_is_bound_by_hbm(monkeypatch):
    _peaks(monkeypatch)
    s = shape("dsv3")
    counts = torch.zeros(s.E, dtype=torch.int64)
    counts[:163] = 1          # 163 live experts
    r = bench._dominant_roofline(s, "dsv3", _kmean(2.0, 1.0), counts, False, region_s=0.07)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    w = 163 * 2.0 * s.f * s.d * 2
    assert r["algorithmic"]["bytes"] == pytest.approx(w + 2.0 * s.T * s.K * s.d + 2.0 * s.T * s.K * s.f)
    assert r["frac"] == pytest.approx(r["algorithmic"]["bytes"] / 2.0e-3 / 1e9 / 7000.0)
    # with the permute fused, GEMM1 reads each token row once (T rows, not T*K)
    f = bench._dominant_roofline(s, "dsv3", _kmean(2.0, 1.0), counts, False, region_s=0.07, fused_permute=True)
    assert r["algorithmic"]["bytes"] - f["algorithmic"]["bytes"] == pytest.approx(2.0 * (s.T * s.K - s.T) * s.d)


def test_kernel_table_marks_a_fused_permute(monkeypatch):
    _peaks(monkeypatch)
    s = shape("skew")
    k = bench._kernel_table(s, _kmean(2.9, 1.4), False, fused_permute=True)
    assert k["permute"]["fused_into"] == "grouped_gemm1_swiglu" and "GB/s" not in k["permute"]
    assert abs(sum(v["share"] for v in k.values()) - 1.0) < 1e-9
    k = bench._kernel_table(s, _kmean(2.9, 1.4), False)
    b = 2.0 * s.T * s.d + 2.0 * s.T * s.K * s.d + 4.0 * s.T * s.K
    assert k["permute"]["GB/s"] == pytest.approx(b / 0.03e-3 / 1e9)


def test_traffic_records_are_keyed_by_kernel_and_workload_and_follow_the_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        recs = json.load(fh)
    assert recs, "no traffic records"
    for key, rec in recs.items():
        kernel, workload = key.split("@")
        assert rec["workload"] == workload
        digest = hashlib.sha256()
        for src in rec["source"]:
            with open(os.path.join(ROOT, src), "rb") as fh:
                digest.update(fh.read())
        current = digest.hexdigest()[:16] == rec["source_sha256_16"]
        got = bench._traffic_record(kernel, workload)
        # a record is used only while its kernel's sources are the ones it was taken on
        assert (got is not None) == current
        if got is not None:
            assert abs(got["dram_bytes_per_launch"] - rec["dram_read"] - rec["dram_write"]) <= 1
        assert bench._traffic_record(kernel, workload + "_other") is None
