"""Host-side pieces of bench.py that need no GPU: the roofline arithmetic, the
peak figures it divides by, and the CPU baseline's bounded sample (the oracle
timed on the host cores)."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0,
         "source": "measured"}


def test_hbm_roofline_is_algorithmic_bytes_over_kernel_time():
    r = bench.hbm_roofline("k", kbytes=3.0e9, kernel_ms=1.0, call_bytes=3.3e9, call_ms=1.1,
                           peaks=PEAKS, traffic=3_100_000_000)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(3000.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["call_achieved"] == pytest.approx(3000.0)
    assert r["call_frac"] == pytest.approx(0.5)
    assert r["traffic"] == 3_100_000_000 and r["peak"] == 6000.0
    assert r["frac_of_8tbs"] == pytest.approx(3000.0 / bench.NOMINAL_HBM_GBS, abs=1e-4)


def test_tensor_roofline_is_flops_over_kernel_time():
    r = bench.tensor_roofline("k", flops=1.0e12, kernel_ms=1.0, call_ms=2.0, peaks=PEAKS,
                              traffic=None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1000.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["call_frac"] == pytest.approx(0.25)
    assert r["traffic"] is None


def test_measured_peaks_are_positive_and_name_their_source():
    p = bench.measured_peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["bf16_tflops_sustained"] > 0
    have_file = os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json"))
    assert p["source"] == ("measured" if have_file else "fallback")


def _tiny_sparse_workload():
    c = synth.sparse_bf16(B=2, T=600, K=100)
    wl = bench.SparseDecode.__new__(bench.SparseDecode)
    wl.c = c
    inp = synth.make_sparse_inputs(c, 1001, device="cpu")
    wl.q, wl.k, wl.v, wl.idx = inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"]
    wl.rows = c.B * c.Hq
    wl._host = dict(q=wl.q, idx=wl.idx, k=wl.k, v=wl.v)
    return wl


def test_cpu_baseline_repeats_whole_passes_up_to_the_budget():
    wl = _tiny_sparse_workload()
    r = bench.cpu_baseline(wl, types.SimpleNamespace(), budget_s=0.3)
    assert r["kind"] == "oracle" and r["unit"] == "query-rows/s"
    assert r["cores"] == (os.cpu_count() or 1)
    assert r["value"] > 0
    # one pass over the 128 rows is far shorter than the budget: whole passes repeat
    assert r["sample"].endswith(f"passes over all {wl.rows} query-rows of one step")
    passes = int(r["sample"].split()[0])
    assert passes >= 2
    assert r["value"] == pytest.approx(passes * wl.rows / r["seconds"], rel=0.02)


def test_traffic_entries_name_known_workloads_and_kernels():
    """Every recorded DRAM-traffic figure belongs to a workload the bench runs
    and to a kernel whose sources it hashes."""
    import synth
    names = {synth.sparse_bf16().name, synth.paged_fp16().name, synth.prefill_bf16().name,
             synth.csa_fp8().name, synth.csa_ratio4_ref().name, synth.index_select_fp4().name,
             "compress_r4"}
    for workload, (kernel, nbytes, digest, how) in bench.TRAFFIC.items():
        assert workload in names, workload
        assert kernel in bench.KERNEL_SOURCES, kernel
        assert nbytes > 0 and len(digest) == 16 and how


def test_traffic_is_withheld_when_the_sources_change(monkeypatch):
    workload, (kernel, nbytes, digest, _) = next(iter(bench.TRAFFIC.items()))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: digest)
    assert bench.traffic_for(workload, kernel) == nbytes
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
    assert bench.traffic_for(workload, kernel) is None
    assert bench.traffic_for("no_such_workload", kernel) is None
