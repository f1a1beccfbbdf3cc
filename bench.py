"""Benchmark of the KV-cache attention hot path on GB300.

Default workload: selected-token decode, bf16, B32 Hq64 Hkv8 D128, cache
8192 tokens, 2048 selected indices per (batch, KV head) row (about 5% of rows
padded).  One step = one sparse_attn_decode call that appends the current
token's K/V into the cache, validates the index rows on the device, gathers
the selected K/V rows and merges the partial softmax results (three kernels).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Prints one JSON line.  Timing: CUDA events around each step on the launching
stream, with an L2 flush (a 512 MB write) between steps outside the events;
the decode call itself is bracketed by its own events for the roofline.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sparse-attn decode query-rows/s and achieved HBM GB/s vs ~8 TB/s peak (1 GB300)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                     d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device, interval_ms: int = 20):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(interval_ms)]
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            pass
        self.cmd = cmd

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=1)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class SparseDecode:
    """Selected-token decode step (append + validate + gather decode)."""

    def __init__(self, sa, c: synth.SparseCase, dev, seed=1001):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_sparse_inputs(c, seed, device=dev)
        self.q, self.k, self.v, self.idx = inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"]
        self.k_cur, self.v_cur = inp["k_cur"], inp["v_cur"]
        self.write_pos = torch.full((c.B,), c.T - c.cur, dtype=torch.int64, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.status = torch.empty(c.B * c.I, dtype=torch.uint8, device=dev)
        self.y = torch.empty((c.B, c.Hq, 1, c.D), dtype=self.q.dtype, device=dev)
        nws = sa.sparse_attn_decode_workspace(self.q, self.k, self.v, self.idx,
                                              scale=c.eff_scale(), k_cur=self.k_cur,
                                              v_cur=self.v_cur, write_pos=self.write_pos,
                                              err_word=self.err, row_status=self.status)
        self.ws = sa.new_workspace(nws, dev)
        self.rows = c.B * c.Hq
        self.valid = int((self.idx >= 0).sum().item())
        es = self.q.element_size()
        # algorithmic bytes of the decode call: each valid selected K and V row
        # once, the index rows, Q, Y, and the current token read + written.
        cur_bytes = 2 * self.k_cur.numel() * es
        self.decode_bytes = (self.valid * 2 * c.D * es + self.idx.numel() * self.idx.element_size()
                             + self.q.numel() * es + self.y.numel() * es + 2 * cur_bytes)
        self.launches_per_step = 3  # plan (validate + positions + append), gather, combine
        # host copies for the end-to-end leg
        self.h_q = self.q.cpu().pin_memory()
        self.h_idx = self.idx.cpu().pin_memory()
        self.h_kc = self.k_cur.cpu().pin_memory()
        self.h_vc = self.v_cur.cpu().pin_memory()
        self.h_y = torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory()
        self.h_err = torch.empty(1, dtype=torch.int32).pin_memory()

    def step(self, ev=None):
        sa, c = self.sa, self.c
        if ev is not None:
            ev[0].record()
        sa.sparse_attn_decode(self.q, self.k, self.v, self.idx, scale=c.eff_scale(), y=self.y,
                              workspace=self.ws, k_cur=self.k_cur, v_cur=self.v_cur,
                              write_pos=self.write_pos, err_word=self.err,
                              row_status=self.status)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        self.q.copy_(self.h_q, non_blocking=True)
        self.idx.copy_(self.h_idx, non_blocking=True)
        self.k_cur.copy_(self.h_kc, non_blocking=True)
        self.v_cur.copy_(self.h_vc, non_blocking=True)
        return sum(t.numel() * t.element_size() for t in (self.h_q, self.h_idx, self.h_kc,
                                                           self.h_vc))

    def d2h(self):
        self.h_y.copy_(self.y, non_blocking=True)
        self.h_err.copy_(self.err, non_blocking=True)
        return self.h_y.numel() * self.h_y.element_size() + 4

    def config(self):
        c = self.c
        return {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
                "head_dim": c.D, "cache_tokens": c.T, "top_k": c.K, "index_heads": c.I,
                "padded_row_prob": c.pad_prob, "valid_selected": self.valid,
                "step": "one sparse_attn_decode call: plan kernel (index validation, candidate "
                        "positions, current-token append) + stream-K gather decode + combine of "
                        "split units (3 kernels)"}

    def oracle_rows(self, rows):
        import oracle
        c = self.c
        if not hasattr(self, "_host"):
            self._host = dict(q=self.q.cpu(), idx=self.idx.cpu(), k=self.k.cpu(),
                              v=self.v.cpu())
        h = self._host
        return oracle.sparse_attention(h["q"], h["idx"], h["k"], h["v"], scale=c.eff_scale(),
                                       rows=rows)

    def roofline(self, decode_ms, peaks):
        achieved = self.decode_bytes / (decode_ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": "sparse_attn_decode call (plan + gather_stream + combine)",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                "peak_source": peaks["source"] + " (copy bandwidth, burst)",
                "algorithmic_bytes": int(self.decode_bytes),
                "decode_us": round(decode_ms * 1e3, 2), "traffic": TRAFFIC.get(self.c.name)}


# DRAM bytes (read + write) per decode launch from an ncu capture of the
# dominant kernel, keyed by workload; None until a capture of the current
# kernel exists.
TRAFFIC: dict = {}


def make_workload(sa, name, dev):
    if name in ("sparse_bf16", "default"):
        return SparseDecode(sa, synth.sparse_bf16(), dev)
    if name == "tiny_sparse":
        return SparseDecode(sa, synth.tiny_sparse(), dev)
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import sparse_top_kv_validate_gb300 as sa
    sa.load()
    wl = make_workload(sa, args.workload, dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        wl.step()
    torch.cuda.synchronize(dev)

    steps = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        t0 = time.perf_counter()
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            wl.step(dec[i])
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if ws > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dec_ms = [a.elapsed_time(b) for a, b in dec]
    total_ms = sum(step_ms)
    if ws > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    value = wl.rows * ws * steps / (total_ms * 1e-3)

    # end-to-end leg: host buffers, copies inside the timed region
    e2e_steps = max(3, min(steps, 200))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    h2d = d2h = 0
    for i in range(e2e_steps):
        flush.zero_()
        e_s[i].record(stream)
        h2d = wl.h2d()
        wl.step()
        d2h = wl.d2h()
        e_e[i].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / e2e_steps
    if ws > 1:
        t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    err = int(wl.err.item())

    if rank == 0:
        peaks = measured_peaks()
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "query-rows/s",
            "n_gpus": ws,
            "steps": steps,
            "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": str(wl.q.dtype).replace("torch.", "").replace("bfloat16", "bf16"),
            "data": "synthetic (seeded N(0,1) Q/K/V, uniform sorted top-k indices)",
            "config": dict(wl.config(), parallelism=f"replicas x{ws}" if ws > 1 else "single GPU",
                           l2="flushed between steps (512 MB write outside the step events)",
                           timing="sum of per-step CUDA events on the launching stream"),
            "roofline": wl.roofline(statistics.median(dec_ms), peaks),
            "e2e": {"value": round(wl.rows * ws / (e2e_ms * 1e-3), 1), "unit": "query-rows/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 5)},
            "gpu_launches": wl.launches_per_step * steps,
            "clocks": clk.summary(),
            "wall_s_timed_region": round(wall, 4),
            "err_word": err,
        }
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, args)
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def _oracle_threads(wl, rows, threads):
    chunks = [rows[i::threads] for i in range(threads)]
    out = [None] * threads

    def work(k):
        if chunks[k]:
            out[k] = wl.oracle_rows(chunks[k])

    ts = [threading.Thread(target=work, args=(k,)) for k in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()


def cpu_baseline(wl, args, budget_s: float = 10.0):
    """The fp64 oracle as it stands, on the host cores, over a bounded sample
    of the same workload's rows (ctypes releases the GIL, so one Python thread
    per core runs the C oracle in parallel)."""
    cores = os.cpu_count() or 1
    wl.oracle_rows([0])  # stage host copies outside the timing
    rows_all = list(range(wl.rows))
    n = min(len(rows_all), cores * 4)
    t0 = time.perf_counter()
    _oracle_threads(wl, rows_all[:n], cores)
    dt = time.perf_counter() - t0
    # grow the sample toward the time budget, capped at the whole step
    if dt < budget_s and n < len(rows_all):
        n2 = min(len(rows_all), max(n, int(n * budget_s / max(dt, 1e-3))))
        t0 = time.perf_counter()
        _oracle_threads(wl, rows_all[:n2], cores)
        dt = time.perf_counter() - t0
        n = n2
    return {"value": round(n / dt, 2), "unit": "query-rows/s", "cores": cores,
            "kind": "oracle", "sample": f"{n} of {wl.rows} query rows of one step",
            "seconds": round(dt, 3)}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    torch.set_num_threads(1)
    dev = "cpu"
    c = synth.sparse_bf16()

    class HostWL(SparseDecode):
        def __init__(self, c):
            self.c = c
            inp = synth.make_sparse_inputs(c, 1001, device=dev)
            self.q, self.k, self.v, self.idx = inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"]
            self.rows = c.B * c.Hq
            self._host = dict(q=self.q, idx=self.idx, k=self.k, v=self.v)

    wl = HostWL(c)
    cores = os.cpu_count() or 1
    per_step = cores  # one (batch, head) row per core per step: a bounded sample
    rows = list(range(wl.rows))
    for i in range(args.warmup):
        _oracle_threads(wl, rows[(i * per_step) % wl.rows:][:per_step], cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        s = (i * per_step) % wl.rows
        _oracle_threads(wl, rows[s:s + per_step], cores)
    dt = time.perf_counter() - t0
    value = args.steps * per_step / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "query-rows/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
                   "head_dim": c.D, "cache_tokens": c.T, "top_k": c.K},
        "cpu_baseline": {"value": round(value, 2), "unit": "query-rows/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{per_step} query rows of the workload per step"},
        "e2e": {"value": round(value, 2), "unit": "query-rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sparse_bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
