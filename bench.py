"""Benchmark of the KV-cache attention hot path on GB300.

Default workload: selected-token decode, bf16, B32 Hq64 Hkv8 D128, cache
8192 tokens, 2048 selected indices per (batch, KV head) row (about 5% of rows
padded).  One step = one sparse_attn_decode call that appends the current
token's K/V into the cache, validates the index rows on the device, gathers
the selected K/V rows and merges the partial softmax results (three kernels).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Prints one JSON line.  Timing: CUDA events around each step on the launching
stream, with an L2 flush (a 512 MB write, then a 256 MB read that writes the
flush's dirty lines back) between steps outside the events.  The roofline
divides the dominant kernel's algorithmic bytes (or flops) by its live
duration, taken in a separate pass in which the library records CUDA events
around that one kernel (sa.kernel_events); the whole call's figures sit beside.
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


def max_over_ranks(x: float, device) -> float:
    """The largest of the ranks' values, returned on every rank (replicas: the
    job takes as long as its slowest rank); x itself when not distributed."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    if torch.distributed.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (weak scaling: every rank runs the same per-rank work)."""
    return units_per_rank_step * world * steps / (total_ms * 1e-3)


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

class Staging:
    """Several tensors as 256-byte-aligned slices of one device buffer, with a
    pinned host twin: a step's inputs (or outputs) cross in one copy.  The
    device slices replace the original tensors (same shapes, dtypes, data)."""

    def __init__(self, tensors, dev):
        offs, off = [], 0
        for t in tensors:
            off = (off + 255) // 256 * 256
            offs.append(off)
            off += t.numel() * t.element_size()
        self.nbytes = off
        self.dev = torch.empty(max(off, 1), dtype=torch.uint8, device=dev)
        self.host = torch.empty(max(off, 1), dtype=torch.uint8).pin_memory()
        self.views = []
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            v = self.dev[o:o + n].view(t.dtype).view(t.shape)
            v.copy_(t)
            self.host[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
            self.views.append(v)

    def h2d(self):
        self.dev.copy_(self.host, non_blocking=True)
        return self.nbytes

    def d2h(self):
        self.host.copy_(self.dev, non_blocking=True)
        return self.nbytes


class SparseDecode:
    """Selected-token decode step (append + validate + gather decode)."""

    metric = METRIC

    def __init__(self, sa, c: synth.SparseCase, dev, seed=1001):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_sparse_inputs(c, seed, device=dev)
        self.k, self.v = inp["k_cache"], inp["v_cache"]
        # the step's inputs and outputs in one staging buffer each (e2e leg)
        self.s_in = Staging([inp["q"], inp["idx"], inp["k_cur"], inp["v_cur"]], dev)
        self.q, self.idx, self.k_cur, self.v_cur = self.s_in.views
        self.write_pos = torch.full((c.B,), c.T - c.cur, dtype=torch.int64, device=dev)
        self.s_out = Staging([torch.empty((c.B, c.Hq, 1, c.D), dtype=self.q.dtype, device=dev),
                              torch.zeros(1, dtype=torch.int32, device=dev)], dev)
        self.y, self.err = self.s_out.views
        self.status = torch.empty(c.B * c.I, dtype=torch.uint8, device=dev)
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
        return self.s_in.h2d()  # Q, indices, current token's K and V

    def d2h(self):
        return self.s_out.d2h()  # Y and the error word

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

    def roofline(self, decode_ms, kernel_ms, peaks):
        # the gather kernel: each valid selected K and V row once, Q read, Y written
        es = self.q.element_size()
        kbytes = self.valid * 2 * self.c.D * es + self.q.numel() * es + self.y.numel() * es
        return hbm_roofline("gather_stream_kernel", kbytes, kernel_ms, self.decode_bytes,
                            decode_ms, peaks, traffic_for(self.c.name, "gather_stream_kernel"))


class PagedDecode:
    """Paged causal decode step: write the new token into the page pool and
    attend over each sequence's whole context (one query per sequence)."""

    metric = METRIC

    def __init__(self, sa, c: synth.PagedCase, dev, seed=1005):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_paged_inputs(c, seed, device=dev)
        self.inp = inp
        self.s_in = Staging([inp["q"], inp["k_new"], inp["v_new"]], dev)
        self.q, inp["k_new"], inp["v_new"] = self.s_in.views
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.s_out = Staging([torch.empty_like(self.q)], dev)
        self.y = self.s_out.views[0]
        nws = sa.paged_attn_decode_workspace(self.q, inp["k_pool"], inp["v_pool"],
                                             inp["block_table"], inp["ctx_len"],
                                             scale=c.eff_scale())
        self.ws = sa.new_workspace(nws, dev)
        self.rows = c.B * c.Hq
        es = self.q.element_size()
        tokens = int(inp["ctx_len"].sum().item())
        self.tokens = tokens
        self.decode_bytes = (tokens * c.Hkv * c.D * es * 2 + inp["block_table"].numel() * 4
                             + 2 * self.q.numel() * es + 2 * inp["k_new"].numel() * es * 2)
        self.launches_per_step = 3  # paged append, gather, combine

    def step(self, ev=None):
        i = self.inp
        if ev is not None:
            ev[0].record()
        self.sa.paged_attn_decode(self.q, i["k_pool"], i["v_pool"], i["block_table"],
                                  i["ctx_len"], k_new=i["k_new"], v_new=i["v_new"],
                                  scale=self.c.eff_scale(), err_word=self.err, y=self.y,
                                  workspace=self.ws)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        return self.s_in.h2d()  # Q and the new token's K and V

    def d2h(self):
        return self.s_out.d2h()  # Y

    def config(self):
        c = self.c
        return {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
                "head_dim": c.D, "ctx_range": [c.ctx_low, c.ctx_high], "page_tokens":
                c.page_tokens, "context_tokens": self.tokens,
                "step": "paged_attn_decode: new-token append + stream-K gather over pages "
                        "+ combine"}

    def oracle_rows(self, rows):
        import oracle
        c, i = self.c, self.inp
        out = []
        if not hasattr(self, "_host"):
            self._host = {}
        for r in rows:
            b, h = divmod(r, c.Hq)
            if b not in self._host:
                n = int(i["ctx_len"][b])
                pages = i["block_table"][b, : (n + c.page_tokens - 1) // c.page_tokens].long()
                self._host[b] = (i["q"][b:b + 1].cpu(), i["k_pool"][pages].cpu(),
                                 i["v_pool"][pages].cpu(), n)
            q, kp, vp, n = self._host[b]
            table = torch.arange(kp.shape[0], dtype=torch.int32)[None]
            y = oracle.paged_decode(q, kp, vp, table, torch.tensor([n], dtype=torch.int32),
                                    page_tokens=c.page_tokens, scale=c.eff_scale(), rows=[h])
            out.append(y[0])
        return np.stack(out)

    def roofline(self, decode_ms, kernel_ms, peaks):
        # the gather kernel: every context token's K and V rows, the table, Q and Y
        es = self.q.element_size()
        kbytes = (self.tokens * self.c.Hkv * self.c.D * es * 2 + self.inp["block_table"].numel() * 4
                  + 2 * self.q.numel() * es)
        return hbm_roofline("gather_stream_kernel (paged)", kbytes, kernel_ms, self.decode_bytes,
                            decode_ms, peaks, traffic_for(self.c.name, "gather_stream_kernel"))


class Prefill:
    """Dense causal prefill step with present K/V emission."""

    metric = "dense causal prefill tokens/s and tensor-core TFLOP/s (1 GB300)"

    def __init__(self, sa, c: synth.PrefillCase, dev, seed=1004):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_prefill_inputs(c, seed, device=dev)
        self.s_in = Staging([inp["q"], inp["k"], inp["v"]], dev)
        self.q, self.k, self.v = self.s_in.views
        self.pk, self.pv = torch.empty_like(self.k), torch.empty_like(self.v)
        self.s_out = Staging([torch.empty_like(self.q)], dev)
        self.y = self.s_out.views[0]
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        nws = sa.attn_prefill_workspace(self.q, self.k, self.v, True, c.eff_scale(), c.softcap)
        self.ws = sa.new_workspace(nws, dev)
        self.rows = c.B * c.S  # tokens
        S = c.S
        pairs = S * (S + 1) // 2 if c.causal else S * S
        self.flops = 4.0 * c.D * pairs * c.B * c.Hq
        self.launches_per_step = 1  # one tensor-core kernel; present K/V written inside it

    def step(self, ev=None):
        c = self.c
        if ev is not None:
            ev[0].record()
        self.sa.attn_prefill(self.q, self.k, self.v, causal=c.causal, scale=c.eff_scale(),
                             softcap=c.softcap, y=self.y, present_k=self.pk, present_v=self.pv,
                             workspace=self.ws)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        return self.s_in.h2d()  # Q, K, V

    def d2h(self):
        return self.s_out.d2h()  # Y

    def config(self):
        c = self.c
        return {"workload": c.name, "batch": c.B, "seq_len": c.S, "q_heads": c.Hq,
                "kv_heads": c.Hkv, "head_dim": c.D, "causal": c.causal, "softcap": c.softcap,
                "step": "attn_prefill with present K/V"}

    def oracle_rows(self, rows):
        import oracle
        c = self.c
        if not hasattr(self, "_host"):
            self._host = (self.q.cpu(), self.k.cpu(), self.v.cpu())
        q, k, v = self._host
        # each requested unit is one token (all its query heads), spread over
        # the batch and positions
        stride = max(1, (c.B * c.S) // max(len(rows), 1))
        picked = []
        for r in rows:
            tok = (r * stride) % (c.B * c.S)
            b, i = divmod(tok, c.S)
            picked += [(b * c.Hq + h) * c.S + i for h in range(c.Hq)]
        return oracle.prefill(q, k, v, scale=c.eff_scale(), causal=c.causal, softcap=c.softcap,
                              rows=picked)

    def roofline(self, ms, kernel_ms, peaks):
        return tensor_roofline("prefill_tc05_kernel", self.flops, kernel_ms, ms, peaks,
                               traffic_for(self.c.name, "prefill_tc05_kernel"))


class CsaFp8Decode:
    """Selected-token decode over the hybrid FP8 latent cache: a dense window of
    the last 128 tokens united with 2048 selected indices, 128 query heads on
    one 576-dim latent head (512 E4M3 + 64 bf16 dims, 648-byte records)."""

    metric = METRIC

    def __init__(self, sa, c: synth.SparseCase, dev, seed=1003):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_sparse_inputs(c, seed, device=dev)
        self.rec = inp["kv_records"]
        self.s_in = Staging([inp["q"], inp["idx"]], dev)
        self.q, self.idx = self.s_in.views
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.status = torch.empty(c.B * c.I, dtype=torch.uint8, device=dev)
        self.s_out = Staging([torch.empty_like(self.q)], dev)
        self.y = self.s_out.views[0]
        nws = sa.sparse_attn_decode_workspace(self.q, self.rec, None, self.idx,
                                              scale=c.eff_scale(), window=c.window,
                                              n_rope=c.n_rope, err_word=self.err,
                                              row_status=self.status)
        self.ws = sa.new_workspace(nws, dev)
        self.rows = c.B * c.Hq
        # candidates: the window plus the selected entries below it (an entry
        # inside the window is the same key, counted once)
        valid = int(((self.idx >= 0) & (self.idx < c.T - c.window)).sum().item())
        self.keys = valid + c.B * c.window
        self.decode_bytes = (self.keys * c.record_stride + self.idx.numel() * 4
                             + 2 * self.q.numel() * 2)
        self.flops = 4.0 * c.Hq * c.D * self.keys
        # plan (validation only), gather-decode (positions, records), tcgen05
        # attention, combine (when the splits are not merged on chip; 128-head
        # blocks) -- else plan, warp-MMA kernel, combine
        self.launches_per_step = 4 if c.Hq % 128 == 0 else 3

    def step(self, ev=None):
        c = self.c
        if ev is not None:
            ev[0].record()
        self.sa.sparse_attn_decode(self.q, self.rec, None, self.idx, scale=c.eff_scale(),
                                   window=c.window, n_rope=c.n_rope, y=self.y,
                                   workspace=self.ws, err_word=self.err, row_status=self.status)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        return self.s_in.h2d()  # Q and the indices

    def d2h(self):
        return self.s_out.d2h()  # Y

    def config(self):
        c = self.c
        return {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "latent_heads": c.Hkv,
                "head_dim": c.D, "fp8_dims": c.D - c.n_rope, "rope_dims": c.n_rope,
                "record_bytes": c.record_stride, "cache_tokens": c.T, "top_k": c.K,
                "window": c.window, "keys_attended": self.keys,
                "step": "sparse_attn_decode on FP8 records: plan kernel (validation, window "
                        "union positions) + gather-decode kernel (exact bf16 rows) + tcgen05 "
                        "attention kernel + split combine"}

    def oracle_rows(self, rows):
        import oracle
        c = self.c
        if not hasattr(self, "_host"):
            self._host = {}
        out = []
        for r in rows:
            b, h = divmod(r, c.Hq)
            if b not in self._host:
                self._host[b] = (self.q[b:b + 1].cpu(), self.idx[b:b + 1].cpu(),
                                 self.rec[b:b + 1].cpu())
            q, idx, rec = self._host[b]
            out.append(oracle.sparse_attention(q, idx, records=rec, n_rope=c.n_rope,
                                               scale=c.eff_scale(), window=c.window,
                                               rows=[h])[0])
        return np.stack(out)

    def roofline(self, ms, kernel_ms, peaks):
        # every flop of the call is in the tensor-core attention kernel
        kern = "fp8_tc05_kernel" if self.c.Hq % 128 == 0 else "fp8_decode_kernel"
        line = tensor_roofline(kern, self.flops, kernel_ms, ms, peaks,
                               traffic_for(self.c.name, kern))
        gbs = self.decode_bytes / (ms * 1e-3) / 1e9
        line.update(algorithmic_bytes=int(self.decode_bytes), call_hbm_gbs=round(gbs, 1),
                    call_hbm_frac=round(gbs / peaks["hbm_gbs"], 4))
        return line


class IndexSelect:
    """Ratio-4 index scoring and top-k selection (the producer of the selected
    indices): B16 decode rows at position 65,535, 16,384 index records of 128
    FP4 dims (68 bytes), 64 index heads, top-k 2,048."""

    metric = "ratio-4 index-select query-rows/s (FP4 index scoring + top-k 2048) on 1 GB300"
    dtype_name = "int8 (FP4 E2M1 codes, dp4a) + f32"
    data_desc = ("synthetic (seeded N(0,1) index queries and head weights; FP4 index records "
                 "with codes drawn from a fixed distribution, scale bytes 124..127)")

    def __init__(self, sa, c: synth.IndexCase, dev, seed=1006):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_index_inputs(c, seed, device=dev)
        self.keys = inp["keys"]                     # resident, like the index-key cache
        self.s_in = Staging([inp["query"], inp["weight"]], dev)
        self.query, self.weight = self.s_in.views
        self.s_out = Staging([torch.empty((c.B, 1, c.S, c.topk), dtype=torch.int32, device=dev),
                              torch.zeros(1, dtype=torch.int32, device=dev)], dev)
        self.sel, self.err = self.s_out.views
        self.status = torch.empty(c.B * c.S, dtype=torch.uint8, device=dev)
        nws = sa.sparse_index_select_workspace(self.query, self.weight, self.keys, topk=c.topk)
        self.ws = sa.new_workspace(nws, dev)
        self.rows = c.B * c.S
        limits = [min(c.R, (c.query_start + s + 1) // 4) for s in range(c.S)] * c.B
        self.records = int(sum(limits))
        # integer multiply-adds of the exact dot products: one per (record, head, dim)
        self.macs = float(self.records) * c.IH * c.ID
        self.decode_bytes = (self.records * c.stride + self.query.numel() * 4
                             + self.weight.numel() * 4 + self.sel.numel() * 4)
        self.launches_per_step = 3  # query finalize, scores, top-k

    def step(self, ev=None):
        c = self.c
        if ev is not None:
            ev[0].record()
        self.sa.sparse_index_select(self.query, self.weight, self.keys, topk=c.topk,
                                    query_start=c.query_start, selected=self.sel,
                                    workspace=self.ws, err_word=self.err,
                                    row_status=self.status)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        return self.s_in.h2d()  # index queries and head weights

    def d2h(self):
        return self.s_out.d2h()  # selected indices and the error word

    def config(self):
        c = self.c
        return {"workload": c.name, "batch": c.B, "queries": c.S, "index_heads": c.IH,
                "index_dim": c.ID, "records": c.R, "top_k": c.topk,
                "query_position": c.query_start, "record_bytes": c.stride,
                "equal_scores": "the synthetic FP4 keys give equal scores in some rows: the "
                                "device ranks them by record and flags them (err_word "
                                "SA_ERRBIT_SEL_TIE = 512), as the oracle does",
                "step": "one sparse_index_select call: query finalize (bf16, Hadamard, FP4), "
                        "scores (exact dp4a block dots), top-k (hash tie check, radix select, "
                        "merge sort) -- 3 kernels"}

    def oracle_rows(self, rows):
        import oracle
        c = self.c
        if not hasattr(self, "_host"):
            self._host = (self.query.cpu(), self.weight.cpu(), self.keys.cpu())
        q, w, k = self._host
        out = []
        for r in rows:
            b, s = divmod(r, c.S)
            sel, _, _ = oracle.index_select(q[b:b + 1, s:s + 1], w[b:b + 1, s:s + 1],
                                            k[b:b + 1], topk=c.topk, query_start=c.query_start + s)
            out.append(sel[0, 0, 0])
        return np.stack(out)

    def roofline(self, ms, kernel_ms, peaks):
        # the score kernel: integer dp4a, bound by the SMs' integer pipes
        dp4a_peak = DP4A_PER_SM_PER_CLOCK * SMS * SM_MAX_GHZ * 1e9 * 4 * 2 / 1e12  # TOP/s
        ops = 2.0 * self.macs
        achieved = ops / (kernel_ms * 1e-3) / 1e12
        call = ops / (ms * 1e-3) / 1e12
        return {"bound": "alu", "kernel": "index_score_kernel", "achieved": round(achieved, 2),
                "peak": round(dp4a_peak, 1), "unit": "TOP/s (int8 multiply + add)",
                "frac": round(achieved / dp4a_peak, 4),
                "traffic": traffic_for(self.c.name, "index_score_kernel"),
                "peak_source": "derived: 152 SMs x %d dp4a per SM per clock x 2.07 GHz "
                               "(measured dp4a issue rate) x 4 multiply-adds" %
                               DP4A_PER_SM_PER_CLOCK,
                "algorithmic_ops": ops, "kernel_us": round(kernel_ms * 1e3, 2),
                "call_us": round(ms * 1e3, 2), "call_achieved": round(call, 2),
                "call_frac": round(call / dp4a_peak, 4),
                "algorithmic_bytes": int(self.decode_bytes),
                "call_hbm_gbs": round(self.decode_bytes / (ms * 1e-3) / 1e9, 1)}


class CsaRef:
    """Compressed sparse attention (ratio 4) in the pages' own form: B16 decode
    rows, 128 heads over one 512-dim latent head, a 128-token current_kv window
    plus 2,048 selected hybrid-FP8 records (583 bytes) of 16,384, sink."""

    metric = METRIC
    dtype_name = "bf16 (FP8 E4M3 records decoded exactly)"

    def __init__(self, sa, c: synth.CsaCase, dev, seed=1007):
        self.sa, self.c, self.dev = sa, c, dev
        inp = synth.make_csa_inputs(c, seed, device=dev)
        self.window, self.records = inp["window"], inp["records"]   # resident, like the caches
        self.s_in = Staging([inp["query"], inp["selected"]], dev)
        self.q, self.sel = self.s_in.views
        self.sink = torch.linspace(-1.0, 1.0, c.H, dtype=torch.float32, device=dev)
        self.s_out = Staging([torch.empty_like(self.q), torch.zeros(1, dtype=torch.int32,
                                                                    device=dev)], dev)
        self.y, self.err = self.s_out.views
        nws = sa.csa_ratio4_attention_workspace(self.q, self.window, self.records, self.sel,
                                                total=c.total, n_rope=c.n_rope, sink=self.sink)
        self.ws = sa.new_workspace(nws, dev)
        self.rows = c.B * c.S * c.H
        valid_sel = int((self.sel >= 0).sum().item())
        self.keys = valid_sel + c.B * c.S * min(c.L, 128)
        es = self.q.element_size()
        self.flops = 4.0 * c.H * c.D * self.keys
        self.decode_bytes = (valid_sel * c.stride + c.B * c.S * min(c.L, 128) * c.D * es
                             + 2 * self.q.numel() * es + self.sel.numel() * 4)
        self.launches_per_step = 3  # assemble, attention, split merge (2 when merged on chip)

    def step(self, ev=None):
        c = self.c
        if ev is not None:
            ev[0].record()
        self.sa.csa_ratio4_attention(self.q, self.window, self.records, self.sel, total=c.total,
                                     n_rope=c.n_rope, sink=self.sink, y=self.y,
                                     workspace=self.ws, err_word=self.err)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        return self.s_in.h2d()  # queries and selected records

    def d2h(self):
        return self.s_out.d2h()  # y and the error word

    def config(self):
        c = self.c
        return {"workload": c.name, "batch": c.B, "queries": c.S, "heads": c.H, "dim": c.D,
                "rope_dims": c.n_rope, "window_rows": c.L, "tokens": c.total,
                "records": c.R, "top_k": c.topk, "record_bytes": c.stride,
                "step": "one csa_ratio4_attention call: candidate assembly (window rows, "
                        "FP8 record decode), tcgen05 attention with sink (128-head blocks, "
                        "two CTAs of 256 output dims; key splits merged on chip in clusters, "
                        "else by a split-merge kernel) -- 2 or 3 kernels"}

    def oracle_rows(self, rows):
        import oracle
        c = self.c
        if not hasattr(self, "_host"):
            self._host = (self.q.cpu(), self.window.cpu(), self.records.cpu(), self.sel.cpu(),
                          self.sink.cpu().double())
        q, w, rec, sel, sink = self._host
        out = []
        for r in rows:
            bs, h = divmod(r, c.H)
            b = bs // c.S
            y, _ = oracle.csa_ratio4_attention(q[b:b + 1], w[b:b + 1], rec[b:b + 1],
                                               sel[b:b + 1], total=c.total, n_rope=c.n_rope,
                                               sink=sink)
            out.append(y.reshape(-1, c.D)[(bs % c.S) * c.H + h])
        return np.stack(out)

    def roofline(self, ms, kernel_ms, peaks):
        # 128-head blocks of bf16 queries run on the tcgen05 attention kernel
        # (fp8_tc05_kernel in its 512-dim geometry)
        line = tensor_roofline("fp8_tc05_kernel", self.flops, kernel_ms, ms, peaks,
                               traffic_for(self.c.name, "fp8_tc05_kernel"))
        line.update(call_algorithmic_bytes=int(self.decode_bytes),
                    call_hbm_gbs=round(self.decode_bytes / (ms * 1e-3) / 1e9, 1))
        return line


class Compress:
    """One ratio-4 layer's compression stages over a prefill chunk: B16, 4,096
    new tokens per sequence ending at position 65,536; the attention-record
    stream (D 512: 448 E4M3 + 64 bf16 RoPE, 583-byte records) and the
    index-key stream (D 128, 64 RoPE, FP4, 68-byte keys)."""

    metric = "CSA compression tokens/s (ratio-4 attention records + index keys) on 1 GB300"
    unit = "tokens/s"
    dtype_name = "f32 (binary32 pooling and RMSNorm; E4M3 / E2M1 records)"
    data_desc = ("synthetic (seeded N(0,1) compressor values and gates, N(0,1)/2 positional "
                 "score biases, 1 + N(0,1)/10 norm scales; carry in the state of position "
                 "61,440)")
    chunk = 64  # tokens per oracle unit of the CPU baseline

    def __init__(self, sa, dev, seed=1008):
        self.sa, self.dev = sa, dev
        self.cm, self.ci = synth.compress_r4(0), synth.compress_r4(1)
        im = synth.make_compress_inputs(self.cm, seed, device=dev)
        ii = synth.make_compress_inputs(self.ci, seed + 1, device=dev)
        self.s_in = Staging([im["kv"], im["gate"], ii["kv"], ii["gate"]], dev)
        self.kv_m, self.g_m, self.kv_i, self.g_i = self.s_in.views
        self.ape_m, self.norm_m, self.carry_m = im["ape"], im["norm"], im["carry"]
        self.ape_i, self.norm_i, self.carry_i = ii["ape"], ii["norm"], ii["carry"]
        cm, ci = self.cm, self.ci
        self.rec_m = torch.zeros((cm.B, cm.R, cm.width), dtype=torch.uint8, device=dev)
        self.rec_i = torch.zeros((ci.B, ci.R, ci.width), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.k0 = cm.start // 4
        self.nk = cm.total // 4 - self.k0
        self.h_rec_m = torch.empty((cm.B, self.nk, cm.width), dtype=torch.uint8).pin_memory()
        self.h_rec_i = torch.empty((ci.B, self.nk, ci.width), dtype=torch.uint8).pin_memory()
        self.h_err = torch.empty(1, dtype=torch.int32).pin_memory()
        self.rows = cm.B * cm.S  # tokens per step
        self.oracle_row_count = cm.B * cm.S // self.chunk
        self.oracle_row_units = self.chunk
        # algorithmic bytes: every new token's value and gate rows once, the
        # previous block's four carry slots, the records written, the carry
        # rewritten (8 slots x 2 channels x W per sequence); ape and norm
        # (a few KB, cache resident) left out
        def stream_bytes(c):
            src = c.B * c.S * 2 * c.W * 4
            rec = c.B * self.nk * c.width
            return src, rec, c.B * 4 * 2 * c.W * 4, c.B * 8 * 2 * c.W * 4
        sm, rm, pm, cym = stream_bytes(cm)
        si, ri, pi, cyi = stream_bytes(ci)
        self.kernel_bytes = sm + rm + pm // 2  # the records kernel reads half of each slot
        self.call_bytes = sm + rm + pm // 2 + cym + si + ri + pi // 2 + cyi
        self.launches_per_step = 4  # two streams: records kernel + carry kernel each

    def step(self, ev=None):
        sa, cm, ci = self.sa, self.cm, self.ci
        if ev is not None:
            ev[0].record()
        # the index stream first, so that the library's measurement events
        # (recorded around each call's record kernel) end on the main stream's
        sa.csa_ratio4_index_compress(self.kv_i, self.g_i, self.ape_i, self.norm_i, self.carry_i,
                                     n_rope=ci.n_rope, total=ci.total, records=self.rec_i,
                                     err_word=self.err)
        sa.csa_ratio4_main_compress(self.kv_m, self.g_m, self.ape_m, self.norm_m, self.carry_m,
                                    n_rope=cm.n_rope, total=cm.total, records=self.rec_m,
                                    err_word=self.err)
        if ev is not None:
            ev[1].record()

    def h2d(self):
        return self.s_in.h2d()  # the chunk's value and gate rows of both streams

    def d2h(self):
        # the records this step wrote (rows k0.. of every sequence) and the error word
        for b in range(self.cm.B):
            self.h_rec_m[b].copy_(self.rec_m[b, self.k0:], non_blocking=True)
            self.h_rec_i[b].copy_(self.rec_i[b, self.k0:], non_blocking=True)
        self.h_err.copy_(self.err, non_blocking=True)
        return self.h_rec_m.numel() + self.h_rec_i.numel() + 4

    def config(self):
        cm, ci = self.cm, self.ci
        return {"workload": cm.name.replace("_attn", "") + "_main_and_index",
                "batch": cm.B, "new_tokens": cm.S, "position_end": cm.total, "ratio": 4,
                "record_dim": cm.D, "record_rope_dims": cm.n_rope, "record_bytes": cm.width,
                "index_dim": ci.D, "index_rope_dims": ci.n_rope, "index_key_bytes": ci.width,
                "records_per_sequence": self.nk,
                "step": "csa_ratio4_index_compress + csa_ratio4_main_compress: per stream a "
                        "record kernel (softmax pool of 8 candidates, RMSNorm, RoPE, "
                        "FP8 / Hadamard + FP4) and a carry kernel -- 4 kernels"}

    def oracle_rows(self, rows):
        import oracle
        if not hasattr(self, "_host"):
            self._host = [(c, tuple(t.cpu() for t in ts)) for c, ts in (
                (self.cm, (self.kv_m, self.g_m, self.ape_m, self.norm_m, self.carry_m)),
                (self.ci, (self.kv_i, self.g_i, self.ape_i, self.norm_i, self.carry_i)))]
        n = self.chunk
        per_b = self.cm.S // n
        for r in rows:
            b, ch = divmod(r, per_b)
            lo, hi = ch * n, ch * n + n
            # one 64-token chunk of both streams from the carry (positions from
            # the chunk's start: the same work as at the step's own positions)
            for c, (kv, g, ape, norm, cy) in self._host:
                oracle.csa_compress(kv[b:b + 1, lo:hi], g[b:b + 1, lo:hi], ape, norm,
                                    cy[b:b + 1], ratio=4, kind=c.kind, n_rope=c.n_rope,
                                    total=hi, rows=hi // 4)

    def roofline(self, ms, kernel_ms, peaks):
        return hbm_roofline("compress_r4_kernel", self.kernel_bytes, kernel_ms, self.call_bytes,
                            ms, peaks, traffic_for("compress_r4", "compress_r4_kernel"))


SMS = 152
SM_MAX_GHZ = 2.07
# dp4a issue rate: 16 per SM sub-partition per clock (a probe kernel measured
# about 60 per SM per clock on this part)
DP4A_PER_SM_PER_CLOCK = 64


# DRAM bytes (read + write) per launch of the dominant kernel from an ncu
# capture, keyed by workload, each with the hash of the kernel's source files
# at capture time (kernel_source_hash): a value whose hash no longer matches
# the current sources is reported as null (stale), never as a measurement.
KERNEL_SOURCES = {
    "gather_stream_kernel": ["k_stream.cu", "gather_common.cuh", "common.cuh", "tc05.cuh",
                             "kernels.h"],
    "fp8_tc05_kernel": ["k_fp8_tc.cu", "e4m3.cuh", "gather_common.cuh", "common.cuh", "tc05.cuh",
                        "kernels.h"],
    "fp8_decode_kernel": ["k_fp8.cu", "e4m3.cuh", "gather_common.cuh", "common.cuh", "kernels.h"],
    "prefill_tc05_kernel": ["k_prefill.cu", "common.cuh", "tc05.cuh", "kernels.h"],
    "index_score_kernel": ["k_index.cu", "codes.cuh", "common.cuh", "kernels.h"],
    "compress_r4_kernel": ["k_compress.cu", "codes.cuh", "common.cuh", "kernels.h"],
    "csa_attn_kernel": ["k_csa.cu", "e4m3.cuh", "gather_common.cuh", "common.cuh", "kernels.h"],
}

TRAFFIC: dict = {
    # workload: (kernel, bytes per launch, source hash at capture, how)
    "csa_fp8_b16_h128_d576_t65536_k2048_w128": (
        "fp8_tc05_kernel", 42_666_496, "4d5499920cc78155",
        "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch of the bench's own "
        "workload (42.67 MB read, 0 written; ncu starts each kernel with cold caches, so the "
        "decoded rows are read from DRAM here and from L2 in a live call)"),
    "index_select_b16_ih64_id128_r16384_k2048": (
        "index_score_kernel", 18_047_232, "7b8479ac54a89ab1",
        "ncu --set full, one launch of the bench's own workload (18.05 MB read, 0 written: the "
        "index records once)"),
    "csa_ref_b16_h128_d512_l128_t65536_k2048": (
        "fp8_tc05_kernel", 37_858_048, "4d5499920cc78155",
        "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch of the bench's own "
        "workload (37.86 MB read, 1,280 B written; cold caches under ncu, as above)"),
    "compress_r4": ("compress_r4_kernel", 546_426_624, "89fe5929934292d9",
                    "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch of the "
                    "bench's own workload (536.98 MB read, 9.45 MB written)"),
    "sparse_bf16_b32_h64_kv8_d128_t8192_k2048": (
        "gather_stream_kernel", 274_255_872, "96f01ec1f92b7531",
        "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch of the bench's own "
        "workload (270.69 MB read, 3.57 MB written)"),
    "paged_fp16_b128_h32_kv8_d128_ctx1k-32k_p16": (
        "gather_stream_kernel", 8_926_250_739, "96f01ec1f92b7531",
        "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch of the same "
        "sequences' distribution at 16 sequences (workload paged_fp16_b16: 1,159.68 MB, 1.0034 x "
        "its algorithmic bytes), scaled by the algorithmic bytes to the 128-sequence batch"),
    "prefill_bf16_b4_s4096_h32_kv8_d128_causal_softcap50": (
        "prefill_tc05_kernel", 427_458_048, "b003441e58206e07",
        "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch of the bench's own "
        "workload (272.07 MB read, 155.39 MB written: part of Y and the present K/V is still in "
        "L2 when the kernel ends)"),
}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_top_kv_validate_gb300", "csrc")
    for name in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def traffic_for(workload: str, kernel: str):
    """ncu DRAM bytes per launch for this workload's dominant kernel, or None
    when no capture of the current kernel source exists."""
    rec = TRAFFIC.get(workload)
    if not rec or rec[0] != kernel or rec[2] != kernel_source_hash(kernel):
        return None
    return rec[1]


def hbm_roofline(kernel, kbytes, kernel_ms, call_bytes, call_ms, peaks, traffic):
    """HBM roofline of the dominant kernel (its algorithmic bytes over its live
    event-bracketed duration), with the whole call's figures beside it."""
    achieved = kbytes / (kernel_ms * 1e-3) / 1e9
    call = call_bytes / (call_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic, "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "peak_source": peaks["source"] + " (copy bandwidth, burst)",
            "algorithmic_bytes": int(kbytes), "kernel_us": round(kernel_ms * 1e3, 2),
            "call_algorithmic_bytes": int(call_bytes), "call_us": round(call_ms * 1e3, 2),
            "call_achieved": round(call, 1), "call_frac": round(call / peaks["hbm_gbs"], 4)}


def tensor_roofline(kernel, flops, kernel_ms, call_ms, peaks, traffic):
    """Tensor roofline of the dominant kernel, with the whole call beside it."""
    tf = flops / (kernel_ms * 1e-3) / 1e12
    call = flops / (call_ms * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": kernel, "achieved": round(tf, 2),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(tf / peaks["bf16_tflops"], 4), "traffic": traffic,
            "peak_source": peaks["source"] + " (cuBLAS bf16, burst)",
            "algorithmic_flops": flops, "kernel_us": round(kernel_ms * 1e3, 2),
            "call_us": round(call_ms * 1e3, 2), "call_achieved": round(call, 2),
            "call_frac": round(call / peaks["bf16_tflops"], 4)}


def unit_of(wl) -> str:
    return getattr(wl, "unit", None) or ("tokens/s" if isinstance(wl, Prefill)
                                         else "query-rows/s")


def make_workload(sa, name, dev):
    if name in ("sparse_bf16", "default"):
        return SparseDecode(sa, synth.sparse_bf16(), dev)
    if name == "tiny_sparse":
        return SparseDecode(sa, synth.tiny_sparse(), dev)
    if name == "paged_fp16":
        return PagedDecode(sa, synth.paged_fp16(), dev)
    if name == "paged_fp16_b16":  # the same sequences' distribution at 1/8 the batch (ncu-sized)
        return PagedDecode(sa, synth.paged_fp16(
            B=16, name="paged_fp16_b16_h32_kv8_d128_ctx1k-32k_p16"), dev)
    if name == "csa_fp8":
        return CsaFp8Decode(sa, synth.csa_fp8(), dev)
    if name == "prefill_bf16":
        return Prefill(sa, synth.prefill_bf16(), dev)
    if name == "index_select":
        return IndexSelect(sa, synth.index_select_fp4(), dev)
    if name == "csa_ref":
        return CsaRef(sa, synth.csa_ratio4_ref(), dev)
    if name == "compress_r4":
        return Compress(sa, dev)
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

# The other workloads, measured after the headline in the default run (one GPU)
# so that one bench line carries every workload's figures.
SECONDARY = ["csa_fp8", "paged_fp16", "prefill_bf16", "index_select", "csa_ref", "compress_r4"]


def measure_secondary(sa, name, dev, flush_l2, peaks, steps=20):
    """One more workload in the same process by the headline's protocol at fewer
    steps: CUDA graph replay of one step, L2 flushed between steps outside the
    events, the dominant kernel timed by events captured as graph nodes.  Its
    buffers are released afterwards."""
    wl = make_workload(sa, name, dev)
    graph = kgraph = None
    try:
        stream = torch.cuda.current_stream(dev)
        for _ in range(3):
            flush_l2()
            wl.step()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            wl.step()
        torch.cuda.synchronize(dev)
        graph.replay()
        torch.cuda.synchronize(dev)
        st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush_l2()
            st[i].record(stream)
            graph.replay()
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        step_ms = [a.elapsed_time(b) for a, b in zip(st, en)]
        kb, ka = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with sa.kernel_events(kb, ka):
            kgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(kgraph):
                wl.step()
        torch.cuda.synchronize(dev)
        ks = []
        for _ in range(min(steps, 10)):
            flush_l2()
            kgraph.replay()
            torch.cuda.synchronize(dev)
            ks.append(kb.elapsed_time(ka))
        rl = wl.roofline(statistics.median(step_ms), statistics.median(ks), peaks)
        keep = ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic", "kernel_us",
                "call_us")
        return {"value": round(job_rate(wl.rows, 1, steps, sum(step_ms)), 1),
                "unit": unit_of(wl), "ms_per_step": round(sum(step_ms) / steps, 5),
                "steps": steps, "workload": wl.config()["workload"],
                "roofline": {k: rl.get(k) for k in keep}, "err_word": int(wl.err.item())}
    finally:
        del graph, kgraph, wl
        torch.cuda.empty_cache()


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
    # L2 flush between steps, outside the events: a 512 MB write evicts the
    # step's inputs, then a 256 MB read of another buffer writes the flush's own
    # dirty lines back, so that this write-back does not land in the next step
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    clean = torch.ones(128 * 1024 * 1024, dtype=torch.float16, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        sink.copy_(clean.sum(dtype=torch.float32))
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        flush_l2()
        wl.step()
    torch.cuda.synchronize(dev)

    # The timed steps replay a CUDA graph of one library call (the call's
    # launches, captured once; the buffers are fixed), so that the host's own
    # argument marshalling does not leave the GPU idle inside a step.
    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                wl.step()
            torch.cuda.synchronize(dev)
            graph.replay()
            torch.cuda.synchronize(dev)
        except Exception as exc:  # capture refused: time the direct calls
            print(f"# CUDA graph capture failed ({exc}); timing direct calls", file=sys.stderr)
            graph = None

    # the library's kernels in one step: counted from the captured graph's
    # kernel nodes (the step is one library call, nothing else), else stated
    launches = wl.launches_per_step
    launches_how = "stated by the workload"
    if graph is not None:
        try:  # a second capture of the step, kept as a graph to read, never replayed
            cg = torch.cuda.CUDAGraph(keep_graph=True)
            with torch.cuda.graph(cg):
                wl.step()
            torch.cuda.synchronize(dev)
            launches = sa.graph_kernel_count(cg)
            launches_how = "kernel nodes of the captured step"
            del cg
        except Exception as exc:  # no graph introspection: the stated count
            print(f"# graph kernel count failed ({exc}); using the stated count", file=sys.stderr)

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
            flush_l2()
            starts[i].record(stream)
            if graph is not None:
                graph.replay()
            else:
                wl.step(dec[i])
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if ws > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # the call alone: the step with a graph, else the events inside step()
    dec_ms = step_ms if graph is not None else [a.elapsed_time(b) for a, b in dec]
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / steps
    value = job_rate(wl.rows, ws, steps, total_ms)

    # end-to-end leg: host buffers, copies inside the timed region
    e2e_steps = max(3, min(steps, 200))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    h2d = d2h = 0

    def e2e_step():
        nonlocal h2d, d2h
        h2d = wl.h2d()
        wl.step()
        d2h = wl.d2h()
    # As the timed steps: a graph of the step (copy in, the call, copy out),
    # replayed, unless --no-graph or the capture is refused.
    e2e_graph = None
    if graph is not None:
        try:
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph):
                e2e_step()
            torch.cuda.synchronize(dev)
            e2e_graph.replay()
            torch.cuda.synchronize(dev)
        except Exception as exc:
            print(f"# e2e graph capture failed ({exc}); timing direct calls", file=sys.stderr)
            e2e_graph = None
    for i in range(e2e_steps):
        flush_l2()
        e_s[i].record(stream)
        if e2e_graph is not None:
            e2e_graph.replay()
        else:
            e2e_step()
        e_e[i].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / e2e_steps, dev)
    # hot-L2 leg: the same step back to back with no flush in between (what a
    # workload smaller than L2 sees when it repeats); reported beside the
    # flushed figure, never as the value
    hot_steps = max(3, min(steps, 50))
    h_s, h_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h_s.record(stream)
    for _ in range(hot_steps):
        if graph is not None:
            graph.replay()
        else:
            wl.step()
    h_e.record(stream)
    torch.cuda.synchronize(dev)
    hot_ms = max_over_ranks(h_s.elapsed_time(h_e) / hot_steps, dev)
    # dominant-kernel leg: the library records events around its dominant
    # kernel (sa.kernel_events); same flush protocol, separate from the timed
    # steps because recording between kernels removes their launch overlap.
    # With a graph the events are nodes of a second captured step, so that no
    # host launch latency falls between them.
    k_steps = max(3, min(steps, 50))
    kernel_samples = []
    kgraph = None
    if graph is not None:
        kb, ka = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        try:
            with sa.kernel_events(kb, ka):
                kgraph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(kgraph):
                    wl.step()
            torch.cuda.synchronize(dev)
        except Exception as exc:
            print(f"# kernel-event graph capture failed ({exc}); timing direct calls",
                  file=sys.stderr)
            kgraph = None
    if kgraph is not None:
        for i in range(k_steps):
            flush_l2()
            kgraph.replay()
            torch.cuda.synchronize(dev)
            kernel_samples.append(kb.elapsed_time(ka))
    else:
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k_steps)]
        for i in range(k_steps):
            flush_l2()
            with sa.kernel_events(*kev[i]):
                wl.step()
        torch.cuda.synchronize(dev)
        kernel_samples = [a.elapsed_time(b) for a, b in kev]
    kernel_ms = statistics.median(kernel_samples)
    err = int(wl.err.item())

    if rank == 0:
        peaks = measured_peaks()
        line = {
            "metric": wl.metric,
            "value": round(value, 1),
            "unit": unit_of(wl),
            "n_gpus": ws,
            "steps": steps,
            "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": getattr(wl, "dtype_name", None)
            or str(wl.q.dtype).replace("torch.", "").replace("bfloat16", "bf16"),
            "data": getattr(wl, "data_desc", None)
            or "synthetic (seeded N(0,1) Q/K/V, uniform sorted top-k indices)",
            "config": dict(wl.config(), parallelism=f"replicas x{ws}" if ws > 1 else "single GPU",
                           l2="flushed between steps outside the step events: a 512 MB write, "
                              "then a 256 MB read that writes the flush's dirty lines back",
                           timing="sum of per-step CUDA events on the launching stream",
                           launch="CUDA graph replay of one library call per step"
                           if graph is not None else "direct library call per step"),
            "roofline": wl.roofline(statistics.median(dec_ms), kernel_ms, peaks),
            "e2e": {"value": round(job_rate(wl.rows, ws, 1, e2e_ms), 1),
                    "unit": unit_of(wl),
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 5),
                    "launch": "CUDA graph replay of the H2D copy, the library call and "
                              "the D2H copy per step" if e2e_graph is not None
                              else "direct copies and library call per step"},
            "hot_l2": {"ms_per_step": round(hot_ms, 5), "steps": hot_steps,
                       "note": "steps back to back, L2 not flushed"},
            "gpu_launches": launches * steps,
            "launches_per_step": {"value": launches, "how": launches_how},
            "clocks": clk.summary(),
            "wall_s_timed_region": round(wall, 4),
            "err_word": err,
        }
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, args)
        if ws == 1 and args.workload in ("sparse_bf16", "default") and not args.no_secondary:
            # after the headline's timed region; each workload's own events
            others = {}
            del graph, e2e_graph, kgraph
            with ClockSampler(dev) as clk2:
                for name in SECONDARY:
                    try:
                        others[name] = measure_secondary(sa, name, dev, flush_l2, peaks)
                    except Exception as exc:  # one failed workload leaves the line intact
                        others[name] = {"error": f"{type(exc).__name__}: {exc}"[:200]}
            line["other_workloads"] = dict(others, clocks=clk2.summary(),
                                           note="measured after the headline by the same "
                                                "protocol at 20 steps; not part of value")
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


class OraclePool:
    """A persistent pool of host threads, one per core, each running the C
    oracle (ctypes releases the GIL) on its share of the rows."""

    def __init__(self, wl, threads):
        import concurrent.futures as cf
        self.wl, self.threads = wl, threads
        self.ex = cf.ThreadPoolExecutor(max_workers=threads)

    def run(self, rows):
        chunks = [rows[i::self.threads] for i in range(self.threads)]
        list(self.ex.map(self.wl.oracle_rows, [ch for ch in chunks if ch]))

    def close(self):
        self.ex.shutdown(wait=True)


def cpu_baseline(wl, args, budget_s: float = 10.0):
    """The fp64 oracle as it stands, on the host cores, over a bounded sample
    of the same workload's rows (a persistent pool of one thread per core):
    part of the step's rows, or whole passes over all of them repeated when
    one pass is shorter than the budget."""
    cores = os.cpu_count() or 1
    pool = OraclePool(wl, cores)
    wl.oracle_rows([0])  # stage host copies outside the timing
    per_row = getattr(wl, "oracle_row_units", 1)  # workload units one oracle row covers
    rows_all = list(range(getattr(wl, "oracle_row_count", wl.rows)))
    n = min(len(rows_all), cores * 4)
    t0 = time.perf_counter()
    pool.run(rows_all[:n])
    dt = time.perf_counter() - t0
    if dt < budget_s and n < len(rows_all):
        n2 = min(len(rows_all), max(n, int(n * budget_s / max(dt, 1e-3))))
        t0 = time.perf_counter()
        pool.run(rows_all[:n2])
        dt = time.perf_counter() - t0
        n = n2
    unit = unit_of(wl)
    what = unit.split('/')[0]
    sample = f"{n * per_row} of {len(rows_all) * per_row} {what} of one step"
    if dt < budget_s and n == len(rows_all):
        passes = min(1000, max(2, math.ceil(budget_s / max(dt, 1e-3))))
        t0 = time.perf_counter()
        for _ in range(passes):
            pool.run(rows_all)
        dt = time.perf_counter() - t0
        n = passes * len(rows_all)
        sample = f"{passes} passes over all {len(rows_all) * per_row} {what} of one step"
    pool.close()
    return {"value": round(n * per_row / dt, 2), "unit": unit, "cores": cores,
            "kind": "oracle", "sample": sample, "seconds": round(dt, 3)}


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
    pool = OraclePool(wl, cores)
    rows = list(range(wl.rows))
    wl.oracle_rows([0])  # host copies staged outside the timing
    # a step is one whole pass over the step's query rows; if K + W such passes
    # would take more than about two minutes, each step takes an equal share
    t0 = time.perf_counter()
    pool.run(rows)
    t_pass = time.perf_counter() - t0
    per_step = len(rows)
    budget = 120.0
    if t_pass * (args.steps + args.warmup) > budget:
        per_step = max(cores, int(len(rows) * budget / (t_pass * (args.steps + args.warmup))))
    for i in range(args.warmup):
        s = (i * per_step) % wl.rows
        pool.run((rows[s:] + rows[:s])[:per_step])
    t0 = time.perf_counter()
    for i in range(args.steps):
        s = (i * per_step) % wl.rows
        pool.run((rows[s:] + rows[:s])[:per_step])
    dt = time.perf_counter() - t0
    pool.close()
    value = args.steps * per_step / dt
    sample = (f"{per_step} of the {wl.rows} query rows of the step per step" if per_step < wl.rows
              else f"every step a whole pass over all {wl.rows} query rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "query-rows/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
                   "head_dim": c.D, "cache_tokens": c.T, "top_k": c.K},
        "cpu_baseline": {"value": round(value, 2), "unit": "query-rows/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
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
    ap.add_argument("--no-secondary", action="store_true",
                    help="default workload only: skip the other workloads' figures")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct library calls instead of a CUDA graph of one call")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
