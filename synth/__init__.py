"""Seeded synthetic inputs for the KV-cache attention hot path.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the oracle tests and the CUDA path take their
inputs from here, so the two sides see identical bytes.

Every generator is deterministic in ``seed``. Large tensors are drawn with a
``torch.Generator`` on the requested device (so an 8 GB paged pool does not
have to be produced on the host); small ones may be drawn on the CPU.

Workload shapes follow the five decode/prefill cases of the problem statement:

* ``tiny_sparse``      fp32 selected-token decode, B1 Hq4 Hkv1 D64, past 256 + 1
* ``sparse_bf16``      bf16 selected-token decode, B32 Hq64 Hkv8 D128 T8192 K2048
* ``csa_fp8``          FP8 block-64 latent cache, B16 Hq128 MQA D576, T65536,
                       window 128 united with top-k 2048
* ``prefill_bf16``     dense causal prefill, B4 S4096 Hq32 Hkv8 D128, softcap 50
* ``paged_fp16``       paged causal decode, B128, ctx ~ U[1024, 32768], 16-token pages
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

__all__ = [
    "normal",
    "sorted_sample_rows",
    "pad_tails",
    "quantize_fp8_block64_records",
    "paged_layout",
    "SparseCase",
    "PrefillCase",
    "PagedCase",
    "tiny_sparse",
    "sparse_bf16",
    "csa_fp8",
    "prefill_bf16",
    "paged_fp16",
    "make_sparse_inputs",
    "make_prefill_inputs",
    "make_paged_inputs",
    "IndexCase",
    "index_select_fp4",
    "fp4_index_records",
    "make_index_inputs",
    "CsaCase",
    "csa_ratio4_ref",
    "make_csa_inputs",
    "CompressCase",
    "compress_r4",
    "compress_r128",
    "make_compress_inputs",
]

_TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal(shape, dtype: str, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) values drawn in fp32 and rounded (RNE) to the storage dtype."""
    g = _gen(seed, device)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return x.to(_TORCH_DT[dtype])


def sorted_sample_rows(rows: int, low: int, high: int, k: int, seed: int,
                       device="cpu") -> torch.Tensor:
    """``rows`` rows of ``k`` distinct integers drawn uniformly from
    ``[low, high)`` without replacement, each row sorted ascending (int64)."""
    n = high - low
    if k > n:
        raise ValueError(f"cannot draw {k} distinct values from a range of {n}")
    g = _gen(seed, device)
    out = torch.empty((rows, k), dtype=torch.int64, device=device)
    # Random keys per candidate, keep the k smallest keys: a uniform k-subset.
    step = max(1, (1 << 26) // max(n, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        keys = torch.rand((r1 - r0, n), generator=g, device=device)
        pick = torch.topk(keys, k, dim=1, largest=False, sorted=False).indices
        out[r0:r1] = torch.sort(pick, dim=1).values + low
    return out


def pad_tails(idx: torch.Tensor, seed: int, prob: float, max_pad: int,
              min_pad: int = 1) -> torch.Tensor:
    """Replace a seeded trailing run of each selected row by ``-1``.

    A row is chosen with probability ``prob``; its pad count is uniform in
    ``[min_pad, max_pad]`` (never the whole row). The largest indices are the
    ones dropped, so the remaining prefix stays strictly increasing.
    """
    rows, k = idx.shape
    rng = np.random.default_rng(seed)
    chosen = rng.random(rows) < prob
    counts = rng.integers(min_pad, max_pad + 1, size=rows)
    counts = np.minimum(counts, k - 1)
    out = idx.clone()
    col = torch.arange(k, device=idx.device)
    lim = torch.tensor(np.where(chosen, k - counts, k), device=idx.device)
    out[col[None, :] >= lim[:, None]] = -1
    return out


def quantize_fp8_block64_records(nope: torch.Tensor, rope: torch.Tensor,
                                 record_stride: int | None = None) -> torch.Tensor:
    """Pack rows into hybrid FP8 records (test-data generation only).

    ``nope`` is ``[..., n_nope]`` (n_nope a multiple of 64), ``rope`` is
    ``[..., n_rope]`` bf16. Each record is ``n_nope/64`` blocks of
    ``[E8M0 scale byte, 64 E4M3FN codes]`` followed by the RoPE dims as
    little-endian bf16. The block exponent is the smallest ``e`` with
    ``amax / 2**e <= 448`` (an all-zero block gets byte 127); codes are the
    round-to-nearest-even E4M3FN encoding of ``x / 2**e``.
    """
    lead = nope.shape[:-1]
    n_nope = nope.shape[-1]
    n_rope = rope.shape[-1]
    if n_nope % 64:
        raise ValueError("non-RoPE width must be a multiple of 64")
    nb = n_nope // 64
    width = nb * 65 + 2 * n_rope
    stride = width if record_stride is None else record_stride
    if stride < width:
        raise ValueError("record stride smaller than the record")
    x = nope.to(torch.float32).reshape(-1, nb, 64)
    amax = x.abs().amax(dim=2)
    e = torch.zeros_like(amax, dtype=torch.int32)
    nz = amax > 0
    e[nz] = torch.ceil(torch.log2(amax[nz] / 448.0)).to(torch.int32)
    # Correct for log2 rounding so that amax / 2**e <= 448 holds exactly.
    for _ in range(2):
        too_big = nz & (amax / torch.exp2(e.to(torch.float32)) > 448.0)
        e = e + too_big.to(torch.int32)
    e = torch.clamp(e, -127, 127)
    scaled = x / torch.exp2(e.to(torch.float32))[:, :, None]
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8)
    n = x.shape[0]
    rec = torch.zeros((n, stride), dtype=torch.uint8, device=nope.device)
    blocks = rec[:, : nb * 65].view(n, nb, 65)
    blocks[:, :, 0] = (e + 127).to(torch.uint8)
    blocks[:, :, 1:] = codes
    rb = rope.to(torch.bfloat16).reshape(n, n_rope).contiguous().view(torch.int16)
    rb = rb.to(torch.int32) & 0xFFFF
    tail = rec[:, nb * 65: nb * 65 + 2 * n_rope].view(n, n_rope, 2)
    tail[:, :, 0] = (rb & 0xFF).to(torch.uint8)
    tail[:, :, 1] = (rb >> 8).to(torch.uint8)
    return rec.reshape(*lead, stride)


def paged_layout(B: int, ctx_low: int, ctx_high: int, page_tokens: int,
                 seed: int, extra_pages: int = 0):
    """Per-sequence context lengths ~ U[ctx_low, ctx_high] and a block table
    that maps each sequence's logical pages onto a seeded random permutation
    of one shared page pool. Returns ``(ctx_len i32 [B], block_table i32
    [B, max_pages], num_pages)``; unused table slots hold ``-1``."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_low, ctx_high + 1, size=B).astype(np.int32)
    pages = (ctx + page_tokens - 1) // page_tokens
    max_pages = int(math.ceil(ctx_high / page_tokens))
    num_pages = int(pages.sum()) + extra_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, : pages[b]] = perm[off: off + pages[b]]
        off += pages[b]
    return torch.from_numpy(ctx), torch.from_numpy(table), num_pages


# --------------------------------------------------------------------------
# Workload descriptions
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class SparseCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T: int                 # cache length (past + current), also the row stride
    K: int                 # selected-index width
    I: int                 # index heads: 1, Hkv or Hq
    dtype: str             # "f32", "f16", "bf16" or "fp8" (hybrid records)
    pad_prob: float = 0.0  # probability that a row gets a -1 tail
    pad_max: int = 0
    pad_min: int = 1
    window: int = 0        # dense window of recent tokens united with the top-k
    n_rope: int = 0        # FP8 only: bf16 RoPE dims at the end of a record
    record_stride: int = 0 # FP8 only: bytes between records (0 = packed)
    softcap: float = 0.0
    scale: float = 0.0     # 0 => 1/sqrt(D)
    idx_i64: bool = False
    cur: int = 1           # tokens appended this step

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def rows(self) -> int:
        return self.B * self.Hq

    def eff_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class PrefillCase:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    causal: bool = True
    softcap: float = 0.0
    scale: float = 0.0
    dtype: str = "bf16"

    def eff_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class PagedCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    ctx_low: int
    ctx_high: int
    page_tokens: int = 16
    dtype: str = "f16"
    scale: float = 0.0

    def eff_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.D)


def tiny_sparse(**kw) -> SparseCase:
    """fp32, B1 Hq4 Hkv1 D64, past 256 + 1 current, per-head rows of 32
    indices from [0, 257) with 0..8 trailing -1 pads, scale 1/8."""
    base = SparseCase("tiny_sparse_f32", B=1, Hq=4, Hkv=1, D=64, T=257, K=32, I=4,
                      dtype="f32", pad_prob=1.0, pad_max=8, pad_min=0, scale=0.125)
    return replace(base, **kw)


def sparse_bf16(**kw) -> SparseCase:
    """bf16, B32 Hq64 Hkv8 D128, cache 8192 (8191 past + 1 current), 2048
    indices per (batch, KV head) row, about 5% rows padded."""
    base = SparseCase("sparse_bf16_b32_h64_kv8_d128_t8192_k2048", B=32, Hq=64, Hkv=8,
                      D=128, T=8192, K=2048, I=8, dtype="bf16", pad_prob=0.05,
                      pad_max=256)
    return replace(base, **kw)


def csa_fp8(**kw) -> SparseCase:
    """FP8 hybrid latent cache, B16 Hq128 over one latent head, 512 E4M3
    dims + 64 bf16 RoPE dims (648-byte records), T 65536, window 128 united
    with 2048 sorted uniform indices, scale 1/sqrt(576)."""
    base = SparseCase("csa_fp8_b16_h128_d576_t65536_k2048_w128", B=16, Hq=128, Hkv=1,
                      D=576, T=65536, K=2048, I=1, dtype="fp8", window=128, n_rope=64,
                      record_stride=648)
    return replace(base, **kw)


def prefill_bf16(**kw) -> PrefillCase:
    base = PrefillCase("prefill_bf16_b4_s4096_h32_kv8_d128_causal_softcap50", B=4, S=4096,
                       Hq=32, Hkv=8, D=128, causal=True, softcap=50.0)
    return replace(base, **kw)


def paged_fp16(**kw) -> PagedCase:
    base = PagedCase("paged_fp16_b128_h32_kv8_d128_ctx1k-32k_p16", B=128, Hq=32, Hkv=8,
                     D=128, ctx_low=1024, ctx_high=32768)
    return replace(base, **kw)


# --------------------------------------------------------------------------
# Input builders
# --------------------------------------------------------------------------

def make_sparse_inputs(c: SparseCase, seed: int, device="cpu") -> dict:
    """Q ``[B,Hq,1,D]``, a KV cache of ``T`` positions whose last ``cur`` are
    the current token(s) (also returned separately as ``k_cur``/``v_cur``), and
    ``selected_indices`` ``[B, I, 1, K]``.

    For the FP8 case the cache is ``[B, 1, T, record_stride]`` bytes (K and V
    are the same latent record) and Q is bf16."""
    out = {}
    qdt = "bf16" if c.dtype == "fp8" else c.dtype
    out["q"] = normal((c.B, c.Hq, 1, c.D), qdt, seed * 7919 + 1, device)
    if c.dtype == "fp8":
        n_nope = c.D - c.n_rope
        stride = c.record_stride or (n_nope // 64 * 65 + 2 * c.n_rope)
        nope = normal((c.B, c.T, n_nope), "f32", seed * 7919 + 2, device)
        rope = normal((c.B, c.T, c.n_rope), "bf16", seed * 7919 + 3, device)
        rec = quantize_fp8_block64_records(nope, rope, stride)
        out["kv_records"] = rec.reshape(c.B, 1, c.T, stride)
    else:
        out["k_cache"] = normal((c.B, c.Hkv, c.T, c.D), c.dtype, seed * 7919 + 2, device)
        out["v_cache"] = normal((c.B, c.Hkv, c.T, c.D), c.dtype, seed * 7919 + 3, device)
        out["k_cur"] = out["k_cache"][:, :, c.T - c.cur:, :].clone()
        out["v_cur"] = out["v_cache"][:, :, c.T - c.cur:, :].clone()
    rows = c.B * c.I
    # the selected indices are drawn from the whole cache, also with a window:
    # entries inside the window overlap it (about K * window / T per row)
    idx = sorted_sample_rows(rows, 0, c.T, c.K, seed * 7919 + 4, device)
    if c.pad_prob > 0 and c.pad_max > 0:
        idx = pad_tails(idx, seed * 7919 + 5, c.pad_prob, c.pad_max, c.pad_min)
    idx = idx.reshape(c.B, c.I, 1, c.K)
    out["idx"] = idx if c.idx_i64 else idx.to(torch.int32)
    return out


def make_prefill_inputs(c: PrefillCase, seed: int, device="cpu") -> dict:
    return {
        "q": normal((c.B, c.Hq, c.S, c.D), c.dtype, seed * 104729 + 1, device),
        "k": normal((c.B, c.Hkv, c.S, c.D), c.dtype, seed * 104729 + 2, device),
        "v": normal((c.B, c.Hkv, c.S, c.D), c.dtype, seed * 104729 + 3, device),
    }


def make_paged_inputs(c: PagedCase, seed: int, device="cpu") -> dict:
    """Pools ``[num_pages, Hkv, page_tokens, D]``; ``ctx_len`` counts the new
    token, whose K/V (``k_new``/``v_new`` ``[B, Hkv, D]``) also sit in the
    pool at slot ``ctx - 1``."""
    ctx, table, num_pages = paged_layout(c.B, c.ctx_low, c.ctx_high, c.page_tokens,
                                         seed * 15485863 + 1)
    shape = (num_pages, c.Hkv, c.page_tokens, c.D)
    k_pool = normal(shape, c.dtype, seed * 15485863 + 2, device)
    v_pool = normal(shape, c.dtype, seed * 15485863 + 3, device)
    ctx_d = ctx.to(device)
    table_d = table.to(device)
    last = (ctx_d - 1).long()
    page = table_d.long().gather(1, (last // c.page_tokens)[:, None])[:, 0]
    slot = last % c.page_tokens
    k_new = k_pool[page, :, slot, :].clone()
    v_new = v_pool[page, :, slot, :].clone()
    return {
        "q": normal((c.B, c.Hq, 1, c.D), c.dtype, seed * 15485863 + 4, device),
        "k_pool": k_pool, "v_pool": v_pool, "k_new": k_new, "v_new": v_new,
        "ctx_len": ctx_d, "block_table": table_d, "num_pages": num_pages,
    }


# --------------------------------------------------------------------------
# Ratio-4 index selection inputs
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class IndexCase:
    name: str
    B: int
    S: int                 # query positions per batch
    IH: int                # index heads
    ID: int                # index head dim (a power of two, a multiple of 32)
    R: int                 # compressed index records per batch (capacity)
    topk: int
    query_start: int       # position of query 0 (the last S positions of the context)
    key_stride: int = 0    # bytes between records (0: ID / 32 * 17)

    @property
    def stride(self) -> int:
        # records padded to a multiple of 4 bytes (68 bytes at ID 128: packed)
        return self.key_stride or (self.ID // 32 * 17 + 3) // 4 * 4


def index_select_fp4(**kw) -> IndexCase:
    """B16 decode rows at the last position of a 65,536-token context: 16,384
    ratio-4 index records of 128 FP4 dims (68 bytes), 64 index heads, top-k
    2,048."""
    base = IndexCase("index_select_b16_ih64_id128_r16384_k2048", B=16, S=1, IH=64, ID=128,
                     R=16384, topk=2048, query_start=65535)
    return replace(base, **kw)


# E2M1 magnitude codes 0..7 (0, 0.5, 1, 1.5, 2, 3, 4, 6) drawn with roughly
# the weights that Gaussian data scaled into [0, 6] per 32-block gives
_E2M1_CODE_WEIGHTS = [0.20, 0.25, 0.20, 0.12, 0.10, 0.08, 0.04, 0.01]


def fp4_index_records(B: int, R: int, ID: int, seed: int, stride: int = 0,
                      device="cpu") -> torch.Tensor:
    """Index-key records ``[B, R, stride]`` uint8: ID/32 blocks of [E8M0 scale
    byte, 16 bytes of E2M1 codes, element 2j in the low nibble of byte j],
    the stride rounded up to a multiple of 4 bytes unless given.
    Codes and scale bytes are drawn directly (magnitudes from a fixed
    categorical distribution, uniform signs, scale bytes 124..127); no
    quantizer is involved."""
    nb = ID // 32
    width = nb * 17
    stride = stride or (width + 3) // 4 * 4
    g = _gen(seed, "cpu")
    w = torch.tensor(_E2M1_CODE_WEIGHTS, dtype=torch.float64)
    mag = torch.multinomial(w, B * R * ID, replacement=True, generator=g).to(torch.uint8)
    sign = torch.randint(0, 2, (B * R * ID,), generator=g, dtype=torch.uint8) << 3
    codes = (mag | sign).reshape(B, R, nb, 16, 2)
    packed = codes[..., 0] | (codes[..., 1] << 4)
    scale = torch.randint(124, 128, (B, R, nb, 1), generator=g, dtype=torch.uint8)
    blocks = torch.cat([scale, packed], dim=3).reshape(B, R, width)
    rec = torch.zeros((B, R, stride), dtype=torch.uint8)
    rec[:, :, :width] = blocks
    return rec.to(device)


def make_index_inputs(c: IndexCase, seed: int, device="cpu") -> dict:
    """Index queries float32 ``[B, S, IH, ID]`` and head weights float32
    ``[B, S, IH]`` ~ N(0, 1), and the FP4 index-key records."""
    return {
        "query": normal((c.B, c.S, c.IH, c.ID), "f32", seed * 49157 + 1, device),
        "weight": normal((c.B, c.S, c.IH), "f32", seed * 49157 + 2, device),
        "keys": fp4_index_records(c.B, c.R, c.ID, seed * 49157 + 3, c.stride, device),
    }


# --------------------------------------------------------------------------
# Compressed sparse attention (ratio 4) in the pages' own form
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class CsaCase:
    name: str
    B: int
    S: int                 # query positions per batch (the last S of the context)
    H: int                 # query heads over one latent head
    D: int                 # logical dims: (D - n_rope) FP8 + n_rope bf16
    n_rope: int
    L: int                 # current_kv rows (the most recent tokens, uncompressed)
    total: int             # tokens so far
    topk: int
    dtype: str = "bf16"    # query and current_kv
    record_stride: int = 0 # 0: packed (7 x 65 + 128 = 583 bytes at D 512)

    @property
    def R(self) -> int:
        return self.total // 4

    @property
    def stride(self) -> int:
        return self.record_stride or ((self.D - self.n_rope) // 64 * 65 + 2 * self.n_rope)


def csa_ratio4_ref(**kw) -> CsaCase:
    """B16 decode rows, 128 heads over one 512-dim latent head (448 E4M3 +
    64 bf16, 583-byte records), a 128-token current_kv window, 65,536 tokens
    (16,384 ratio-4 records), top-k 2,048."""
    base = CsaCase("csa_ref_b16_h128_d512_l128_t65536_k2048", B=16, S=1, H=128, D=512,
                   n_rope=64, L=128, total=65536, topk=2048)
    return replace(base, **kw)


def make_csa_inputs(c: CsaCase, seed: int, device="cpu") -> dict:
    """query ``[B, S, H, D]`` and current_kv ``[B, L, D]`` ~ N(0, 1) in the
    case dtype; ``[B, R, stride]`` hybrid FP8 records quantized from N(0, 1)
    (with ``quantize_fp8_block64_records``); ``selected [B, S, topk]`` int32:
    distinct records below ``(position + 1) / 4`` sampled uniformly (sorted,
    as a top-k in record order), -1 where fewer exist."""
    out = {
        "query": normal((c.B, c.S, c.H, c.D), c.dtype, seed * 31337 + 1, device),
        "window": normal((c.B, c.L, c.D), c.dtype, seed * 31337 + 2, device),
    }
    nope = normal((c.B, c.R, c.D - c.n_rope), "f32", seed * 31337 + 3, device)
    rope = normal((c.B, c.R, c.n_rope), "bf16", seed * 31337 + 4, device)
    out["records"] = quantize_fp8_block64_records(nope, rope, c.stride)
    sel = torch.full((c.B, c.S, c.topk), -1, dtype=torch.int32)
    for s in range(c.S):
        valid = min(c.R, (c.total - c.S + s + 1) // 4)
        k = min(valid, c.topk)
        rows = sorted_sample_rows(c.B, 0, valid, k, seed * 31337 + 5 + s)
        sel[:, s, :k] = rows.to(torch.int32)
    out["selected"] = sel.to(device)
    return out


# --------------------------------------------------------------------------
# CSA compression streams (ratio 4 attention records / index keys, ratio 128)
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class CompressCase:
    name: str
    B: int
    S: int          # new tokens per sequence in this call
    D: int          # record dims (ratio 4 sources are 2 * D wide)
    n_rope: int
    ratio: int      # 4 or 128
    kind: int       # 0 attention record (FP8 + bf16 tail), 1 index key (FP4)
    total: int      # tokens so far, these S included
    rows: int = 0   # record rows per sequence (0: total / ratio)

    @property
    def W(self) -> int:
        return 2 * self.D if self.ratio == 4 else self.D

    @property
    def slots(self) -> int:
        return 8 if self.ratio == 4 else 128

    @property
    def start(self) -> int:
        return self.total - self.S

    @property
    def R(self) -> int:
        return self.rows or self.total // self.ratio

    @property
    def width(self) -> int:
        if self.kind == 0:
            return (self.D - self.n_rope) // 64 * 65 + 2 * self.n_rope
        return self.D // 32 * 17


def compress_r4(kind: int = 0, **kw) -> CompressCase:
    """One ratio-4 layer's chunk: B16, 4,096 new tokens ending at 65,536;
    attention records D 512 (448 E4M3 + 64 bf16 RoPE, 583 bytes) or index
    keys D 128 (64 RoPE, FP4, 68 bytes)."""
    D = 512 if kind == 0 else 128
    base = CompressCase(f"compress_r4_{'attn' if kind == 0 else 'index'}_b16_s4096_t65536_d{D}",
                        B=16, S=4096, D=D, n_rope=64, ratio=4, kind=kind, total=65536)
    return replace(base, **kw)


def compress_r128(**kw) -> CompressCase:
    """A ratio-128 layer's chunk: B16, 4,096 new tokens ending at 65,536,
    D 512 records (583 bytes)."""
    base = CompressCase("compress_r128_b16_s4096_t65536_d512", B=16, S=4096, D=512,
                        n_rope=64, ratio=128, kind=0, total=65536)
    return replace(base, **kw)


def make_compress_inputs(c: CompressCase, seed: int, device="cpu") -> dict:
    """kv, gate ``[B, S, W]`` ~ N(0, 1); ape ``[ratio, W]`` ~ N(0, 1) / 2;
    norm ``[D]`` = 1 + N(0, 1) / 10 (all float32), and a carry ``[B, slots,
    2, W]`` in the state a stream at position ``start`` holds: the slots of
    the positions already seen in the open block (and, for ratio 4, the
    previous block's four slots once a block has closed) carry N(0, 1)
    values and scores, every other slot value 0 and score -inf."""
    out = {
        "kv": normal((c.B, c.S, c.W), "f32", seed * 7919 + 1, device),
        "gate": normal((c.B, c.S, c.W), "f32", seed * 7919 + 2, device),
        "ape": normal((c.ratio, c.W), "f32", seed * 7919 + 3, device) * 0.5,
        "norm": 1.0 + normal((c.D,), "f32", seed * 7919 + 4, device) * 0.1,
    }
    carry = torch.zeros((c.B, c.slots, 2, c.W), dtype=torch.float32)
    carry[:, :, 1, :] = float("-inf")
    vals = normal((c.B, c.slots, 2, c.W), "f32", seed * 7919 + 5)
    st = c.start
    open_from = st - st % c.ratio
    live = []
    if c.ratio == 4:
        live += [4 + (p % 4) for p in range(open_from, st)]
        if open_from >= 4:
            live += [0, 1, 2, 3]
    else:
        live += [p % 128 for p in range(open_from, st)]
    for sl in live:
        carry[:, sl] = vals[:, sl]
    out["carry"] = carry.to(device)
    return out
