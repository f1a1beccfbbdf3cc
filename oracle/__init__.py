"""Python entry to the fp64 CPU oracle (``sa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The product library never
imports this package, and this package imports nothing from the product.

Arguments are torch CPU tensors (or numpy arrays) in their storage dtype; the
C code widens them exactly to double itself.  Results come back as float64
numpy arrays.  Every call releases the GIL (ctypes), so disjoint row subsets
can be evaluated from several Python threads at once.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16, FP8REC = 0, 1, 2, 3
IDX_OK = 0
IDX_BELOW_SENTINEL = 1
IDX_AFTER_PADDING = 2
IDX_OUT_OF_RANGE = 4
IDX_NOT_INCREASING = 8
IDX_DUPLICATE = 16
IDX_ALL_PADDING = 32

_i64 = C.c_int64
_p = C.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp,
                    _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _SparseArgs(C.Structure):
    _fields_ = [
        ("q", _p), ("q_dtype", C.c_int), ("k", _p), ("v", _p), ("kv_dtype", C.c_int),
        ("idx", _p), ("idx_is_i64", C.c_int),
        ("B", _i64), ("Hq", _i64), ("Hkv", _i64), ("Sq", _i64), ("D", _i64), ("Dv", _i64),
        ("T", _i64), ("I", _i64), ("K", _i64),
        ("kv_len", _p), ("past_len", _i64), ("causal", C.c_int),
        ("scale", C.c_double), ("softcap", C.c_double), ("window", _i64), ("sink", _p),
        ("record_bytes", _i64), ("n_rope", _i64),
        ("bias", _p), ("bias_rank", _i64), ("bias_dims", _i64 * 4),
    ]


class _SelectArgs(C.Structure):
    _fields_ = [
        ("query", _p), ("weight", _p), ("keys", _p),
        ("B", _i64), ("S", _i64), ("IH", _i64), ("ID", _i64), ("R", _i64), ("topk", _i64),
        ("key_stride", _i64), ("query_start", _i64), ("query_start_b", _p),
        ("out_heads", _i64), ("ascending", C.c_int),
    ]


SEL_TIE, SEL_NONFINITE = 1, 2


class _PrefillMask(C.Structure):
    _fields_ = [("mask", _p), ("kind", C.c_int), ("rank", _i64), ("dims", _i64 * 4),
                ("nonpad", _p)]


MASK_NONE, MASK_F32, MASK_F16, MASK_BF16, MASK_BOOL = 0, 1, 2, 3, 4


class _CsaArgs(C.Structure):
    _fields_ = [
        ("query", _p), ("q_dtype", C.c_int), ("window", _p), ("w_dtype", C.c_int),
        ("records", _p), ("selected", _p), ("sink", _p), ("bias", _p), ("bias_rank", _i64),
        ("bias_dims", _i64 * 4),
        ("B", _i64), ("S", _i64), ("H", _i64), ("D", _i64), ("L", _i64), ("R", _i64),
        ("topk", _i64), ("record_bytes", _i64), ("n_rope", _i64), ("total", _i64),
        ("scale", C.c_double),
    ]


class _CompressArgs(C.Structure):
    _fields_ = [
        ("kv", _p), ("gate", _p), ("ape", _p), ("norm", _p), ("carry", _p),
        ("records", _p), ("logical", _p),
        ("B", _i64), ("S", _i64), ("D", _i64), ("n_rope", _i64), ("ratio", _i64),
        ("kind", _i64), ("rows", _i64), ("record_stride", _i64), ("total", _i64),
    ]


COMPRESS_ATTN, COMPRESS_INDEX = 0, 1


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.orc_f16_to_double.restype = C.c_double
            L.orc_f16_to_double.argtypes = [C.c_uint16]
            L.orc_bf16_to_double.restype = C.c_double
            L.orc_bf16_to_double.argtypes = [C.c_uint16]
            L.orc_e4m3fn_to_double.restype = C.c_double
            L.orc_e4m3fn_to_double.argtypes = [C.c_uint8]
            L.orc_e8m0_to_double.restype = C.c_double
            L.orc_e8m0_to_double.argtypes = [C.c_uint8]
            L.orc_decode_fp8_record.restype = None
            L.orc_decode_fp8_record.argtypes = [_p, _i64, _i64, _p]
            L.orc_validate_row.restype = C.c_int
            L.orc_validate_row.argtypes = [_p, C.c_int, _i64, _i64, C.POINTER(_i64)]
            L.orc_validate_indices.restype = None
            L.orc_validate_indices.argtypes = [_p, C.c_int, _i64, _i64, _i64, _i64, _p, _i64,
                                               _p, _p]
            L.orc_present_concat.restype = None
            L.orc_present_concat.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                             _i64]
            L.orc_present_append.restype = None
            L.orc_present_append.argtypes = [_p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _p]
            L.orc_sparse_attention.restype = C.c_int
            L.orc_sparse_attention.argtypes = [C.POINTER(_SparseArgs), _p, _i64, _p]
            L.orc_prefill.restype = C.c_int
            L.orc_prefill.argtypes = [_p, _p, _p, C.c_int, _i64, _i64, _i64, _i64, _i64,
                                      C.c_int, C.c_double, C.c_double, _p, _i64, _p]
            L.orc_e2m1_to_double.restype = C.c_double
            L.orc_e2m1_to_double.argtypes = [C.c_uint8]
            L.orc_round_bf16.restype = C.c_float
            L.orc_round_bf16.argtypes = [C.c_float]
            L.orc_fp4_quantize_block.restype = None
            L.orc_fp4_quantize_block.argtypes = [_p, _p, _p]
            L.orc_fp4_element.restype = C.c_float
            L.orc_fp4_element.argtypes = [C.c_uint8, _p, C.c_int]
            L.orc_hadamard_bf16.restype = None
            L.orc_hadamard_bf16.argtypes = [_p, _i64]
            L.orc_index_query_finalize.restype = None
            L.orc_index_query_finalize.argtypes = [_p, _i64, _p]
            L.orc_index_select.restype = C.c_int
            L.orc_index_select.argtypes = [C.POINTER(_SelectArgs), _p, _p, _p, _p]
            L.orc_prefill_masked.restype = C.c_int
            L.orc_prefill_masked.argtypes = [_p, _p, _p, C.c_int, _i64, _i64, _i64, _i64, _i64,
                                             C.c_int, C.c_double, C.c_double,
                                             C.POINTER(_PrefillMask), _p, _i64, _p]
            L.orc_csa_ratio4_attention.restype = C.c_int
            L.orc_csa_ratio4_attention.argtypes = [C.POINTER(_CsaArgs), _p, C.POINTER(C.c_int)]
            L.orc_pool_weight.restype = C.c_float
            L.orc_pool_weight.argtypes = [C.c_float]
            L.orc_rope_rotation.restype = None
            L.orc_rope_rotation.argtypes = [_i64, _i64, _p, _p]
            L.orc_fp8_quantize_block.restype = None
            L.orc_fp8_quantize_block.argtypes = [_p, _p]
            L.orc_pool_candidates.restype = C.c_int
            L.orc_pool_candidates.argtypes = [_p, _p, _i64, _i64, _p]
            L.orc_finalize_record.restype = C.c_int
            L.orc_finalize_record.argtypes = [_p, _p, _i64, _i64, C.c_int, _i64, _p]
            L.orc_csa_compress.restype = C.c_int
            L.orc_csa_compress.argtypes = [C.POINTER(_CompressArgs), C.POINTER(_i64)]
            L.orc_paged_decode.restype = C.c_int
            L.orc_paged_decode.argtypes = [_p, _p, _p, C.c_int, _p, _p, _i64, _i64, _i64,
                                           _i64, _i64, _i64, C.c_double, _p, _i64, _p]
            _lib = L
    return _lib


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _host(x):
    """Contiguous CPU torch tensor (kept alive by the caller's reference)."""
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x))
    return x.detach().to("cpu").contiguous()


def _dtype_code(t: torch.Tensor) -> int:
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[t.dtype]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64)).contiguous()
    return r, int(r.numel())


# ---------------------------------------------------------------------------
# scalar decoders
# ---------------------------------------------------------------------------

def f16_to_double(bits: int) -> float:
    return lib().orc_f16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(bits)


def e4m3fn_to_double(code: int) -> float:
    return lib().orc_e4m3fn_to_double(code)


def e8m0_to_double(b: int) -> float:
    return lib().orc_e8m0_to_double(b)


def decode_fp8_record(rec, n_nope: int, n_rope: int) -> np.ndarray:
    r = _host(torch.as_tensor(rec, dtype=torch.uint8))
    out = np.zeros(n_nope + n_rope, dtype=np.float64)
    lib().orc_decode_fp8_record(r.data_ptr(), n_nope, n_rope, out.ctypes.data)
    return out


# ---------------------------------------------------------------------------
# index validation / present KV
# ---------------------------------------------------------------------------

def validate_row(row, bound: int):
    r = _host(torch.as_tensor(row, dtype=torch.int64))
    col = _i64(-1)
    code = lib().orc_validate_row(r.data_ptr(), 1, r.numel(), bound, C.byref(col))
    return code, col.value


def validate_indices(idx, bound: int = 0, bound_per_batch=None):
    """idx ``[B, I, Sq, K]`` int32/int64 → (status uint8 ``[B*I*Sq]``, err)."""
    t = _host(idx)
    B, I, Sq, K = t.shape
    bb = None if bound_per_batch is None else _host(torch.as_tensor(bound_per_batch,
                                                                    dtype=torch.int64))
    status = np.zeros(B * I * Sq, dtype=np.uint8)
    err = C.c_uint32(0)
    lib().orc_validate_indices(t.data_ptr(), int(t.dtype == torch.int64), B, I, Sq, K,
                               _ptr(bb), bound, status.ctypes.data, C.addressof(err))
    return status, err.value


def present_concat(past, cur, out_stride=None):
    """past ``[B,H,P,D]`` (or None), cur ``[B,H,C,D]`` → ``[B,H,stride,D]``
    (positions beyond P+C are zero)."""
    c = _host(cur)
    B, H, Cn, D = c.shape
    if past is None:
        p = torch.empty((B, H, 0, D), dtype=c.dtype)
    else:
        p = _host(past)
    P = p.shape[2]
    stride = P + Cn if out_stride is None else out_stride
    out = torch.zeros((B, H, stride, D), dtype=c.dtype)
    lib().orc_present_concat(p.data_ptr(), c.data_ptr(), out.data_ptr(), c.element_size(),
                             B, H, P, Cn, D, stride)
    return out


def present_append(cache, cur, write_pos):
    """Returns a copy of ``cache [B,H,cap,D]`` with ``cur [B,H,C,D]`` written
    at ``write_pos[b]``."""
    out = _host(cache).clone()
    c = _host(cur)
    B, H, Cn, D = c.shape
    wp = _host(torch.as_tensor(write_pos, dtype=torch.int64))
    lib().orc_present_append(c.data_ptr(), out.data_ptr(), c.element_size(), B, H, Cn, D,
                             out.shape[2], wp.data_ptr())
    return out


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def sparse_attention(q, idx, k=None, v=None, records=None, *, scale: float,
                     softcap: float = 0.0, window: int = 0, kv_len=None,
                     past_len: int = 0, causal: bool = False, sink=None,
                     n_rope: int = 0, Dv=None, rows=None, bias=None) -> np.ndarray:
    """Selected-token attention; see ``orc_sparse_attention``.

    Dense cache: ``k``/``v`` ``[B, Hkv, T, D]``.  FP8: ``records``
    ``[B, Hkv, T, record_bytes]`` uint8 (K and V are the decoded record),
    ``n_rope`` the bf16 tail width, logical ``D = 64*blocks + n_rope``.
    ``bias``: optional float32 tensor of rank <= 4, broadcast right-aligned
    against ``[B, Hq, Sq, T]`` and added to the score of cache position j."""
    qh = _host(q)
    B, Hq, Sq, D = qh.shape
    ih = _host(idx)
    _, I, _, K = ih.shape
    a = _SparseArgs()
    a.q, a.q_dtype = qh.data_ptr(), _dtype_code(qh)
    keep = [qh, ih]
    if records is not None:
        rh = _host(records)
        keep.append(rh)
        a.k = a.v = rh.data_ptr()
        a.kv_dtype = FP8REC
        a.Hkv, a.T = rh.shape[1], rh.shape[2]
        a.record_bytes = rh.shape[3]
        a.n_rope = n_rope
        a.Dv = D if Dv is None else Dv
    else:
        kh, vh = _host(k), _host(v)
        keep += [kh, vh]
        a.k, a.v, a.kv_dtype = kh.data_ptr(), vh.data_ptr(), _dtype_code(kh)
        a.Hkv, a.T = kh.shape[1], kh.shape[2]
        a.Dv = vh.shape[3]
    a.idx, a.idx_is_i64 = ih.data_ptr(), int(ih.dtype == torch.int64)
    a.B, a.Hq, a.Sq, a.D, a.I, a.K = B, Hq, Sq, D, I, K
    kl = None if kv_len is None else _host(torch.as_tensor(kv_len, dtype=torch.int64))
    a.kv_len = _ptr(kl)
    a.past_len, a.causal = past_len, int(causal)
    a.scale, a.softcap, a.window = scale, softcap, window
    sk = None if sink is None else _host(torch.as_tensor(sink, dtype=torch.float64))
    a.sink = _ptr(sk)
    bh = None
    if bias is not None:
        bh = _host(torch.as_tensor(bias)).to(torch.float32)
        if bh.dim() > 4:
            raise ValueError("bias rank exceeds 4")
        a.bias, a.bias_rank = bh.data_ptr(), bh.dim()
        for r_, e_ in enumerate(bh.shape):
            a.bias_dims[r_] = e_
    r, nr = _rows_arg(rows)
    n = nr if r is not None else B * Hq * Sq
    y = np.zeros((n, a.Dv), dtype=np.float64)
    rc = lib().orc_sparse_attention(C.byref(a), _ptr(r), nr, y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the sparse attention shape")
    return y


def prefill(q, k, v, *, scale: float, causal: bool = True, softcap: float = 0.0,
            rows=None, attn_mask=None, nonpad_kv_seqlen=None) -> np.ndarray:
    """Dense prefill; ``attn_mask`` (float32 / float16 / bfloat16 / bool, rank
    <= 4, broadcast against ``[B, Hq, S, S]``) and ``nonpad_kv_seqlen`` (int64
    ``[B]``) as in ``orc_prefill_masked``."""
    qh, kh, vh = _host(q), _host(k), _host(v)
    B, Hq, S, D = qh.shape
    Hkv = kh.shape[1]
    r, nr = _rows_arg(rows)
    n = nr if r is not None else B * Hq * S
    y = np.zeros((n, D), dtype=np.float64)
    if attn_mask is None and nonpad_kv_seqlen is None:
        rc = lib().orc_prefill(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), _dtype_code(qh), B,
                               Hq, Hkv, S, D, int(causal), scale, softcap, _ptr(r), nr,
                               y.ctypes.data)
    else:
        mk = _PrefillMask()
        mh = None
        if attn_mask is not None:
            mh = _host(torch.as_tensor(attn_mask))
            kinds = {torch.float32: MASK_F32, torch.float16: MASK_F16,
                     torch.bfloat16: MASK_BF16, torch.bool: MASK_BOOL}
            mk.kind = kinds[mh.dtype]
            if mh.dtype == torch.bool:
                mh = mh.to(torch.uint8)
            mk.mask, mk.rank = mh.data_ptr(), mh.dim()
            for i_, e_ in enumerate(mh.shape):
                mk.dims[i_] = e_
        npad = None if nonpad_kv_seqlen is None else _host(
            torch.as_tensor(nonpad_kv_seqlen, dtype=torch.int64))
        mk.nonpad = _ptr(npad)
        rc = lib().orc_prefill_masked(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(),
                                      _dtype_code(qh), B, Hq, Hkv, S, D, int(causal), scale,
                                      softcap, C.byref(mk), _ptr(r), nr, y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the prefill shape")
    return y


def paged_decode(q, k_pool, v_pool, block_table, ctx_len, *, page_tokens: int,
                 scale: float, rows=None) -> np.ndarray:
    qh, kp, vp = _host(q), _host(k_pool), _host(v_pool)
    bt = _host(block_table).to(torch.int32)
    cl = _host(ctx_len).to(torch.int32)
    B, Hq = qh.shape[0], qh.shape[1]
    D = qh.shape[-1]
    Hkv = kp.shape[1]
    r, nr = _rows_arg(rows)
    n = nr if r is not None else B * Hq
    y = np.zeros((n, D), dtype=np.float64)
    rc = lib().orc_paged_decode(qh.data_ptr(), kp.data_ptr(), vp.data_ptr(), _dtype_code(qh),
                                bt.data_ptr(), cl.data_ptr(), B, Hq, Hkv, D, page_tokens,
                                bt.shape[1], scale, _ptr(r), nr, y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the paged shape")
    return y


# ---------------------------------------------------------------------------
# ratio-4 index scoring and top-k selection
# ---------------------------------------------------------------------------

def e2m1_to_double(nibble: int) -> float:
    return lib().orc_e2m1_to_double(nibble)


def round_bf16(x: float) -> float:
    return lib().orc_round_bf16(x)


def fp4_quantize_block(x):
    """32 float32 values -> (E8M0 scale byte, 16 packed bytes, the 32
    dequantized values as float32)."""
    xh = _host(torch.as_tensor(x, dtype=torch.float32))
    assert xh.numel() == 32
    sb = C.c_uint8(0)
    packed = (C.c_uint8 * 16)()
    lib().orc_fp4_quantize_block(xh.data_ptr(), C.addressof(sb), C.addressof(packed))
    vals = np.array([lib().orc_fp4_element(sb.value, C.addressof(packed), i) for i in range(32)],
                    dtype=np.float32)
    return sb.value, bytes(packed), vals


def hadamard_bf16(x) -> np.ndarray:
    v = np.array(x, dtype=np.float32).copy()
    lib().orc_hadamard_bf16(v.ctypes.data, v.size)
    return v


def index_query_finalize(x) -> np.ndarray:
    v = np.array(x, dtype=np.float32).copy()
    out = np.zeros_like(v)
    lib().orc_index_query_finalize(v.ctypes.data, v.size, out.ctypes.data)
    return out


def index_select(query, weight, keys, *, topk: int, query_start: int = 0,
                 query_start_b=None, out_heads: int = 1, ascending: bool = False,
                 want_scores: bool = False):
    """Ratio-4 index selection; see ``orc_index_select``.

    query float32 ``[B, S, IH, ID]``, weight float32 ``[B, S, IH]``, keys uint8
    ``[B, R, key_stride]``.  Returns ``(selected int32 [B, out_heads, S, topk],
    status uint8 [B*S], err)`` and, with ``want_scores``, float32 scores
    ``[B, S, R]``."""
    qh = _host(torch.as_tensor(query, dtype=torch.float32))
    wh = _host(torch.as_tensor(weight, dtype=torch.float32))
    kh = _host(torch.as_tensor(keys, dtype=torch.uint8))
    B, S, IH, ID = qh.shape
    R, stride = kh.shape[1], kh.shape[2]
    a = _SelectArgs()
    a.query, a.weight, a.keys = qh.data_ptr(), wh.data_ptr(), kh.data_ptr()
    a.B, a.S, a.IH, a.ID, a.R, a.topk, a.key_stride = B, S, IH, ID, R, topk, stride
    a.query_start = int(query_start)
    qsb = None if query_start_b is None else _host(torch.as_tensor(query_start_b,
                                                                   dtype=torch.int64))
    a.query_start_b = _ptr(qsb)
    a.out_heads, a.ascending = int(out_heads), int(bool(ascending))
    sel = np.zeros((B, out_heads, S, topk), dtype=np.int32)
    status = np.zeros(B * S, dtype=np.uint8)
    err = C.c_uint32(0)
    scores = np.zeros((B, S, R), dtype=np.float32) if want_scores else None
    rc = lib().orc_index_select(C.byref(a), sel.ctypes.data, status.ctypes.data,
                                C.addressof(err), None if scores is None else scores.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the index selection shape")
    if want_scores:
        return sel, status, err.value, scores
    return sel, status, err.value


# ---------------------------------------------------------------------------
# compressed sparse attention, ratio 4, the pages' own form
# ---------------------------------------------------------------------------

def csa_ratio4_attention(query, window, records, selected, *, total: int, n_rope: int,
                         scale: float = 0.0, sink=None, bias=None):
    """See ``orc_csa_ratio4_attention``.  query ``[B, S, H, D]`` and window
    (current_kv) ``[B, L, D]`` float32 or bfloat16; records uint8
    ``[B, R, record_bytes]``; selected int32 ``[B, S, topk]``; sink ``[H]``;
    bias float32 of rank <= 4 broadcast against ``[B, H, S, C]``.  Returns
    ``(y float64 [B, S, H, D], bad_record)``."""
    qh, wh = _host(query), _host(window)
    rh = _host(torch.as_tensor(records, dtype=torch.uint8))
    sh = _host(torch.as_tensor(selected, dtype=torch.int32))
    B, S, H, D = qh.shape
    a = _CsaArgs()
    a.query, a.q_dtype = qh.data_ptr(), _dtype_code(qh)
    a.window, a.w_dtype = wh.data_ptr(), _dtype_code(wh)
    a.records, a.selected = rh.data_ptr(), sh.data_ptr()
    sk = None if sink is None else _host(torch.as_tensor(sink, dtype=torch.float64))
    a.sink = _ptr(sk)
    bh = None
    if bias is not None:
        bh = _host(torch.as_tensor(bias)).to(torch.float32)
        a.bias, a.bias_rank = bh.data_ptr(), bh.dim()
        for r_, e_ in enumerate(bh.shape):
            a.bias_dims[r_] = e_
    a.B, a.S, a.H, a.D = B, S, H, D
    a.L, a.R, a.topk = wh.shape[1], rh.shape[1], sh.shape[2]
    a.record_bytes, a.n_rope, a.total, a.scale = rh.shape[2], n_rope, int(total), float(scale)
    y = np.zeros((B, S, H, D), dtype=np.float64)
    bad = C.c_int(0)
    rc = lib().orc_csa_ratio4_attention(C.byref(a), y.ctypes.data, C.byref(bad))
    if rc != 0:
        raise ValueError("oracle rejected the CSA shape")
    return y, bad.value


# ---------------------------------------------------------------------------
# CSA compression (ratio 128, ratio 4 attention records and index keys)
# ---------------------------------------------------------------------------

def _np(x):
    return x.detach().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x)


def pool_weight(t: float) -> float:
    return lib().orc_pool_weight(float(t))


def rope_rotation(position: int, n_rope: int):
    """(cos, sin) float32 ``[n_rope / 2]`` of the compressed RoPE."""
    cs = np.zeros(max(n_rope // 2, 1), dtype=np.float32)
    sn = np.zeros_like(cs)
    lib().orc_rope_rotation(int(position), int(n_rope), cs.ctypes.data, sn.ctypes.data)
    return cs[: n_rope // 2], sn[: n_rope // 2]


def fp8_quantize_block(x) -> bytes:
    """64 float32 values -> 65 bytes: E8M0 scale byte, then 64 E4M3FN codes."""
    v = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    assert v.size == 64
    out = (C.c_uint8 * 65)()
    lib().orc_fp8_quantize_block(v.ctypes.data, C.addressof(out))
    return bytes(out)


def pool_candidates(value, score):
    """value, score float32 ``[n, D]`` -> (pooled float32 ``[D]``, ok)."""
    v = np.ascontiguousarray(np.asarray(value, dtype=np.float32))
    s = np.ascontiguousarray(np.asarray(score, dtype=np.float32))
    n, D = v.shape
    out = np.zeros(D, dtype=np.float32)
    ok = lib().orc_pool_candidates(v.ctypes.data, s.ctypes.data, n, D, out.ctypes.data)
    return out, bool(ok)


def record_width(D: int, n_rope: int, kind: int) -> int:
    return ((D - n_rope) // 64) * 65 + 2 * n_rope if kind == COMPRESS_ATTN else (D // 32) * 17


def finalize_record(pooled, norm, *, n_rope: int, kind: int, block_start: int):
    """-> (logical float32 ``[D]``, stored bytes, ok)."""
    rec = np.array(pooled, dtype=np.float32).copy()
    nm = np.ascontiguousarray(np.asarray(norm, dtype=np.float32))
    D = rec.size
    out = (C.c_uint8 * record_width(D, n_rope, kind))()
    ok = lib().orc_finalize_record(rec.ctypes.data, nm.ctypes.data, D, n_rope, int(kind),
                                   int(block_start), C.addressof(out))
    return rec, bytes(out), bool(ok)


def csa_compress(kv, gate, ape, norm, carry, *, ratio: int, kind: int, n_rope: int,
                 total: int, rows: int, records=None, logical=None, record_stride=None):
    """One call of the compression stream; see ``orc_csa_compress``.

    kv, gate float32 ``[B, S, W]``; ape ``[ratio, W]``; norm ``[D]``; carry
    ``[B, slots, 2, W]`` (a copy is updated and returned).  ``records`` uint8
    ``[B, rows, stride]`` and ``logical`` float32 ``[B, rows, D]`` hold the
    past records on entry (zeros when None).  Returns ``(records, logical,
    carry, invalid)``."""
    kvh, gh, ah, nh = (np.ascontiguousarray(_np(x), dtype=np.float32)
                       for x in (kv, gate, ape, norm))
    cy = np.array(_np(carry), dtype=np.float32, copy=True, order="C")
    B, S, W = kvh.shape
    D = W // 2 if ratio == 4 else W
    width = record_width(D, n_rope, kind)
    stride = width if record_stride is None else int(record_stride)
    recs = (np.zeros((B, rows, stride), dtype=np.uint8) if records is None
            else np.array(_np(records), dtype=np.uint8, copy=True, order="C"))
    logi = (np.zeros((B, rows, D), dtype=np.float32) if logical is None
            else np.array(_np(logical), dtype=np.float32, copy=True, order="C"))
    a = _CompressArgs()
    a.kv, a.gate, a.ape, a.norm = kvh.ctypes.data, gh.ctypes.data, ah.ctypes.data, nh.ctypes.data
    a.carry, a.records, a.logical = cy.ctypes.data, recs.ctypes.data, logi.ctypes.data
    a.B, a.S, a.D, a.n_rope, a.ratio, a.kind = B, S, D, n_rope, ratio, kind
    a.rows, a.record_stride, a.total = rows, stride, int(total)
    bad = _i64(0)
    rc = lib().orc_csa_compress(C.byref(a), C.byref(bad))
    if rc != 0:
        raise ValueError("oracle rejected the compression shape")
    return recs, logi, cy, bad.value
