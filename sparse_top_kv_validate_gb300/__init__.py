"""GB300 KV-cache attention library: Python binding of ``libsa.so``.

This module only marshals arguments: it turns torch CUDA tensors into the
device pointers and sizes of the C ABI declared in ``include/sa.h`` and
passes torch's current stream.  Every step of the computation runs in the
library's CUDA kernels; if ``libsa.so`` is missing the calls raise instead of
falling back to anything else.

Entry points (same names as the C ABI):
    validate_indices, build_present_kv, sparse_attn_decode, attn_prefill,
    paged_attn_decode, sparse_index_select, csa_ratio4_attention,
    csa_ratio128_compress, csa_ratio4_main_compress, csa_ratio4_index_compress,
    csa_pool_weight
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

__all__ = [
    "load", "lib_path", "SAError", "status_string", "check_wait_timeout", "graph_kernel_count",
    "validate_indices", "build_present_kv", "sparse_attn_decode", "attn_prefill",
    "paged_attn_decode", "sparse_attn_decode_workspace", "attn_prefill_workspace",
    "paged_attn_decode_workspace", "new_workspace", "sparse_attn_decode_noalloc",
    "NOALLOC_SCRATCH_BYTES", "ERR_SCRATCH_LIMIT", "OPT_ROW_COPIES", "OPT_FP8_WARP_MMA",
    "F32", "F16", "BF16", "FP8_E4M3_B64",
    "IDX_BELOW_SENTINEL", "IDX_AFTER_PADDING", "IDX_OUT_OF_RANGE", "IDX_NOT_INCREASING",
    "IDX_DUPLICATE", "IDX_ALL_PADDING", "ERRBIT_WRITE_POS", "ERRBIT_PAGE", "ERRBIT_TIMEOUT",
    "SparseParams", "PrefillParams", "PagedParams", "kernel_events",
    "IndexSelectParams", "sparse_index_select", "sparse_index_select_workspace",
    "SEL_TIE", "SEL_NONFINITE", "ERRBIT_SEL_TIE", "ERRBIT_SEL_NONFINITE",
    "CsaParams", "csa_ratio4_attention", "csa_ratio4_attention_workspace", "ERRBIT_RECORD",
    "CompressParams", "csa_ratio128_compress", "csa_ratio4_main_compress",
    "csa_ratio4_index_compress", "csa_pool_weight", "ERRBIT_COMPRESS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "_build", "libsa.so")

F32, F16, BF16, FP8_E4M3_B64 = 0, 1, 2, 3
IDX_BELOW_SENTINEL, IDX_AFTER_PADDING, IDX_OUT_OF_RANGE = 1, 2, 4
IDX_NOT_INCREASING, IDX_DUPLICATE, IDX_ALL_PADDING = 8, 16, 32
ERRBIT_WRITE_POS, ERRBIT_PAGE, ERRBIT_TIMEOUT = 64, 128, 256
ERR_SCRATCH_LIMIT = -9
NOALLOC_SCRATCH_BYTES = 16 << 20
OPT_ROW_COPIES, OPT_FP8_WARP_MMA = 1, 2
SEL_TIE, SEL_NONFINITE = 1, 2
ERRBIT_SEL_TIE, ERRBIT_SEL_NONFINITE = 512, 1024
ERRBIT_RECORD = 2048
ERRBIT_COMPRESS = 4096

_p = C.c_void_p
_i64 = C.c_int64
_i32 = C.c_int32


class SparseParams(C.Structure):
    _fields_ = [
        ("q", _p), ("k_cache", _p), ("v_cache", _p), ("idx", _p), ("sink", _p), ("y", _p),
        ("q_dtype", _i32), ("kv_dtype", _i32), ("idx_is_i64", _i32), ("causal", _i32),
        ("B", _i64), ("Hq", _i64), ("Hkv", _i64), ("Sq", _i64), ("D", _i64), ("Dv", _i64),
        ("T", _i64), ("I", _i64), ("K", _i64),
        ("kv_len", _p), ("past_len", _i64),
        ("scale", C.c_float), ("softcap", C.c_float),
        ("window", _i64), ("record_stride", _i64), ("n_rope", _i64),
        ("err_word", _p), ("row_status", _p),
        ("k_cur", _p), ("v_cur", _p), ("write_pos", _p), ("cur_len", _i64),
        ("workspace", _p), ("workspace_bytes", C.c_size_t),
        ("bias", _p), ("bias_rank", _i64), ("bias_dims", _i64 * 4),
        ("options", C.c_uint32), ("reserved_", C.c_uint32),
    ]


class PrefillParams(C.Structure):
    _fields_ = [
        ("q", _p), ("k", _p), ("v", _p), ("y", _p), ("present_k", _p), ("present_v", _p),
        ("dtype", _i32), ("causal", _i32),
        ("B", _i64), ("Hq", _i64), ("Hkv", _i64), ("S", _i64), ("D", _i64),
        ("scale", C.c_float), ("softcap", C.c_float),
        ("workspace", _p), ("workspace_bytes", C.c_size_t), ("err_word", _p),
        ("attn_mask", _p), ("mask_kind", _i32), ("reserved_", _i32), ("mask_rank", _i64),
        ("mask_dims", _i64 * 4), ("nonpad_kv_seqlen", _p),
    ]


class PagedParams(C.Structure):
    _fields_ = [
        ("q", _p), ("k_pool", _p), ("v_pool", _p), ("k_new", _p), ("v_new", _p),
        ("block_table", _p), ("ctx_len", _p), ("y", _p),
        ("dtype", _i32), ("options", C.c_uint32),
        ("B", _i64), ("Hq", _i64), ("Hkv", _i64), ("D", _i64), ("page_tokens", _i64),
        ("max_pages", _i64), ("num_pages", _i64),
        ("scale", C.c_float), ("pad2_", C.c_float),
        ("err_word", _p), ("workspace", _p), ("workspace_bytes", C.c_size_t),
    ]


class IndexSelectParams(C.Structure):
    _fields_ = [
        ("query", _p), ("weight", _p), ("keys", _p), ("selected", _p), ("row_status", _p),
        ("err_word", _p),
        ("B", _i64), ("S", _i64), ("IH", _i64), ("ID", _i64), ("R", _i64), ("topk", _i64),
        ("key_stride", _i64), ("out_heads", _i64), ("query_start", _i64),
        ("query_start_b", _p), ("ascending", _i32), ("reserved_", _i32),
        ("workspace", _p), ("workspace_bytes", C.c_size_t),
    ]


class CsaParams(C.Structure):
    _fields_ = [
        ("query", _p), ("current_kv", _p), ("records", _p), ("selected", _p), ("sink", _p),
        ("bias", _p), ("bias_rank", _i64), ("bias_dims", _i64 * 4), ("y", _p),
        ("q_dtype", _i32), ("kv_dtype", _i32),
        ("B", _i64), ("S", _i64), ("H", _i64), ("D", _i64), ("n_rope", _i64), ("L", _i64),
        ("R", _i64), ("topk", _i64), ("record_stride", _i64), ("total", _i64),
        ("scale", C.c_float), ("reserved_", _i32), ("err_word", _p),
        ("workspace", _p), ("workspace_bytes", C.c_size_t),
    ]


class CompressParams(C.Structure):
    _fields_ = [
        ("kv", _p), ("gate", _p), ("ape", _p), ("norm", _p), ("carry", _p), ("records", _p),
        ("logical", _p), ("err_word", _p),
        ("B", _i64), ("S", _i64), ("D", _i64), ("n_rope", _i64), ("rows", _i64),
        ("record_stride", _i64), ("total", _i64), ("reserved_", _i64),
    ]


class SAError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call}: status {status} ({status_string(status)})")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def load():
    """Load ``libsa.so`` (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB):
            raise RuntimeError(
                f"{_LIB} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = C.CDLL(_LIB)
        L.sa_status_string.restype = C.c_char_p
        L.sa_status_string.argtypes = [C.c_int]
        L.sa_version.restype = C.c_int
        L.sa_version.argtypes = []
        L.sa_set_kernel_events.restype = C.c_int
        L.sa_set_kernel_events.argtypes = [_p, _p]
        L.validate_indices.restype = C.c_int
        L.validate_indices.argtypes = [_p, C.c_int, _i64, _i64, _i64, _i64, _p, _i64, _p, _p, _p]
        L.build_present_kv.restype = C.c_int
        L.build_present_kv.argtypes = [_p, _p, _p, _p, _p, _p, C.c_int, _i64, _i64, _i64, _i64,
                                       _i64, _i64, _p, _p, _p]
        L.sparse_attn_decode_workspace.restype = C.c_size_t
        L.sparse_attn_decode_workspace.argtypes = [C.POINTER(SparseParams)]
        L.sparse_attn_decode.restype = C.c_int
        L.sparse_attn_decode.argtypes = [C.POINTER(SparseParams), _p]
        L.sparse_attn_decode_noalloc.restype = C.c_int
        L.sparse_attn_decode_noalloc.argtypes = [C.POINTER(SparseParams), _p]
        L.attn_prefill_workspace.restype = C.c_size_t
        L.attn_prefill_workspace.argtypes = [C.POINTER(PrefillParams)]
        L.attn_prefill.restype = C.c_int
        L.attn_prefill.argtypes = [C.POINTER(PrefillParams), _p]
        L.sparse_index_select_workspace.restype = C.c_size_t
        L.sparse_index_select_workspace.argtypes = [C.POINTER(IndexSelectParams)]
        L.sparse_index_select.restype = C.c_int
        L.sparse_index_select.argtypes = [C.POINTER(IndexSelectParams), _p]
        L.csa_ratio4_attention_workspace.restype = C.c_size_t
        L.csa_ratio4_attention_workspace.argtypes = [C.POINTER(CsaParams)]
        L.csa_ratio4_attention.restype = C.c_int
        L.csa_ratio4_attention.argtypes = [C.POINTER(CsaParams), _p]
        for name in ("csa_ratio128_compress", "csa_ratio4_main_compress",
                     "csa_ratio4_index_compress"):
            fn = getattr(L, name)
            fn.restype = C.c_int
            fn.argtypes = [C.POINTER(CompressParams), _p]
        L.csa_pool_weight.restype = C.c_int
        L.csa_pool_weight.argtypes = [_p, _p, _i64, _p]
        L.sa_check_wait_timeout.restype = C.c_int
        L.sa_check_wait_timeout.argtypes = [_p, _p, _p]
        L.sa_graph_kernel_count.restype = C.c_int
        L.sa_graph_kernel_count.argtypes = [_p]
        L.paged_attn_decode_workspace.restype = C.c_size_t
        L.paged_attn_decode_workspace.argtypes = [C.POINTER(PagedParams)]
        L.paged_attn_decode.restype = C.c_int
        L.paged_attn_decode.argtypes = [C.POINTER(PagedParams), _p]
        _lib = L
        return _lib


class kernel_events:
    """Measurement hook: within the ``with`` block, every call of this library
    from this host thread records ``before`` / ``after`` (timing
    ``torch.cuda.Event`` objects, recorded once here so that they exist) on its
    stream around its dominant kernel; ``before.elapsed_time(after)`` is then
    that kernel's duration for the last call."""

    def __init__(self, before, after):
        self.before, self.after = before, after

    def __enter__(self):
        for ev in (self.before, self.after):
            if not ev.cuda_event:
                ev.record()
        torch.cuda.synchronize()
        _check("sa_set_kernel_events",
               load().sa_set_kernel_events(C.c_void_p(self.before.cuda_event),
                                           C.c_void_p(self.after.cuda_event)))
        return self

    def __exit__(self, *exc):
        load().sa_set_kernel_events(None, None)
        return False


def status_string(status: int) -> str:
    return load().sa_status_string(int(status)).decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

_DT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _dev(t, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(call, rc):
    if rc != 0:
        raise SAError(call, rc)


_ws_cache: dict = {}


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned workspace of at least ``nbytes`` (contents irrelevant)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _workspace(nbytes: int, device, workspace=None):
    """Caller-owned scratch: the given tensor, or a cached torch allocation
    per (device, stream)."""
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = new_workspace(max(nbytes, 1 << 20), device)
        _ws_cache[key] = buf
    return buf, buf.numel()


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def validate_indices(idx: torch.Tensor, bound: int = 0, bound_per_batch=None, *,
                     row_status: torch.Tensor | None = None,
                     err_word: torch.Tensor | None = None, stream=None):
    """Validate ``idx`` ``[B, I, Sq, K]`` (int32/int64) on the device.

    Returns ``(row_status uint8 [B*I*Sq], err_word uint32 [1])`` device tensors;
    ``err_word`` is zeroed here unless passed in."""
    L = load()
    _dev(idx, "idx")
    B, I, Sq, K = idx.shape
    if row_status is None:
        row_status = torch.empty(B * I * Sq, dtype=torch.uint8, device=idx.device)
    if err_word is None:
        err_word = torch.zeros(1, dtype=torch.int32, device=idx.device)
    bb = _dev(bound_per_batch, "bound_per_batch")
    rc = L.validate_indices(idx.data_ptr(), int(idx.dtype == torch.int64), B, I, Sq, K, _ptr(bb),
                            int(bound), _ptr(row_status), err_word.data_ptr(), _stream(stream))
    _check("validate_indices", rc)
    return row_status, err_word


def build_present_kv(cur_k, present_k, past_k=None, cur_v=None, present_v=None, past_v=None, *,
                     write_pos=None, err_word=None, stream=None):
    """Present K/V: concat (``write_pos`` None: present = past ++ cur along the
    sequence axis, present ``[B,H,stride,D]``) or append (cur written at
    ``write_pos[b]`` of the capacity cache ``present``)."""
    L = load()
    for n, t in (("cur_k", cur_k), ("present_k", present_k), ("past_k", past_k), ("cur_v", cur_v),
                 ("present_v", present_v), ("past_v", past_v), ("write_pos", write_pos),
                 ("err_word", err_word)):
        _dev(t, n)
    B, H, Cn, D = cur_k.shape
    P = 0 if (past_k is None or write_pos is not None) else past_k.shape[2]
    rc = L.build_present_kv(_ptr(past_k), cur_k.data_ptr(), present_k.data_ptr(), _ptr(past_v),
                            _ptr(cur_v), _ptr(present_v), _dt(cur_k), B, H, P, Cn, D,
                            present_k.shape[2], _ptr(write_pos), _ptr(err_word), _stream(stream))
    _check("build_present_kv", rc)
    return present_k, present_v


def _sparse_params(q, k_cache, v_cache, idx, y, *, scale, softcap, window, kv_len, past_len,
                   causal, sink, err_word, row_status, n_rope=0, Dv=None, k_cur=None,
                   v_cur=None, write_pos=None, bias=None, options=0):
    p = SparseParams()
    B, Hq, Sq, D = q.shape
    p.q, p.y = q.data_ptr(), _ptr(y)
    p.q_dtype = _dt(q)
    if k_cache.dtype == torch.uint8:
        p.k_cache = k_cache.data_ptr()
        p.v_cache = None
        p.kv_dtype = FP8_E4M3_B64
        p.record_stride = k_cache.shape[3]
        p.n_rope = n_rope
        p.Dv = D if Dv is None else Dv
    else:
        p.k_cache, p.v_cache = k_cache.data_ptr(), _ptr(v_cache)
        p.kv_dtype = _dt(k_cache)
        p.Dv = v_cache.shape[3]
    p.Hkv, p.T = k_cache.shape[1], k_cache.shape[2]
    if idx is not None:
        p.idx = idx.data_ptr()
        p.idx_is_i64 = int(idx.dtype == torch.int64)
        p.I, p.K = idx.shape[1], idx.shape[3]
    else:
        p.idx, p.I, p.K = None, 1, 0
    p.B, p.Hq, p.Sq, p.D = B, Hq, Sq, D
    p.sink = _ptr(sink)
    p.kv_len = _ptr(kv_len)
    p.past_len = int(past_len)
    p.causal = int(bool(causal))
    p.scale = float(scale)
    p.softcap = float(softcap)
    p.window = int(window)
    p.err_word = _ptr(err_word)
    p.row_status = _ptr(row_status)
    p.k_cur, p.v_cur, p.write_pos = _ptr(k_cur), _ptr(v_cur), _ptr(write_pos)
    p.cur_len = 0 if k_cur is None else k_cur.shape[2]
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() > 4:
            raise ValueError("bias must be float32 of rank <= 4")
        p.bias, p.bias_rank = bias.data_ptr(), bias.dim()
        for r, e in enumerate(bias.shape):
            p.bias_dims[r] = e
    p.options = int(options)
    return p


def sparse_attn_decode_workspace(q, k_cache, v_cache, idx, **kw) -> int:
    p = _sparse_params(q, k_cache, v_cache, idx, None, **_sparse_defaults(kw))
    return int(load().sparse_attn_decode_workspace(C.byref(p)))


def _sparse_defaults(kw):
    d = dict(scale=0.0, softcap=0.0, window=0, kv_len=None, past_len=0, causal=False, sink=None,
             err_word=None, row_status=None, n_rope=0, Dv=None, k_cur=None, v_cur=None,
             write_pos=None, bias=None, options=0)
    d.update(kw)
    return d


def sparse_attn_decode(q, k_cache, v_cache, idx, *, y=None, workspace=None, stream=None, **kw):
    """Selected-token attention.  ``q [B,Hq,Sq,D]``; dense cache
    ``k_cache/v_cache [B,Hkv,T,D]`` (same dtype as q) or FP8 hybrid records
    ``k_cache uint8 [B,Hkv,T,record_stride]`` (``v_cache`` None, pass
    ``n_rope``); ``idx [B,I,Sq,K]`` int32/int64.  Keyword options: scale,
    softcap, window, kv_len (int64 [B]), past_len, causal, sink (float32
    [Hq]), err_word (int32 [1], caller-zeroed), row_status (uint8 [B*I*Sq]),
    n_rope, Dv, the fused append k_cur / v_cur ([B,Hkv,C,D]) with
    write_pos (int64 [B], default T - C), bias (float32, rank <= 4,
    broadcast against [B,Hq,Sq,T]: added to the score of cache position j)
    and options (OPT_* bits).  Returns ``y [B,Hq,Sq,Dv]``."""
    L = load()
    kw = _sparse_defaults(kw)
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("idx", idx),
                 ("kv_len", kw["kv_len"]), ("sink", kw["sink"]), ("err_word", kw["err_word"]),
                 ("row_status", kw["row_status"]), ("k_cur", kw["k_cur"]), ("v_cur", kw["v_cur"]),
                 ("write_pos", kw["write_pos"]), ("bias", kw["bias"])):
        _dev(t, n)
    B, Hq, Sq, D = q.shape
    Dv = kw["Dv"] if k_cache.dtype == torch.uint8 else v_cache.shape[3]
    if Dv is None:
        Dv = D
    if y is None:
        y = torch.empty((B, Hq, Sq, Dv), dtype=q.dtype, device=q.device)
    p = _sparse_params(q, k_cache, v_cache, idx, y, **kw)
    need = int(L.sparse_attn_decode_workspace(C.byref(p)))
    ws, nb = _workspace(need, q.device, workspace)
    p.workspace, p.workspace_bytes = _ptr(ws), nb
    _check("sparse_attn_decode", L.sparse_attn_decode(C.byref(p), _stream(stream)))
    return y


_MASK_KIND = {torch.float32: 1, torch.float16: 2, torch.bfloat16: 3, torch.bool: 4,
              torch.uint8: 4}


def _prefill_params(q, k, v, y, present_k, present_v, causal, scale, softcap, err_word=None,
                    attn_mask=None, nonpad_kv_seqlen=None):
    p = PrefillParams()
    B, Hq, S, D = q.shape
    p.q, p.k, p.v, p.y = q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(y)
    p.present_k, p.present_v = _ptr(present_k), _ptr(present_v)
    p.dtype, p.causal = _dt(q), int(bool(causal))
    p.B, p.Hq, p.Hkv, p.S, p.D = B, Hq, k.shape[1], S, D
    p.scale, p.softcap = float(scale), float(softcap)
    p.err_word = _ptr(err_word)
    if attn_mask is not None:
        if attn_mask.dtype not in _MASK_KIND or attn_mask.dim() > 4:
            raise ValueError("attn_mask: float32/float16/bfloat16/bool of rank <= 4")
        p.attn_mask, p.mask_kind = attn_mask.data_ptr(), _MASK_KIND[attn_mask.dtype]
        p.mask_rank = attn_mask.dim()
        for r, e in enumerate(attn_mask.shape):
            p.mask_dims[r] = e
    p.nonpad_kv_seqlen = _ptr(nonpad_kv_seqlen)
    return p


def attn_prefill_workspace(q, k, v, causal=True, scale=0.0, softcap=0.0, attn_mask=None,
                           nonpad_kv_seqlen=None) -> int:
    p = _prefill_params(q, k, v, None, None, None, causal, scale, softcap, None, attn_mask,
                        nonpad_kv_seqlen)
    return int(load().attn_prefill_workspace(C.byref(p)))


def attn_prefill(q, k, v, *, causal=True, scale=0.0, softcap=0.0, y=None, present_k=None,
                 present_v=None, err_word=None, workspace=None, stream=None, attn_mask=None,
                 nonpad_kv_seqlen=None):
    """Dense prefill, ``q [B,Hq,S,D]``, ``k/v [B,Hkv,S,D]``; optional exact
    present K/V copies, ``attn_mask`` (float32/float16/bfloat16/bool, rank <=
    4, broadcast against ``[B,Hq,S,S]``) and ``nonpad_kv_seqlen`` (int64
    ``[B]``).  Returns ``y``."""
    L = load()
    for n, t in (("q", q), ("k", k), ("v", v), ("present_k", present_k),
                 ("present_v", present_v), ("attn_mask", attn_mask),
                 ("nonpad_kv_seqlen", nonpad_kv_seqlen)):
        _dev(t, n)
    if y is None:
        y = torch.empty_like(q)
    p = _prefill_params(q, k, v, y, present_k, present_v, causal, scale, softcap, err_word,
                        attn_mask, nonpad_kv_seqlen)
    need = int(L.attn_prefill_workspace(C.byref(p)))
    ws, nb = _workspace(need, q.device, workspace)
    p.workspace, p.workspace_bytes = _ptr(ws), nb
    _check("attn_prefill", L.attn_prefill(C.byref(p), _stream(stream)))
    return y


def _paged_params(q, k_pool, v_pool, block_table, ctx_len, y, k_new, v_new, scale, err_word,
                  options=0):
    p = PagedParams()
    B, Hq = q.shape[0], q.shape[1]
    D = q.shape[-1]
    p.q, p.k_pool, p.v_pool = q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr()
    p.k_new, p.v_new = _ptr(k_new), _ptr(v_new)
    p.block_table, p.ctx_len, p.y = block_table.data_ptr(), ctx_len.data_ptr(), _ptr(y)
    p.dtype = _dt(q)
    p.B, p.Hq, p.Hkv, p.D = B, Hq, k_pool.shape[1], D
    p.page_tokens, p.max_pages, p.num_pages = k_pool.shape[2], block_table.shape[1], k_pool.shape[0]
    p.scale = float(scale)
    p.err_word = _ptr(err_word)
    p.options = int(options)
    return p


def paged_attn_decode_workspace(q, k_pool, v_pool, block_table, ctx_len, scale=0.0) -> int:
    p = _paged_params(q, k_pool, v_pool, block_table, ctx_len, None, None, None, scale, None)
    return int(load().paged_attn_decode_workspace(C.byref(p)))


def paged_attn_decode(q, k_pool, v_pool, block_table, ctx_len, *, k_new=None, v_new=None,
                      scale=0.0, err_word=None, y=None, workspace=None, stream=None,
                      options=0):
    """Paged causal decode: ``q [B,Hq,1,D]`` (or ``[B,Hq,D]``), pools
    ``[num_pages,Hkv,page_tokens,D]``, ``block_table int32 [B,max_pages]``,
    ``ctx_len int32 [B]``; optional ``k_new/v_new [B,Hkv,D]`` written at token
    ``ctx_len-1`` first.  Returns ``y`` shaped like ``q``."""
    L = load()
    for n, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("block_table", block_table),
                 ("ctx_len", ctx_len), ("k_new", k_new), ("v_new", v_new),
                 ("err_word", err_word)):
        _dev(t, n)
    if block_table.dtype != torch.int32 or ctx_len.dtype != torch.int32:
        raise TypeError("block_table and ctx_len must be int32")
    if y is None:
        y = torch.empty_like(q)
    p = _paged_params(q, k_pool, v_pool, block_table, ctx_len, y, k_new, v_new, scale, err_word,
                      options)
    need = int(L.paged_attn_decode_workspace(C.byref(p)))
    ws, nb = _workspace(need, q.device, workspace)
    p.workspace, p.workspace_bytes = _ptr(ws), nb
    _check("paged_attn_decode", L.paged_attn_decode(C.byref(p), _stream(stream)))
    return y


def sparse_attn_decode_noalloc(q, k_cache, v_cache, idx, *, y=None, stream=None, **kw):
    """``sparse_attn_decode`` without caller-provided scratch: the library's
    built-in device buffer (``NOALLOC_SCRATCH_BYTES``) serves every call, so
    calls must not overlap on the GPU.  Same arguments, minus ``workspace``."""
    L = load()
    kw = _sparse_defaults(kw)
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("idx", idx),
                 ("kv_len", kw["kv_len"]), ("sink", kw["sink"]), ("err_word", kw["err_word"]),
                 ("row_status", kw["row_status"]), ("k_cur", kw["k_cur"]), ("v_cur", kw["v_cur"]),
                 ("write_pos", kw["write_pos"]), ("bias", kw["bias"])):
        _dev(t, n)
    B, Hq, Sq, D = q.shape
    Dv = kw["Dv"] if k_cache.dtype == torch.uint8 else v_cache.shape[3]
    if Dv is None:
        Dv = D
    if y is None:
        y = torch.empty((B, Hq, Sq, Dv), dtype=q.dtype, device=q.device)
    p = _sparse_params(q, k_cache, v_cache, idx, y, **kw)
    _check("sparse_attn_decode_noalloc", L.sparse_attn_decode_noalloc(C.byref(p), _stream(stream)))
    return y


def _index_params(query, weight, keys, selected, *, topk, query_start, query_start_b,
                  out_heads, ascending, row_status, err_word):
    p = IndexSelectParams()
    B, S, IH, ID = query.shape
    p.query, p.weight, p.keys = query.data_ptr(), weight.data_ptr(), keys.data_ptr()
    p.selected = _ptr(selected)
    p.row_status, p.err_word = _ptr(row_status), _ptr(err_word)
    p.B, p.S, p.IH, p.ID = B, S, IH, ID
    p.R, p.key_stride = keys.shape[1], keys.shape[2]
    p.topk, p.out_heads = int(topk), int(out_heads)
    p.query_start = int(query_start)
    p.query_start_b = _ptr(query_start_b)
    p.ascending = int(bool(ascending))
    return p


def sparse_index_select_workspace(query, weight, keys, *, topk, out_heads=1) -> int:
    p = _index_params(query, weight, keys, None, topk=topk, query_start=0, query_start_b=None,
                      out_heads=out_heads, ascending=False, row_status=None, err_word=None)
    return int(load().sparse_index_select_workspace(C.byref(p)))


def sparse_index_select(query, weight, keys, *, topk, query_start=0, query_start_b=None,
                        out_heads=1, ascending=False, row_status=None, err_word=None,
                        selected=None, workspace=None, stream=None):
    """Ratio-4 index scoring and top-k selection.  ``query`` float32
    ``[B, S, IH, ID]``, ``weight`` float32 ``[B, S, IH]``, ``keys`` uint8
    ``[B, R, key_stride]`` FP4 records; query s of batch b sits at position
    ``query_start + s`` (or ``query_start_b[b] + s``, int64 ``[B]``).
    Returns ``selected`` int32 ``[B, out_heads, S, topk]`` (score order, or
    ascending records with ``ascending``), -1 past the causal records;
    ``row_status`` (uint8 ``[B*S]``) / ``err_word`` receive the tie and
    non-finite flags."""
    L = load()
    for n, t in (("query", query), ("weight", weight), ("keys", keys),
                 ("query_start_b", query_start_b), ("row_status", row_status),
                 ("err_word", err_word), ("selected", selected)):
        _dev(t, n)
    if query.dtype != torch.float32 or weight.dtype != torch.float32 or keys.dtype != torch.uint8:
        raise TypeError("query and weight must be float32, keys uint8")
    B, S = query.shape[0], query.shape[1]
    if selected is None:
        selected = torch.empty((B, out_heads, S, topk), dtype=torch.int32, device=query.device)
    p = _index_params(query, weight, keys, selected, topk=topk, query_start=query_start,
                      query_start_b=query_start_b, out_heads=out_heads, ascending=ascending,
                      row_status=row_status, err_word=err_word)
    need = int(L.sparse_index_select_workspace(C.byref(p)))
    ws, nb = _workspace(need, query.device, workspace)
    p.workspace, p.workspace_bytes = _ptr(ws), nb
    _check("sparse_index_select", L.sparse_index_select(C.byref(p), _stream(stream)))
    return selected


def _csa_params(query, current_kv, records, selected, y, *, total, n_rope, scale, sink, bias,
                err_word):
    p = CsaParams()
    B, S, H, D = query.shape
    p.query, p.current_kv = query.data_ptr(), _ptr(current_kv)
    p.records, p.selected, p.y = records.data_ptr(), selected.data_ptr(), _ptr(y)
    p.sink, p.err_word = _ptr(sink), _ptr(err_word)
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() > 4:
            raise ValueError("bias must be float32 of rank <= 4")
        p.bias, p.bias_rank = bias.data_ptr(), bias.dim()
        for r, e in enumerate(bias.shape):
            p.bias_dims[r] = e
    p.q_dtype = _dt(query)
    p.kv_dtype = _dt(current_kv) if current_kv is not None else _dt(query)
    p.B, p.S, p.H, p.D = B, S, H, D
    p.n_rope = int(n_rope)
    p.L = current_kv.shape[1] if current_kv is not None else 0
    p.R, p.record_stride = records.shape[1], records.shape[2]
    p.topk, p.total, p.scale = selected.shape[2], int(total), float(scale)
    return p


def csa_ratio4_attention_workspace(query, current_kv, records, selected, *, total, n_rope,
                                   scale=0.0, sink=None, bias=None) -> int:
    p = _csa_params(query, current_kv, records, selected, None, total=total, n_rope=n_rope,
                    scale=scale, sink=sink, bias=bias, err_word=None)
    return int(load().csa_ratio4_attention_workspace(C.byref(p)))


def csa_ratio4_attention(query, current_kv, records, selected, *, total, n_rope, scale=0.0,
                         sink=None, bias=None, err_word=None, y=None, workspace=None,
                         stream=None):
    """Compressed sparse attention, ratio 4, in the pages' own form.  ``query``
    ``[B, S, H, D]`` (float32 / bfloat16), ``current_kv`` ``[B, L, D]``,
    ``records`` uint8 ``[B, R, record_stride]`` hybrid FP8, ``selected`` int32
    ``[B, S, topk]``; ``total`` tokens so far; optional ``sink`` float32 ``[H]``
    and ``bias`` float32 (rank <= 4, against ``[B, H, S, candidates]``).
    Returns ``y`` shaped and typed like ``query``."""
    L = load()
    for n, t in (("query", query), ("current_kv", current_kv), ("records", records),
                 ("selected", selected), ("sink", sink), ("bias", bias), ("err_word", err_word)):
        _dev(t, n)
    if selected.dtype != torch.int32 or records.dtype != torch.uint8:
        raise TypeError("selected must be int32 and records uint8")
    if y is None:
        y = torch.empty_like(query)
    p = _csa_params(query, current_kv, records, selected, y, total=total, n_rope=n_rope,
                    scale=scale, sink=sink, bias=bias, err_word=err_word)
    need = int(L.csa_ratio4_attention_workspace(C.byref(p)))
    ws, nb = _workspace(need, query.device, workspace)
    p.workspace, p.workspace_bytes = _ptr(ws), nb
    _check("csa_ratio4_attention", L.csa_ratio4_attention(C.byref(p), _stream(stream)))
    return y


# ---- CSA compression stages ---------------------------------------------------------------

def _compress(name, ratio, D, kv, gate, ape, norm, carry, *, n_rope, total, records, logical,
              err_word, stream):
    L = load()
    for n, t in (("kv", kv), ("gate", gate), ("ape", ape), ("norm", norm), ("carry", carry),
                 ("records", records), ("logical", logical), ("err_word", err_word)):
        _dev(t, n)
    for n, t in (("kv", kv), ("gate", gate), ("ape", ape), ("norm", norm), ("carry", carry),
                 ("logical", logical)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise TypeError(f"{n} must be a contiguous float32 tensor")
    if records is not None and (records.dtype != torch.uint8 or not records.is_contiguous()):
        raise TypeError("records must be a contiguous uint8 tensor")
    B, S = kv.shape[0], kv.shape[1]
    p = CompressParams()
    p.kv, p.gate, p.ape, p.norm = kv.data_ptr(), gate.data_ptr(), ape.data_ptr(), norm.data_ptr()
    p.carry, p.records, p.logical = carry.data_ptr(), _ptr(records), _ptr(logical)
    p.err_word = _ptr(err_word)
    p.B, p.S, p.D, p.n_rope, p.total = B, S, D, int(n_rope), int(total)
    if records is not None:
        p.rows, p.record_stride = records.shape[1], records.shape[2]
    else:
        p.rows, p.record_stride = logical.shape[1], 0
    _check(name, getattr(L, name)(C.byref(p), _stream(stream)))


def csa_ratio128_compress(kv, gate, ape, norm, carry, *, n_rope, total, records=None,
                          logical=None, err_word=None, stream=None):
    """Append ``S`` tokens to a ratio-128 compression stream.  ``kv``, ``gate``
    float32 ``[B, S, D]``, ``ape`` ``[128, D]``, ``norm`` ``[D]``, ``carry``
    ``[B, 128, 2, D]`` (updated in place); every block of 128 tokens that
    closes is written to ``records`` (uint8 ``[B, rows, stride]``, hybrid
    FP8) and/or ``logical`` (float32 ``[B, rows, D]``) at row ``p // 128``."""
    _compress("csa_ratio128_compress", 128, kv.shape[2], kv, gate, ape, norm, carry,
              n_rope=n_rope, total=total, records=records, logical=logical,
              err_word=err_word, stream=stream)


def csa_ratio4_main_compress(kv, gate, ape, norm, carry, *, n_rope, total, records=None,
                             logical=None, err_word=None, stream=None):
    """Append ``S`` tokens to a ratio-4 attention-record stream.  ``kv``,
    ``gate`` float32 ``[B, S, 2D]``, ``ape`` ``[4, 2D]``, ``norm`` ``[D]``,
    ``carry`` ``[B, 8, 2, 2D]`` (updated in place); records as for ratio 128,
    at row ``p // 4``."""
    _compress("csa_ratio4_main_compress", 4, kv.shape[2] // 2, kv, gate, ape, norm, carry,
              n_rope=n_rope, total=total, records=records, logical=logical,
              err_word=err_word, stream=stream)


def csa_ratio4_index_compress(kv, gate, ape, norm, carry, *, n_rope, total, records=None,
                              logical=None, err_word=None, stream=None):
    """Append ``S`` tokens to a ratio-4 index-key stream (FP4 keys of
    ``D / 32 * 17`` bytes, Hadamard-transformed); shapes as for
    ``csa_ratio4_main_compress``."""
    _compress("csa_ratio4_index_compress", 4, kv.shape[2] // 2, kv, gate, ape, norm, carry,
              n_rope=n_rope, total=total, records=records, logical=logical,
              err_word=err_word, stream=stream)


def graph_kernel_count(graph) -> int:
    """Kernel nodes in a captured ``torch.cuda.CUDAGraph`` (measurement hook:
    how many kernels one captured call launches)."""
    n = load().sa_graph_kernel_count(C.c_void_p(graph.raw_cuda_graph()))
    _check("sa_graph_kernel_count", min(n, 0))
    return n


def check_wait_timeout(device="cuda", stream=None):
    """Runs the library's bounded-wait timeout path once (one warp waits on a
    barrier nothing arrives on, about a second); returns ``(err_word, out)``,
    int32 CUDA tensors of 1 and 4 entries (see ``sa_check_wait_timeout``)."""
    err = torch.zeros(1, dtype=torch.int32, device=device)
    out = torch.zeros(4, dtype=torch.int32, device=device)
    _check("sa_check_wait_timeout",
           load().sa_check_wait_timeout(err.data_ptr(), out.data_ptr(), _stream(stream)))
    return err, out


def csa_pool_weight(t, *, w=None, stream=None):
    """``e^t`` rounded to binary32 as the compression pool computes it;
    ``t`` a contiguous float32 CUDA tensor."""
    _dev(t, "t")
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError("t must be a contiguous float32 tensor")
    if w is None:
        w = torch.empty_like(t)
    _check("csa_pool_weight", load().csa_pool_weight(t.data_ptr(), w.data_ptr(), t.numel(),
                                                      _stream(stream)))
    return w
