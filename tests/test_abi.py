"""CPU-only checks of the C ABI: the library loads, exports every function
that include/sa.h declares, the Python structs match the C layout, and the
host-side argument checks reject bad requests before anything is launched."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

import sparse_top_kv_validate_gb300 as sa
from sparse_top_kv_validate_gb300 import build as sa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sa.h")


@pytest.fixture(scope="module")
def lib():
    sa_build.build()
    return sa.load()


@pytest.fixture(scope="module")
def host_lib(lib):
    """The library, for calls on fake device addresses that the host checks
    must refuse.  Skipped where a GPU is present: a request that passed the
    checks by mistake must never reach a real device."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake-address checks run on hosts without a GPU")
    return lib


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_seven_operations():
    names = declared_functions()
    for n in ("validate_indices", "build_present_kv", "sparse_attn_decode", "attn_prefill",
              "paged_attn_decode"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sa.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def _c_layout(struct_name, fields):
    src = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"', "int main(void){",
           f'printf("%zu\\n", sizeof({struct_name}));']
    for f in fields:
        src.append(f'printf("%zu\\n", offsetof({struct_name}, {f}));')
    src.append("return 0;}")
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        with open(c, "w") as f:
            f.write("\n".join(src))
        subprocess.run(["gcc", "-o", exe, c], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                               check=True).stdout.split()]
    return vals[0], vals[1:]


@pytest.mark.parametrize("cname,py", [("sa_sparse_params", sa.SparseParams),
                                      ("sa_prefill_params", sa.PrefillParams),
                                      ("sa_paged_params", sa.PagedParams),
                                      ("sa_index_select_params", sa.IndexSelectParams),
                                      ("sa_csa_params", sa.CsaParams),
                                      ("sa_compress_params", sa.CompressParams)])
def test_struct_layout_matches_header(cname, py):
    fields = [f for f, _ in py._fields_]
    size, offs = _c_layout(cname, fields)
    assert C.sizeof(py) == size
    assert [getattr(py, f).offset for f in fields] == offs


def test_status_strings(lib):
    assert sa.status_string(0) == "ok"
    assert "NULL" in sa.status_string(-1)
    assert lib.sa_version() >= 100


def test_kernel_event_hook_needs_both_events_or_none(lib):
    assert lib.sa_set_kernel_events(C.c_void_p(0x1000), None) == -1
    assert lib.sa_set_kernel_events(None, C.c_void_p(0x1000)) == -1
    assert lib.sa_set_kernel_events(None, None) == 0


def test_host_checks_reject_bad_requests_without_launching(host_lib):
    # validate_indices: null pointers, bad shapes
    assert host_lib.validate_indices(None, 0, 1, 1, 1, 4, None, 10, None, None, None) == -1
    fake = C.c_void_p(0x1000)
    word = C.c_void_p(0x2000)
    assert host_lib.validate_indices(fake, 0, 0, 1, 1, 4, None, 10, None, word, None) == -2
    assert host_lib.validate_indices(C.c_void_p(0x1002), 0, 1, 1, 1, 4, None, 10, None, word,
                                     None) == -4
    # sparse decode
    p = sa.SparseParams()
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -1
    p.q, p.k_cache, p.v_cache, p.y, p.idx = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    p.B, p.Hq, p.Hkv, p.Sq, p.D, p.Dv, p.T, p.I, p.K = 1, 6, 4, 1, 64, 64, 32, 4, 8
    p.q_dtype = p.kv_dtype = sa.BF16
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -2   # Hq % Hkv
    p.Hkv = 2
    p.I = 3
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -2   # I not in {1, Hkv, Hq}
    p.I = 2
    p.kv_dtype = sa.F16
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -3   # q/kv dtype mismatch
    p.kv_dtype = sa.BF16
    p.y = 0x10000 + 64                                       # y overlaps q
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -6
    p.y = 0x40000
    p.K, p.window = 0, 0
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -2   # no candidates at all
    # present: concat output overlapping an input
    assert host_lib.build_present_kv(None, C.c_void_p(0x1000), C.c_void_p(0x1000), None, None,
                                     None, sa.BF16, 1, 1, 0, 4, 8, 4, None, None, None) == -6
    assert host_lib.build_present_kv(None, C.c_void_p(0x1000), C.c_void_p(0x9000), None, None,
                                     None, 7, 1, 1, 0, 4, 8, 4, None, None, None) == -3
    # prefill / paged
    q = sa.PrefillParams()
    assert host_lib.attn_prefill(C.byref(q), None) == -1
    g = sa.PagedParams()
    assert host_lib.paged_attn_decode(C.byref(g), None) == -1


def test_empty_sizes_are_shape_errors_without_launching(host_lib):
    # An empty batch, sequence, head or index width is SA_ERR_SHAPE, returned by
    # the host checks (the pointers below are never dereferenced).
    fake, word = C.c_void_p(0x1000), C.c_void_p(0x2000)
    assert host_lib.validate_indices(fake, 0, 1, 1, 1, 0, None, 10, None, word, None) == -2
    assert host_lib.build_present_kv(None, fake, C.c_void_p(0x9000), None, None, None,
                                     sa.BF16, 0, 1, 0, 4, 8, 4, None, None, None) == -2
    for field in ("B", "Hq", "Sq", "D", "T"):
        p = sa.SparseParams()
        p.q, p.k_cache, p.v_cache, p.y, p.idx = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
        p.B, p.Hq, p.Hkv, p.Sq, p.D, p.Dv, p.T, p.I, p.K = 1, 4, 2, 1, 64, 64, 32, 2, 8
        p.q_dtype = p.kv_dtype = sa.BF16
        setattr(p, field, 0)
        assert host_lib.sparse_attn_decode(C.byref(p), None) == -2, field
        assert host_lib.sparse_attn_decode_workspace(C.byref(p)) == 0, field
    for field in ("B", "S", "Hq"):
        q = sa.PrefillParams()
        q.q, q.k, q.v, q.y = 0x10000, 0x20000, 0x30000, 0x40000
        q.dtype = sa.BF16
        q.B, q.Hq, q.Hkv, q.S, q.D = 1, 4, 2, 16, 64
        setattr(q, field, 0)
        assert host_lib.attn_prefill(C.byref(q), None) == -2, field
    for field in ("B", "max_pages", "page_tokens"):
        g = sa.PagedParams()
        g.q, g.k_pool, g.v_pool, g.y = 0x10000, 0x20000, 0x30000, 0x40000
        g.block_table, g.ctx_len = 0x50000, 0x60000
        g.dtype = sa.F16
        g.B, g.Hq, g.Hkv, g.D, g.page_tokens, g.max_pages, g.num_pages = 1, 4, 2, 64, 16, 2, 4
        setattr(g, field, 0)
        assert host_lib.paged_attn_decode(C.byref(g), None) == -2, field


def _fp8_params():
    # A well-formed FP8 request on fake, non-overlapping, aligned addresses; the
    # tests below only ever call the library after breaking one field of it,
    # so every call is refused by the host checks and nothing is launched.
    p = sa.SparseParams()
    p.q, p.k_cache, p.v_cache, p.y, p.idx = 0x100000, 0x10000000, None, 0x200000, 0x300000
    p.B, p.Hq, p.Hkv, p.Sq, p.D, p.Dv, p.T, p.I, p.K = 2, 128, 1, 1, 576, 576, 1000, 1, 64
    p.q_dtype, p.kv_dtype = sa.BF16, sa.FP8_E4M3_B64
    p.record_stride, p.n_rope, p.window = 648, 64, 128
    return p


@pytest.mark.parametrize("field,value,status", [
    ("q_dtype", sa.F16, -3),            # FP8 records take bf16 queries
    ("D", 512, -7), ("n_rope", 32, -7),  # 512 E4M3 + 64 bf16 dims only
    ("Dv", 512, -7),                     # V is the whole record
    ("I", 128, -7),                      # one index head
    ("Hq", 48, -7),                      # query heads in blocks of 32
    ("record_stride", 644, -2), ("record_stride", 652, -2),
    ("k_cache", 0x10000004, -4),         # records must be 8-byte aligned
    ("y", 0x10000000 + 4096, -6),        # the output overlaps the records
    ("softcap", -1.0, -2), ("scale", float("inf"), -2),
])
def test_fp8_requests_the_library_does_not_serve_are_refused(host_lib, field, value, status):
    p = _fp8_params()
    setattr(p, field, value)
    assert host_lib.sparse_attn_decode(C.byref(p), None) == status


def test_fp8_refuses_a_fused_append_and_a_second_latent_head(host_lib):
    p = _fp8_params()
    p.k_cur = 0x400000
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -7
    p = _fp8_params()
    p.Hkv = 2
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -7


def _paged_params():
    g = sa.PagedParams()
    g.q, g.k_pool, g.v_pool, g.y = 0x100000, 0x10000000, 0x20000000, 0x200000
    g.block_table, g.ctx_len = 0x300000, 0x400000
    g.dtype = sa.F16
    g.B, g.Hq, g.Hkv, g.D, g.page_tokens, g.max_pages, g.num_pages = 2, 8, 2, 128, 16, 4, 8
    return g


@pytest.mark.parametrize("field,value,status", [
    ("dtype", 7, -3),
    ("Hq", 7, -2),                                  # Hq % Hkv
    ("num_pages", 1 << 27, -7),                     # pool rows beyond 2^31
    ("v_pool", 0x10000000 + 512, -6),               # the pools overlap
    ("y", 0x100000 + 64, -6),                       # the output overlaps q
    ("scale", float("nan"), -2),
])
def test_paged_requests_the_library_does_not_serve_are_refused(host_lib, field, value, status):
    g = _paged_params()
    setattr(g, field, value)
    assert host_lib.paged_attn_decode(C.byref(g), None) == status


def test_workspace_query_needs_no_output_pointer(lib):
    p = sa.SparseParams()
    p.q, p.k_cache, p.v_cache, p.idx = 0x10000, 0x20000, 0x30000, 0x50000
    p.B, p.Hq, p.Hkv, p.Sq, p.D, p.Dv, p.T, p.I, p.K = 4, 64, 8, 1, 128, 128, 8192, 8, 2048
    p.q_dtype = p.kv_dtype = sa.BF16
    assert lib.sparse_attn_decode_workspace(C.byref(p)) > 0


def _dense_params():
    p = sa.SparseParams()
    p.q, p.k_cache, p.v_cache, p.y, p.idx = 0x100000, 0x10000000, 0x20000000, 0x200000, 0x300000
    p.B, p.Hq, p.Hkv, p.Sq, p.D, p.Dv, p.T, p.I, p.K = 2, 8, 2, 1, 128, 128, 100, 2, 16
    p.q_dtype = p.kv_dtype = sa.BF16
    p.bias = 0x400000
    return p


@pytest.mark.parametrize("dims,status", [
    ((9,), -2),               # the last axis lines up with T = 100
    ((3, 1, 100), -2),        # 3 is neither 1 nor Hq = 8
    ((2, 8, 1, 100, 1), -2),  # rank 5
    ((2, 8, 2, 100), -2),     # Sq is 1
])
def test_bias_shapes_that_do_not_broadcast_are_refused(host_lib, dims, status):
    # [IS] validate_bias_shape: rank <= 4, every axis 1 or its target extent.
    p = _dense_params()
    p.bias_rank = len(dims)
    for r, e in enumerate(dims[:4]):
        p.bias_dims[r] = e
    assert host_lib.sparse_attn_decode(C.byref(p), None) == status
    assert host_lib.sparse_attn_decode_workspace(C.byref(p)) == 0


def test_unknown_option_bits_and_misaligned_bias_are_refused(host_lib):
    p = _dense_params()
    p.bias_rank, p.bias_dims[0] = 1, 100
    p.options = 4
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -7
    p.options, p.reserved_ = 0, 1
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -7
    p.reserved_ = 0
    p.bias = 0x400002
    assert host_lib.sparse_attn_decode(C.byref(p), None) == -4
    g = _paged_params()
    g.options = 2
    assert host_lib.paged_attn_decode(C.byref(g), None) == -7



def _index_params():
    p = sa.IndexSelectParams()
    p.query, p.weight, p.keys, p.selected = 0x100000, 0x200000, 0x10000000, 0x300000
    p.B, p.S, p.IH, p.ID, p.R, p.topk, p.key_stride, p.out_heads = 2, 1, 64, 128, 1000, 64, 68, 1
    p.query_start = 4000
    return p


@pytest.mark.parametrize("field,value,status", [
    ("ID", 96, -7), ("ID", 512, -7),        # 32, 64, 128 or 256 dims
    ("topk", 0, -2), ("topk", 5000, -7),    # 1 .. 4096
    ("IH", 0, -2), ("IH", 300, -7),
    ("key_stride", 66, -2), ("key_stride", 70, -2),  # >= 68 and a multiple of 4
    ("keys", 0x10000002, -4),
    ("selected", 0x100000 + 64, -6),       # the output overlaps the queries
    ("out_heads", 0, -2), ("reserved_", 1, -7),
])
def test_index_select_requests_the_library_does_not_serve_are_refused(host_lib, field, value,
                                                                      status):
    p = _index_params()
    setattr(p, field, value)
    assert host_lib.sparse_index_select(C.byref(p), None) == status


def test_index_select_workspace_query_needs_no_output_pointer(lib):
    p = _index_params()
    p.selected = None
    assert lib.sparse_index_select_workspace(C.byref(p)) > 0
    p.ID = 100
    assert lib.sparse_index_select_workspace(C.byref(p)) == 0


def test_compress_host_checks(host_lib):
    def params(**kw):
        p = sa.CompressParams()
        p.kv, p.gate, p.ape, p.norm = 0x100000, 0x200000, 0x300000, 0x400000
        p.carry, p.records = 0x500000, 0x600000
        p.B, p.S, p.D, p.n_rope, p.total = 2, 8, 512, 64, 8
        p.rows, p.record_stride = 2, 583
        for k, v in kw.items():
            setattr(p, k, v)
        return p

    main, index, r128 = (host_lib.csa_ratio4_main_compress, host_lib.csa_ratio4_index_compress,
                         host_lib.csa_ratio128_compress)
    assert main(C.byref(sa.CompressParams()), None) == -1
    assert main(C.byref(params(records=None)), None) == -1          # no output at all
    assert main(C.byref(params(kv=None)), None) == -1               # S > 0 needs rows
    assert main(C.byref(params(reserved_=1)), None) == -7
    assert main(C.byref(params(total=7)), None) == -2               # total < S
    assert main(C.byref(params(n_rope=63)), None) == -2             # odd RoPE width
    assert main(C.byref(params(D=520, n_rope=64)), None) == -2      # 456 not a multiple of 64
    assert main(C.byref(params(rows=1)), None) == -2                # 8 / 4 records need 2 rows
    assert main(C.byref(params(record_stride=582)), None) == -2     # 583-byte records
    assert index(C.byref(params(D=96, n_rope=64, record_stride=51)), None) == -2
    assert index(C.byref(params(D=128, n_rope=64, record_stride=67)), None) == -2  # 68 bytes
    assert r128(C.byref(params(rows=0, total=200, S=200)), None) == -2  # one 128-block closes
    assert main(C.byref(params(kv=0x100004)), None) == -4           # 16-byte alignment
    assert main(C.byref(params(records=0x500000 + 64)), None) == -6  # records inside the carry
    assert host_lib.csa_pool_weight(None, None, 4, None) == -1
    assert host_lib.csa_pool_weight(None, None, -1, None) == -2
