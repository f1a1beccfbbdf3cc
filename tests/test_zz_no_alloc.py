"""sparse_attn_decode_noalloc: the entry point for callers that cannot
allocate device memory (fixed-budget runtimes, plugins handed no scratch,
code that must avoid cudaMalloc's implicit synchronisation).  It must give
the same results as sparse_attn_decode with a caller workspace, call after
call on its shared built-in buffer, and refuse requests that do not fit.

Kept in a file that pytest collects last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
from helpers import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    c = synth.sparse_bf16(B=8, Hq=64, Hkv=8, T=4096, K=1024, I=8, pad_prob=0.3, pad_max=200)
    return c, {k: v.to(DEV) for k, v in synth.make_sparse_inputs(c, seed=seed).items()}


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cuda_lib):
    sa = cuda_lib
    lib = sa.load()
    for seed in (3, 4):  # two calls in a row on the shared built-in buffer
        c, inp = _case(seed)
        err_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
        st_ref = torch.zeros(c.B * c.I, dtype=torch.uint8, device=DEV)
        y_ref = sa.sparse_attn_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"],
                                      scale=c.eff_scale(), err_word=err_ref, row_status=st_ref)
        # the same request through the C ABI, with no workspace at all
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        st = torch.full((c.B * c.I,), 77, dtype=torch.uint8, device=DEV)
        y = torch.full_like(y_ref, float("nan"))
        p = sa._sparse_params(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"], y,
                              scale=c.eff_scale(), softcap=0.0, window=0, kv_len=None,
                              past_len=0, causal=False, sink=None, err_word=err, row_status=st)
        p.workspace, p.workspace_bytes = None, 0
        rc = lib.sparse_attn_decode_noalloc(C.byref(p), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, sa.status_string(rc)
        torch.cuda.synchronize()
        assert_close(to64(y), to64(y_ref).reshape(-1), y.dtype, f"noalloc seed {seed}")
        assert int(err.item()) == int(err_ref.item()) == 0
        assert torch.equal(st, st_ref)


def test_noalloc_refuses_requests_beyond_its_buffer(cuda_lib):
    sa = cuda_lib
    lib = sa.load()
    c = synth.sparse_bf16(B=64, Hq=64, Hkv=8, T=8192, K=8192, I=8)
    q = torch.zeros((c.B, c.Hq, 1, c.D), dtype=torch.bfloat16, device=DEV)
    k = torch.empty((c.B, c.Hkv, c.T, c.D), dtype=torch.bfloat16, device=DEV)
    v = torch.empty_like(k)
    idx = torch.full((c.B, c.I, 1, c.K), -1, dtype=torch.int32, device=DEV)
    y = torch.empty_like(q)
    p = sa._sparse_params(q, k, v, idx, y, scale=0.0, softcap=0.0, window=0, kv_len=None,
                          past_len=0, causal=False, sink=None, err_word=None, row_status=None)
    need = lib.sparse_attn_decode_workspace(C.byref(p))
    assert need > sa.NOALLOC_SCRATCH_BYTES
    rc = lib.sparse_attn_decode_noalloc(C.byref(p), torch.cuda.current_stream().cuda_stream)
    assert rc == sa.ERR_SCRATCH_LIMIT
    assert "no-allocation" in sa.status_string(rc)
