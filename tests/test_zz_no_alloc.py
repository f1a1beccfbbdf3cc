"""sparse_attn_decode_noalloc: the entry point for callers that cannot
allocate device memory (fixed-budget runtimes, plugins handed no scratch,
code that must avoid cudaMalloc's implicit synchronisation).  It runs the
same kernels as sparse_attn_decode with a caller workspace, so its outputs
must be identical bit for bit, call after call on its shared built-in
buffer, and it must refuse requests that do not fit.

The file is named to be collected last so that a run stopping at its first
failure has already run every other test; it depends on no other test and
passes alone in a fresh process as well.
"""
import ctypes as C

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, **over):
    kw = dict(B=8, Hq=64, Hkv=8, T=4096, K=1024, I=8, pad_prob=0.3, pad_max=200)
    kw.update(over)
    c = synth.sparse_bf16(**kw)
    return c, {k: v.to(DEV) for k, v in synth.make_sparse_inputs(c, seed=seed).items()}


def _reference(sa, c, inp):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = torch.zeros(c.B * c.I, dtype=torch.uint8, device=DEV)
    y = sa.sparse_attn_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"],
                              scale=c.eff_scale(), err_word=err, row_status=st)
    return y, err, st


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cuda_lib):
    sa = cuda_lib
    lib = sa.load()
    # A large request first, then a smaller one with another padding pattern,
    # so the second call runs on what the first left in the shared buffer.
    cases = [_case(3), _case(4, B=3, T=1500, K=400, pad_prob=0.8, pad_max=350)]
    for n, (c, inp) in enumerate(cases):
        y_ref, err_ref, st_ref = _reference(sa, c, inp)
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
        assert torch.equal(y, y_ref), f"call {n}"
        assert int(err.item()) == int(err_ref.item()) == 0
        assert torch.equal(st, st_ref)
    # a third call through the Python wrapper, on the first request again
    c, inp = cases[0]
    y_ref, _, _ = _reference(sa, c, inp)
    y = sa.sparse_attn_decode_noalloc(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"],
                                      scale=c.eff_scale())
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)


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
