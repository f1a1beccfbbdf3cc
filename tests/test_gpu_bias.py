"""GPU parity of the additive attention bias of selected-token decode
(IndexShare, onnx-runtime-ep-cuda src/kernels/index_share.rs: index_share_row
adds the bias entry of each selected key's cache position to its score;
bias_at broadcasts a rank <= 4 tensor right-aligned against
[batch, q_head, query, cache position]) against the fp64 oracle, through the
C ABI, on every kernel that serves the sparse call."""
import math

import pytest
import torch

import oracle
import synth
from helpers import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bias(shape, seed, neg_inf_every=0):
    g = torch.Generator().manual_seed(seed)
    b = (torch.randn(shape, generator=g) * 1.5).to(torch.float32)
    if neg_inf_every:
        flat = b.view(-1)
        flat[::neg_inf_every] = -math.inf
    return b


def _shape(kind, c, Sq):
    return {"h1t": (c.Hq, 1, c.T), "b11t": (c.B, 1, 1, c.T), "t": (c.T,),
            "full": (c.B, c.Hq, Sq, c.T), "st": (Sq, c.T)}[kind]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("kind", ["h1t", "b11t", "t", "full", "st"])
def test_dense_cache_bias_matches_oracle(cuda_lib, dt, kind):
    # GQA group of 8 sharing one index row per KV head (the stream kernel for
    # f16/bf16, the split-K kernel for f32); two query positions, a window,
    # a softcap and per-batch lengths, so the bias meets every stage.
    c = synth.sparse_bf16(dtype=dt, B=2, Hq=16, Hkv=2, T=600, K=200, I=2, pad_prob=0.3,
                          pad_max=40)
    inp = synth.make_sparse_inputs(c, seed=101)
    Sq = 2
    q2 = synth.normal((c.B, c.Hq, Sq, c.D), dt, 102)
    idx2 = inp["idx"].repeat(1, 1, Sq, 1)
    kv_len = torch.tensor([600, 377], dtype=torch.int64)
    bias = _bias(_shape(kind, c, Sq), 103, neg_inf_every=37)
    y = cuda_lib.sparse_attn_decode(q2.to(DEV), inp["k_cache"].to(DEV), inp["v_cache"].to(DEV),
                                    idx2.to(DEV), scale=c.eff_scale(), window=48, softcap=5.0,
                                    kv_len=kv_len.to(DEV), bias=bias.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_attention(q2, idx2, inp["k_cache"], inp["v_cache"], scale=c.eff_scale(),
                                  window=48, softcap=5.0, kv_len=kv_len, bias=bias)
    assert_close(to64(y), ref, y.dtype, f"bias {kind} {dt}")


@pytest.mark.parametrize("over", [dict(I=8, Hq=8, Hkv=2),        # one index row per query head
                                  dict(D=96, Hq=4, Hkv=1, I=1),  # the split-K kernel
                                  dict(D=64, Hq=32, Hkv=2, I=2)])
def test_bias_on_other_unit_shapes(cuda_lib, over):
    c = synth.sparse_bf16(B=2, T=400, K=150, pad_prob=0.4, pad_max=30, **over)
    inp = synth.make_sparse_inputs(c, seed=104)
    bias = _bias((c.B, c.Hq, 1, c.T), 105, neg_inf_every=11)
    y = cuda_lib.sparse_attn_decode(inp["q"].to(DEV), inp["k_cache"].to(DEV),
                                    inp["v_cache"].to(DEV), inp["idx"].to(DEV),
                                    scale=c.eff_scale(), bias=bias.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_attention(inp["q"], inp["idx"], inp["k_cache"], inp["v_cache"],
                                  scale=c.eff_scale(), bias=bias)
    assert_close(to64(y), ref, y.dtype, f"bias {over}")


def test_bias_of_minus_infinity_everywhere_gives_zero(cuda_lib):
    c = synth.sparse_bf16(B=2, Hq=8, Hkv=1, T=300, K=90, I=1)
    inp = synth.make_sparse_inputs(c, seed=106)
    bias = torch.full((c.T,), -math.inf, dtype=torch.float32)
    for dt in ("bf16", "f32"):
        q = inp["q"].to(torch.float32 if dt == "f32" else torch.bfloat16)
        k = inp["k_cache"].to(q.dtype)
        v = inp["v_cache"].to(q.dtype)
        y = cuda_lib.sparse_attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), inp["idx"].to(DEV),
                                        scale=c.eff_scale(), bias=bias.to(DEV),
                                        sink=torch.ones(c.Hq, device=DEV))
        torch.cuda.synchronize()
        assert torch.count_nonzero(y).item() == 0, dt


def _fp8_case(**over):
    kw = dict(B=2, Hq=128, T=3000, K=400, pad_prob=0.3, pad_max=50)
    kw.update(over)
    return synth.csa_fp8(**kw)


@pytest.mark.parametrize("Hq", [128, 32])
@pytest.mark.parametrize("kind", ["h1t", "b11t", "t"])
def test_fp8_records_bias_matches_oracle(cuda_lib, Hq, kind):
    # Requests with a bias run on the warp-level MMA kernel for every head count.
    c = _fp8_case(Hq=Hq)
    inp = synth.make_sparse_inputs(c, seed=107)
    bias = _bias(_shape(kind, c, 1), 108, neg_inf_every=23)
    y = cuda_lib.sparse_attn_decode(inp["q"].to(DEV), inp["kv_records"].to(DEV), None,
                                    inp["idx"].to(DEV), scale=c.eff_scale(), window=c.window,
                                    n_rope=c.n_rope, softcap=8.0, bias=bias.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_attention(inp["q"], inp["idx"], records=inp["kv_records"],
                                  n_rope=c.n_rope, scale=c.eff_scale(), window=c.window,
                                  softcap=8.0, bias=bias)
    assert_close(to64(y), ref, y.dtype, f"fp8 bias {kind} Hq{Hq}")


def test_fp8_warp_mma_option_serves_128_head_blocks(cuda_lib):
    c = _fp8_case(B=3, T=5000, K=1000)
    inp = synth.make_sparse_inputs(c, seed=109)
    ys = []
    for opt in (0, cuda_lib.OPT_FP8_WARP_MMA):
        ys.append(cuda_lib.sparse_attn_decode(inp["q"].to(DEV), inp["kv_records"].to(DEV), None,
                                              inp["idx"].to(DEV), scale=c.eff_scale(),
                                              window=c.window, n_rope=c.n_rope, options=opt))
    torch.cuda.synchronize()
    ref = oracle.sparse_attention(inp["q"], inp["idx"], records=inp["kv_records"],
                                  n_rope=c.n_rope, scale=c.eff_scale(), window=c.window)
    assert_close(to64(ys[0]), ref, ys[0].dtype, "fp8 tcgen05")
    assert_close(to64(ys[1]), ref, ys[1].dtype, "fp8 warp mma")
