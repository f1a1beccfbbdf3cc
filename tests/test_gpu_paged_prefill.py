"""GPU parity of paged causal decode and dense prefill against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _paged_small(dt, seed, **over):
    base = dict(B=5, Hq=16, Hkv=4, D=128, ctx_low=1, ctx_high=300, dtype=dt)
    base.update(over)
    c = synth.PagedCase("small", **base)
    return c, synth.make_paged_inputs(c, seed)


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("over", [dict(), dict(Hq=32, Hkv=8), dict(D=64, Hq=8, Hkv=8),
                                  dict(page_tokens=32, ctx_high=1000)])
def test_paged_decode_matches_oracle(cuda_lib, dt, over):
    c, inp = _paged_small(dt, seed=3, **over)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    # Remove the new token from the pool first: the call must write it there.
    pool_k, pool_v = g["k_pool"].clone(), g["v_pool"].clone()
    last = (g["ctx_len"] - 1).long()
    page = g["block_table"].long().gather(1, (last // c.page_tokens)[:, None])[:, 0]
    pool_k[page, :, last % c.page_tokens, :] = 0
    pool_v[page, :, last % c.page_tokens, :] = 0
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.paged_attn_decode(g["q"], pool_k, pool_v, g["block_table"], g["ctx_len"],
                                   k_new=g["k_new"], v_new=g["v_new"], scale=c.eff_scale(),
                                   err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pool_k.cpu(), inp["k_pool"]) and torch.equal(pool_v.cpu(), inp["v_pool"])
    ref = oracle.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_table"],
                              inp["ctx_len"], page_tokens=c.page_tokens, scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, f"paged {dt} {over}")


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("page_tokens", [16, 32])
def test_paged_slots_past_the_context_never_reach_the_output(cuda_lib, dt, page_tokens):
    """Pool slots past each sequence's context, in its last page, hold NaN: the
    tensor-core path loads whole pages, so those rows must be masked in K and
    zeroed in V before P.V."""
    c, inp = _paged_small(dt, seed=6, page_tokens=page_tokens, ctx_high=700)
    pool_k, pool_v = inp["k_pool"].clone(), inp["v_pool"].clone()
    for b in range(c.B):
        n = int(inp["ctx_len"][b])
        last_page = int(inp["block_table"][b, (n - 1) // c.page_tokens])
        first_free = n % c.page_tokens
        if first_free:
            pool_k[last_page, :, first_free:, :] = float("nan")
            pool_v[last_page, :, first_free:, :] = float("nan")
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.paged_attn_decode(inp["q"].to(DEV), pool_k.to(DEV), pool_v.to(DEV),
                                   inp["block_table"].to(DEV), inp["ctx_len"].to(DEV),
                                   scale=c.eff_scale(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(y.float()).all()
    ref = oracle.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_table"],
                              inp["ctx_len"], page_tokens=c.page_tokens, scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, f"paged NaN tail {dt} p{page_tokens}")


def test_paged_row_copy_path_matches_oracle(cuda_lib):
    """OPT_ROW_COPIES: pages fetched row by row instead of as TMA boxes."""
    c, inp = _paged_small("f16", seed=7, page_tokens=32, ctx_high=600)
    y = cuda_lib.paged_attn_decode(inp["q"].to(DEV), inp["k_pool"].to(DEV), inp["v_pool"].to(DEV),
                                   inp["block_table"].to(DEV), inp["ctx_len"].to(DEV),
                                   scale=c.eff_scale(), options=cuda_lib.OPT_ROW_COPIES)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_table"],
                              inp["ctx_len"], page_tokens=c.page_tokens, scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, "paged row copies")


def test_paged_batches_past_the_stream_limit_use_the_split_kernel(cuda_lib):
    """2,050 sequences (the stream kernel keeps a per-sequence prefix for at most
    2,048): the split-K kernel and its combine serve the call; contexts of 1 to
    40 tokens include single-token sequences and partial last pages."""
    c, inp = _paged_small("f16", seed=8, B=2050, Hq=8, Hkv=2, D=64, ctx_low=1, ctx_high=40)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.paged_attn_decode(inp["q"].to(DEV), inp["k_pool"].to(DEV), inp["v_pool"].to(DEV),
                                   inp["block_table"].to(DEV), inp["ctx_len"].to(DEV),
                                   scale=c.eff_scale(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_table"],
                              inp["ctx_len"], page_tokens=c.page_tokens, scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, "paged B=2050")


def test_paged_bad_table_entry_latches_and_skips(cuda_lib):
    c, inp = _paged_small("f16", seed=4)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    table = g["block_table"].clone()
    table[2, 0] = 10 ** 8
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.paged_attn_decode(g["q"], g["k_pool"], g["v_pool"], table, g["ctx_len"],
                                   scale=c.eff_scale(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & cuda_lib.ERRBIT_PAGE
    assert torch.isfinite(y.float()).all()


def test_full_size_paged_fp16_sampled_sequences(cuda_lib):
    """B128 Hq32 Hkv8 D128, ctx ~ U[1024, 32768], 16-token pages: the
    benchmark's launch configuration, checked on sampled sequences."""
    c = synth.paged_fp16()
    inp = synth.make_paged_inputs(c, seed=1, device=DEV)
    y = cuda_lib.paged_attn_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_table"],
                                   inp["ctx_len"], k_new=inp["k_new"], v_new=inp["v_new"],
                                   scale=c.eff_scale())
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    for b in rng.choice(c.B, size=6, replace=False).tolist():
        n = int(inp["ctx_len"][b])
        pages = inp["block_table"][b, : (n + c.page_tokens - 1) // c.page_tokens].long()
        kp = inp["k_pool"][pages].cpu()
        vp = inp["v_pool"][pages].cpu()
        table = torch.arange(len(pages), dtype=torch.int32)[None]
        ref = oracle.paged_decode(inp["q"][b:b + 1].cpu(), kp, vp, table,
                                  torch.tensor([n], dtype=torch.int32),
                                  page_tokens=c.page_tokens, scale=c.eff_scale())
        assert_close(to64(y[b]), ref, y.dtype, f"seq {b} ctx {n}")


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("over", [dict(), dict(causal=False), dict(softcap=0.0),
                                  dict(S=200, Hq=8, Hkv=8), dict(S=77, Hq=4, Hkv=1, D=64),
                                  dict(S=1, Hq=4, Hkv=2), dict(S=256, Hq=6, Hkv=2),
                                  dict(B=1, S=129, Hq=3, Hkv=1, causal=False),
                                  dict(S=300, D=64, softcap=0.0, causal=False),
                                  dict(S=260, softcap=5.0), dict(S=260, softcap=2.0, causal=False),
                                  dict(S=300, softcap=100.0), dict(S=129, softcap=80.0, causal=False),
                                  # D = 256: the stream kernel's dense source (TMA boxes of
                                  # consecutive rows) instead of the tcgen05 prefill
                                  dict(B=1, S=150, Hq=4, Hkv=2, D=256),
                                  dict(B=2, S=70, Hq=2, Hkv=2, D=256, causal=False)])
def test_prefill_matches_oracle_and_present_is_exact(cuda_lib, dt, over):
    base = dict(B=2, S=333, Hq=16, Hkv=4, D=128, causal=True, softcap=50.0, dtype=dt)
    base.update(over)
    c = synth.PrefillCase("small", **base)
    inp = synth.make_prefill_inputs(c, seed=5)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    pk, pv = torch.empty_like(k), torch.empty_like(v)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.attn_prefill(q, k, v, causal=c.causal, scale=c.eff_scale(), softcap=c.softcap,
                              present_k=pk, present_v=pv, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pk.cpu(), inp["k"]) and torch.equal(pv.cpu(), inp["v"])
    ref = oracle.prefill(inp["q"], inp["k"], inp["v"], scale=c.eff_scale(), causal=c.causal,
                         softcap=c.softcap)
    assert_close(to64(y), ref, y.dtype, f"prefill {dt} {over}")


def test_prefill_reports_no_timeout_and_is_deterministic(cuda_lib):
    c = synth.PrefillCase("small", B=2, S=700, Hq=8, Hkv=2, D=128, causal=True, softcap=50.0)
    inp = synth.make_prefill_inputs(c, seed=9, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ys = [cuda_lib.attn_prefill(inp["q"], inp["k"], inp["v"], causal=True, scale=c.eff_scale(),
                                softcap=c.softcap, err_word=err) for _ in range(2)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(ys[0], ys[1])


def test_full_size_prefill_sampled_rows(cuda_lib):
    """B4 S4096 Hq32 Hkv8 D128 causal softcap 50 with present K/V, checked on
    sampled rows (first, last and random positions)."""
    c = synth.prefill_bf16()
    inp = synth.make_prefill_inputs(c, seed=1, device=DEV)
    pk, pv = torch.empty_like(inp["k"]), torch.empty_like(inp["v"])
    y = cuda_lib.attn_prefill(inp["q"], inp["k"], inp["v"], causal=True, scale=c.eff_scale(),
                              softcap=c.softcap, present_k=pk, present_v=pv)
    torch.cuda.synchronize()
    assert torch.equal(pk, inp["k"]) and torch.equal(pv, inp["v"])
    rng = np.random.default_rng(2)
    qc, kc, vc = inp["q"].cpu(), inp["k"].cpu(), inp["v"].cpu()
    rows = []
    for _ in range(48):
        b, h = int(rng.integers(c.B)), int(rng.integers(c.Hq))
        i = int(rng.choice([0, 1, c.S - 1, int(rng.integers(c.S))]))
        rows.append((b * c.Hq + h) * c.S + i)
    ref = oracle.prefill(qc, kc, vc, scale=c.eff_scale(), causal=True, softcap=c.softcap,
                         rows=rows)
    got = y.reshape(-1, c.D)[torch.tensor(rows, device=DEV)]
    assert_close(to64(got), ref, y.dtype, "prefill sampled")
