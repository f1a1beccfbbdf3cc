"""GPU parity of index validation, present-KV and selected-token decode
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_sparse(sa, c, inp, **kw):
    q = inp["q"].to(DEV)
    k = inp["k_cache"].to(DEV)
    v = inp["v_cache"].to(DEV)
    idx = inp["idx"].to(DEV)
    return sa.sparse_attn_decode(q, k, v, idx, scale=c.eff_scale(), **kw)


def _oracle_sparse(c, inp, **kw):
    return oracle.sparse_attention(inp["q"], inp["idx"], inp["k_cache"], inp["v_cache"],
                                   scale=c.eff_scale(), **kw)


# ---------------------------------------------------------------------------
# index validation (bit-exact)
# ---------------------------------------------------------------------------

def _mutated_rows(rows, K, T, seed):
    """Valid rows plus one planted fault per faulty row (each rule)."""
    rng = np.random.default_rng(seed)
    idx = synth.sorted_sample_rows(rows, 0, T, K, seed).numpy()
    kinds = rng.integers(0, 8, size=rows)
    for r in range(rows):
        col = int(rng.integers(1, K))
        k = kinds[r]
        if k == 1:
            idx[r, col] = -int(rng.integers(2, 1000))           # below sentinel
        elif k == 2:
            idx[r, col - 1] = -1                                  # value after padding
        elif k == 3:
            idx[r, col] = T + int(rng.integers(0, 5))             # out of range
        elif k == 4:
            idx[r, col] = idx[r, col - 1]                         # duplicate
        elif k == 5 and idx[r, col - 1] > 0:
            idx[r, col] = idx[r, col - 1] - 1                     # decreasing
        elif k == 6:
            idx[r, :] = -1                                        # all padding
        elif k == 7:
            idx[r, col:] = -1                                     # valid tail
    return torch.from_numpy(idx)


@pytest.mark.parametrize("K", [1, 7, 32, 129, 300, 2048, 2500, 5000])
@pytest.mark.parametrize("i64", [False, True])
def test_validate_indices_bit_exact(cuda_lib, K, i64):
    sa = cuda_lib
    B, I, Sq, T = 3, 4, 2, 6000
    rows = B * I * Sq
    idx = _mutated_rows(rows, K, T, seed=K + 17 * i64) if K > 1 else \
        torch.tensor([[3], [-1], [-5], [7000], [0], [5999]] * 4)[:rows]
    idx = idx.reshape(B, I, Sq, K).to(torch.int64 if i64 else torch.int32)
    bpb = torch.tensor([T, T - 100, T], dtype=torch.int64)
    st_o, err_o = oracle.validate_indices(idx, bound=0, bound_per_batch=bpb)
    st_g, err_g = sa.validate_indices(idx.to(DEV), 0, bpb.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(st_g.cpu().numpy(), st_o)
    assert int(err_g.item()) == err_o


def test_validate_indices_unaligned_width_scalar_path(cuda_lib):
    idx = _mutated_rows(40, 13, 100, seed=5).reshape(2, 2, 10, 13).to(torch.int32)
    st_o, err_o = oracle.validate_indices(idx, bound=100)
    st_g, err_g = cuda_lib.validate_indices(idx.to(DEV), 100)
    torch.cuda.synchronize()
    assert np.array_equal(st_g.cpu().numpy(), st_o) and int(err_g.item()) == err_o


# ---------------------------------------------------------------------------
# present KV (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128, 3])
def test_present_concat_bit_exact(cuda_lib, dt, D):
    past_k, past_v = synth.normal((2, 3, 37, D), dt, 1), synth.normal((2, 3, 37, D), dt, 2)
    cur_k, cur_v = synth.normal((2, 3, 2, D), dt, 3), synth.normal((2, 3, 2, D), dt, 4)
    pk = torch.zeros((2, 3, 41, D), dtype=past_k.dtype, device=DEV)
    pv = torch.zeros_like(pk)
    cuda_lib.build_present_kv(cur_k.to(DEV), pk, past_k.to(DEV), cur_v.to(DEV), pv, past_v.to(DEV))
    torch.cuda.synchronize()
    ek = oracle.present_concat(past_k, cur_k, out_stride=41)
    ev = oracle.present_concat(past_v, cur_v, out_stride=41)
    assert torch.equal(pk.cpu().view(torch.uint8), ek.view(torch.uint8))
    assert torch.equal(pv.cpu().view(torch.uint8), ev.view(torch.uint8))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_present_append_in_place_touches_only_the_slot(cuda_lib, dt):
    cache_k = synth.normal((4, 2, 64, 128), dt, 7)
    cache_v = synth.normal((4, 2, 64, 128), dt, 8)
    cur_k = synth.normal((4, 2, 1, 128), dt, 9)
    cur_v = synth.normal((4, 2, 1, 128), dt, 10)
    wp = torch.tensor([0, 17, 63, 70], dtype=torch.int64)   # last one is out of range
    gk, gv = cache_k.to(DEV), cache_v.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cuda_lib.build_present_kv(cur_k.to(DEV), gk, gk, cur_v.to(DEV), gv, gv, write_pos=wp.to(DEV),
                              err_word=err)
    torch.cuda.synchronize()
    ok_wp = wp.clone()
    ok_wp[3] = 0
    ek = oracle.present_append(cache_k, cur_k, ok_wp)
    ev = oracle.present_append(cache_v, cur_v, ok_wp)
    ek[3] = cache_k[3]
    ev[3] = cache_v[3]
    assert torch.equal(gk.cpu().view(torch.uint8), ek.view(torch.uint8))
    assert torch.equal(gv.cpu().view(torch.uint8), ev.view(torch.uint8))
    assert int(err.item()) == cuda_lib.ERRBIT_WRITE_POS


def test_present_append_with_separate_past(cuda_lib):
    past = synth.normal((2, 2, 16, 64), "f16", 11)
    cur = synth.normal((2, 2, 3, 64), "f16", 12)
    out = torch.full((2, 2, 16, 64), 7.0, dtype=torch.float16, device=DEV)
    wp = torch.tensor([2, 13], dtype=torch.int64)
    cuda_lib.build_present_kv(cur.to(DEV), out, past.to(DEV), write_pos=wp.to(DEV))
    torch.cuda.synchronize()
    exp = oracle.present_append(past, cur, wp)
    assert torch.equal(out.cpu().view(torch.int16), exp.view(torch.int16))


# ---------------------------------------------------------------------------
# selected-token decode
# ---------------------------------------------------------------------------

def test_tiny_fp32_sparse_decode_matches_oracle(cuda_lib):
    c = synth.tiny_sparse()
    for seed in (1, 2):
        inp = synth.make_sparse_inputs(c, seed)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        y = _run_sparse(cuda_lib, c, inp, err_word=err)
        torch.cuda.synchronize()
        assert_close(to64(y), _oracle_sparse(c, inp), torch.float32, "tiny fp32")
        assert int(err.item()) == 0


CASES = [
    # name, case overrides
    ("gqa8_rows_per_kvhead", dict(B=2, Hq=16, Hkv=2, T=700, K=300, I=2)),
    ("rows_per_query_head", dict(B=2, Hq=8, Hkv=2, T=500, K=130, I=8)),
    ("one_shared_row", dict(B=3, Hq=12, Hkv=3, T=400, K=77, I=1)),
    ("mha_g1", dict(B=2, Hq=4, Hkv=4, T=300, K=65, I=4)),
    ("g16_two_ntiles", dict(B=1, Hq=32, Hkv=2, T=600, K=200, I=2)),
    ("d64", dict(B=2, Hq=8, Hkv=1, T=350, K=100, I=1, D=64)),
    ("d256", dict(B=1, Hq=8, Hkv=1, T=300, K=140, I=1, D=256)),
    ("d96_simt", dict(B=1, Hq=4, Hkv=1, T=300, K=100, I=1, D=96)),
    ("single_key_rows", dict(B=2, Hq=8, Hkv=1, T=100, K=1, I=1)),
]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("name,over", CASES, ids=[c[0] for c in CASES])
def test_sparse_decode_matches_oracle(cuda_lib, dt, name, over):
    c = synth.sparse_bf16(dtype=dt, pad_prob=0.3, pad_max=40, **over)
    inp = synth.make_sparse_inputs(c, seed=11)
    y = _run_sparse(cuda_lib, c, inp)
    torch.cuda.synchronize()
    assert_close(to64(y), _oracle_sparse(c, inp), y.dtype, name)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_sparse_decode_options(cuda_lib, dt):
    """window, per-batch kv_len, causal frontier, softcap, sink, int64 indices,
    several query positions."""
    c = synth.sparse_bf16(dtype=dt, B=3, Hq=16, Hkv=2, T=520, K=150, I=2, pad_prob=0.4,
                          pad_max=30, idx_i64=True)
    inp = synth.make_sparse_inputs(c, seed=21)
    # Sq = 2 query positions: reuse the index rows for both
    q2 = synth.normal((c.B, c.Hq, 2, c.D), dt, 22)
    idx2 = inp["idx"].repeat(1, 1, 2, 1)
    kv_len = torch.tensor([520, 431, 200], dtype=torch.int64)
    sink = torch.linspace(-1.0, 2.0, c.Hq, dtype=torch.float32)
    for opts in (dict(window=64), dict(softcap=1.5), dict(causal=True, past_len=300),
                 dict(sink=sink), dict(kv_len=kv_len, window=32, softcap=3.0)):
        inp2 = dict(inp, q=q2, idx=idx2)
        gkw = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in opts.items()}
        y = _run_sparse(cuda_lib, c, inp2, **gkw)
        torch.cuda.synchronize()
        okw = dict(opts)
        if "sink" in okw:
            okw["sink"] = okw["sink"].double()
        ref = _oracle_sparse(c, inp2, **okw)
        assert_close(to64(y), ref, y.dtype, str(list(opts)))


def test_fully_masked_rows_give_zero(cuda_lib):
    c = synth.sparse_bf16(B=2, Hq=8, Hkv=1, T=200, K=50, I=1)
    inp = synth.make_sparse_inputs(c, seed=31)
    kv_len = torch.tensor([0, 200], dtype=torch.int64, device=DEV)
    y = _run_sparse(cuda_lib, c, inp, kv_len=kv_len)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y[0]) == 0
    assert torch.count_nonzero(y[1]) > 0


def test_garbage_beyond_valid_length_does_not_change_output(cuda_lib):
    c = synth.sparse_bf16(B=2, Hq=16, Hkv=2, T=400, K=100, I=2, window=16)
    inp = synth.make_sparse_inputs(c, seed=41)
    kv_len = torch.tensor([300, 350], dtype=torch.int64, device=DEV)
    y1 = _run_sparse(cuda_lib, c, inp, kv_len=kv_len)
    k2, v2 = inp["k_cache"].clone(), inp["v_cache"].clone()
    k2[0, :, 300:] = 1e4
    v2[0, :, 300:] = float("nan")
    k2[1, :, 350:] = -3e3
    y2 = _run_sparse(cuda_lib, c, dict(inp, k_cache=k2, v_cache=v2), kv_len=kv_len)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_malformed_rows_latch_error_and_stay_finite(cuda_lib):
    c = synth.sparse_bf16(B=2, Hq=16, Hkv=2, T=300, K=64, I=2, pad_prob=0.0)
    inp = synth.make_sparse_inputs(c, seed=51)
    idx = inp["idx"].clone()
    idx[0, 0, 0, 5] = 10_000          # out of range
    idx[1, 1, 0, 3] = idx[1, 1, 0, 2]  # duplicate
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = torch.full((4,), 255, dtype=torch.uint8, device=DEV)
    y = _run_sparse(cuda_lib, c, dict(inp, idx=idx), err_word=err, row_status=st)
    torch.cuda.synchronize()
    assert int(err.item()) == (4 | 16)
    assert st.cpu().tolist() == [4, 0, 0, 16]
    assert torch.isfinite(y.float()).all()


def test_decode_is_deterministic(cuda_lib):
    c = synth.sparse_bf16(B=4, Hq=64, Hkv=8, T=4096, K=1024, I=8)
    inp = {k: v.to(DEV) for k, v in synth.make_sparse_inputs(c, seed=61).items()}
    ys = [cuda_lib.sparse_attn_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"],
                                      scale=c.eff_scale()) for _ in range(4)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(ys[0], y)


def test_full_size_sparse_bf16_sampled_rows(cuda_lib):
    """B32 Hq64 Hkv8 D128 T8192 K2048 in the benchmark's launch configuration,
    checked on sampled (batch, KV head) groups against the oracle."""
    c = synth.sparse_bf16()
    inp = synth.make_sparse_inputs(c, seed=1, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.sparse_attn_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"],
                                    scale=c.eff_scale(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(0)
    for _ in range(12):
        b, kvh = int(rng.integers(c.B)), int(rng.integers(c.Hkv))
        hs = slice(kvh * c.g, (kvh + 1) * c.g)
        ref = oracle.sparse_attention(inp["q"][b:b + 1, hs].cpu(),
                                      inp["idx"][b:b + 1, kvh:kvh + 1].cpu(),
                                      inp["k_cache"][b:b + 1, kvh:kvh + 1].cpu(),
                                      inp["v_cache"][b:b + 1, kvh:kvh + 1].cpu(),
                                      scale=c.eff_scale())
        assert_close(to64(y[b, hs]), ref, y.dtype, f"b={b} kvh={kvh}")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_fused_append_matches_append_then_decode(cuda_lib, dt):
    """k_cur/v_cur written at write_pos inside the decode call: the output equals
    the oracle over the appended cache, and the cache holds the new rows."""
    c = synth.sparse_bf16(dtype=dt, B=3, Hq=16, Hkv=2, T=600, K=200, I=2, pad_prob=0.2,
                          pad_max=30)
    inp = synth.make_sparse_inputs(c, seed=71)
    k_cur = synth.normal((c.B, c.Hkv, 2, c.D), dt, 72)
    v_cur = synth.normal((c.B, c.Hkv, 2, c.D), dt, 73)
    wp = torch.tensor([598, 100, 0], dtype=torch.int64)
    # make sure the selected sets include the appended positions
    idx = inp["idx"].clone()
    for b, w in enumerate(wp.tolist()):
        row = sorted(set(idx[b, 0, 0][idx[b, 0, 0] >= 0].tolist()[:-2]) | {w, w + 1})
        idx[b, 0, 0] = -1
        idx[b, 0, 0, :len(row)] = torch.tensor(row)
    kc, vc = inp["k_cache"].to(DEV), inp["v_cache"].to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.sparse_attn_decode(inp["q"].to(DEV), kc, vc, idx.to(DEV), scale=c.eff_scale(),
                                    k_cur=k_cur.to(DEV), v_cur=v_cur.to(DEV),
                                    write_pos=wp.to(DEV), err_word=err)
    torch.cuda.synchronize()
    ek = oracle.present_append(inp["k_cache"], k_cur, wp)
    ev = oracle.present_append(inp["v_cache"], v_cur, wp)
    assert torch.equal(kc.cpu(), ek) and torch.equal(vc.cpu(), ev)
    ref = oracle.sparse_attention(inp["q"], idx, ek, ev, scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, "fused append")
    assert int(err.item()) == 0


def test_workspace_contents_on_entry_do_not_matter(cuda_lib):
    c = synth.sparse_bf16(B=4, Hq=64, Hkv=8, T=2048, K=700, I=8, pad_prob=0.3, pad_max=100)
    inp = {k: v.to(DEV) for k, v in synth.make_sparse_inputs(c, seed=81).items()}
    err0 = torch.zeros(1, dtype=torch.int32, device=DEV)
    st0 = torch.zeros(c.B * c.I, dtype=torch.uint8, device=DEV)
    need = cuda_lib.sparse_attn_decode_workspace(inp["q"], inp["k_cache"], inp["v_cache"],
                                                 inp["idx"], scale=c.eff_scale(), err_word=err0,
                                                 row_status=st0)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)
    ys = []
    for fill in (0xAB, 0x00, 0xFF):
        ws.fill_(fill)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        st = torch.full((c.B * c.I,), 99, dtype=torch.uint8, device=DEV)
        ys.append(cuda_lib.sparse_attn_decode(inp["q"], inp["k_cache"], inp["v_cache"],
                                              inp["idx"], scale=c.eff_scale(), workspace=ws,
                                              err_word=err, row_status=st))
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and int(st.max().item()) == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_stream_row_copy_path_matches_oracle(cuda_lib, dt):
    """OPT_ROW_COPIES: the stream kernel's per-row bulk copies (the path taken
    when the caches cannot be described by tensor maps) for selected rows."""
    c = synth.sparse_bf16(B=3, T=2000, K=500, dtype=dt, pad_prob=0.5, pad_max=100)
    inp = synth.make_sparse_inputs(c, seed=33)
    y = cuda_lib.sparse_attn_decode(inp["q"].to(DEV), inp["k_cache"].to(DEV), inp["v_cache"].to(DEV),
                                    inp["idx"].to(DEV), scale=c.eff_scale(),
                                    options=cuda_lib.OPT_ROW_COPIES)
    torch.cuda.synchronize()
    ref = oracle.sparse_attention(inp["q"], inp["idx"], inp["k_cache"], inp["v_cache"],
                                  scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, f"row copies {dt}")


def test_kernel_events_bracket_the_gather_kernel_only(cuda_lib):
    c = synth.sparse_bf16(B=4, T=3000, K=700)
    inp = synth.make_sparse_inputs(c, seed=31, device=DEV)
    y = torch.empty_like(inp["q"])
    run = lambda: cuda_lib.sparse_attn_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["idx"],
                                              scale=c.eff_scale(), y=y)
    run()
    call0, call1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with cuda_lib.kernel_events(k0, k1):
        call0.record()
        run()
        call1.record()
    torch.cuda.synchronize()
    kernel_ms, call_ms = k0.elapsed_time(k1), call0.elapsed_time(call1)
    assert 0.0 < kernel_ms < call_ms
    ref = oracle.sparse_attention(inp["q"].cpu(), inp["idx"].cpu(), inp["k_cache"].cpu(),
                                  inp["v_cache"].cpu(), scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, "hooked call")


# ---------------------------------------------------------------------------
# FP8 hybrid-record latent cache (MQA, 512 E4M3 + 64 bf16 dims)
# ---------------------------------------------------------------------------

def _fp8_case(**over):
    base = dict(B=2, Hq=64, T=3000, K=300, window=128, pad_prob=0.5, pad_max=60)
    base.update(over)
    return synth.csa_fp8(**base)


def _run_fp8(sa, c, inp, **kw):
    return sa.sparse_attn_decode(inp["q"].to(DEV), inp["kv_records"].to(DEV), None,
                                 inp["idx"].to(DEV), scale=c.eff_scale(), window=c.window,
                                 n_rope=c.n_rope, **kw)


@pytest.mark.parametrize("over", [dict(), dict(record_stride=656), dict(Hq=32, K=40, T=500),
                                  dict(window=0, K=700), dict(B=3, Hq=128, T=5000, K=1000)])
def test_fp8_records_match_oracle(cuda_lib, over):
    c = _fp8_case(**over)
    inp = synth.make_sparse_inputs(c, seed=91)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = _run_fp8(cuda_lib, c, inp, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.sparse_attention(inp["q"], inp["idx"], records=inp["kv_records"],
                                  n_rope=c.n_rope, scale=c.eff_scale(), window=c.window)
    assert_close(to64(y), ref, y.dtype, f"fp8 {over}")


def test_fp8_options_kv_len_softcap_sink_and_query_positions(cuda_lib):
    c = _fp8_case(B=2, Hq=32, T=2000, K=200)
    inp = synth.make_sparse_inputs(c, seed=92)
    q2 = synth.normal((c.B, c.Hq, 2, c.D), "bf16", 93)
    idx2 = inp["idx"].repeat(1, 1, 2, 1)
    kv_len = torch.tensor([2000, 1500], dtype=torch.int64)
    sink = torch.linspace(-2.0, 1.0, c.Hq, dtype=torch.float32)
    inp2 = dict(inp, q=q2, idx=idx2)
    y = _run_fp8(cuda_lib, c, inp2, kv_len=kv_len.to(DEV), softcap=4.0, sink=sink.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_attention(q2, idx2, records=inp["kv_records"], n_rope=c.n_rope,
                                  scale=c.eff_scale(), window=c.window, kv_len=kv_len,
                                  softcap=4.0, sink=sink.double())
    assert_close(to64(y), ref, y.dtype, "fp8 options")


# Blocks of 128 query heads run on the tcgen05 kernel (128-key tiles, three
# CTAs per output block): every option, several head blocks, many key splits.
@pytest.mark.parametrize("over", [dict(Hq=128), dict(Hq=128, record_stride=656),
                                  dict(Hq=128, window=0, K=700, pad_prob=0.0),
                                  dict(Hq=256, B=1, T=4000, K=900),
                                  dict(Hq=128, B=1, T=30000, K=6000),
                                  dict(Hq=128, B=5, T=700, K=60, window=16)])
def test_fp8_tc05_head_blocks_match_oracle(cuda_lib, over):
    c = _fp8_case(**over)
    inp = synth.make_sparse_inputs(c, seed=94)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = _run_fp8(cuda_lib, c, inp, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.sparse_attention(inp["q"], inp["idx"], records=inp["kv_records"],
                                  n_rope=c.n_rope, scale=c.eff_scale(), window=c.window)
    assert_close(to64(y), ref, y.dtype, f"fp8 tc05 {over}")


def test_fp8_tc05_malformed_rows_status_and_outputs(cuda_lib):
    # The tcgen05 FP8 path plans its candidates inside the decode kernel while
    # the plan kernel only validates beside it: statuses must equal the
    # oracle's, valid rows must match the oracle (a malformed row's output is
    # only required to be finite), and the output must not depend on whether
    # a status output was asked for.
    c = _fp8_case(B=5, Hq=128, T=2000, K=300, pad_prob=0.0)
    inp = synth.make_sparse_inputs(c, seed=96)
    idx = inp["idx"].clone()
    idx[0, 0, 0, 7] = 5_000                 # out of range
    idx[1, 0, 0, 10] = idx[1, 0, 0, 9]      # duplicate
    idx[2, 0, 0, 20:] = -1                  # valid trailing padding
    idx[2, 0, 0, 25] = 3                    # after padding
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = torch.full((c.B,), 255, dtype=torch.uint8, device=DEV)
    dev = dict(q=inp["q"].to(DEV), rec=inp["kv_records"].to(DEV), idx=idx.to(DEV))
    y = cuda_lib.sparse_attn_decode(dev["q"], dev["rec"], None, dev["idx"], scale=c.eff_scale(),
                                    window=c.window, n_rope=c.n_rope, err_word=err, row_status=st)
    y_plain = cuda_lib.sparse_attn_decode(dev["q"], dev["rec"], None, dev["idx"],
                                          scale=c.eff_scale(), window=c.window, n_rope=c.n_rope)
    torch.cuda.synchronize()
    status, e = oracle.validate_indices(idx, bound=c.T)
    assert st.cpu().tolist() == status.tolist()
    assert int(err.item()) == e and e != 0
    assert torch.equal(y, y_plain)
    assert torch.isfinite(y.float()).all()
    ok = [b for b in range(c.B) if status[b] == 0]
    assert ok == [3, 4]
    rows = [b * c.Hq + h for b in ok for h in range(c.Hq)]
    ref = oracle.sparse_attention(inp["q"], idx, records=inp["kv_records"], n_rope=c.n_rope,
                                  scale=c.eff_scale(), window=c.window, rows=rows)
    assert_close(to64(y.reshape(-1, c.D)[rows]), ref, y.dtype, "fp8 tc05 valid rows")


@pytest.mark.parametrize("kv_len", [None, [700, 300, 90]])
def test_fp8_tc05_window_only_matches_oracle(cuda_lib, kv_len):
    # No index rows (K = 0): the candidates are the window alone, and no plan
    # kernel runs before the decode.
    c = _fp8_case(B=3, Hq=128, T=700, K=8, window=128, pad_prob=0.0)
    inp = synth.make_sparse_inputs(c, seed=97)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kl = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int64)
    y = cuda_lib.sparse_attn_decode(inp["q"].to(DEV), inp["kv_records"].to(DEV), None, None,
                                    scale=c.eff_scale(), window=c.window, n_rope=c.n_rope,
                                    err_word=err, kv_len=None if kl is None else kl.to(DEV))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    idx0 = torch.empty((c.B, 1, 1, 0), dtype=torch.int32)
    ref = oracle.sparse_attention(inp["q"], idx0, records=inp["kv_records"], n_rope=c.n_rope,
                                  scale=c.eff_scale(), window=c.window, kv_len=kl)
    assert_close(to64(y), ref, y.dtype, f"fp8 tc05 window only kv_len={kv_len}")


@pytest.mark.parametrize("stride,shift", [(664, 0), (648, 8), (656, 8), (704, 8)])
def test_fp8_tc05_record_windows_match_oracle(cuda_lib, stride, shift):
    # Records are 8-byte aligned; the decoder fetches each as the 16-byte-aligned
    # window around it, which starts 0 or 8 bytes before the record.  Strides and
    # a cache base 8 bytes past a 16-byte boundary cover both starts.
    c = _fp8_case(Hq=128, record_stride=stride)
    inp = synth.make_sparse_inputs(c, seed=95)
    rec = inp["kv_records"]
    buf = torch.zeros(rec.numel() + 16, dtype=torch.uint8, device=DEV)
    dev_rec = buf[shift:shift + rec.numel()].view(rec.shape)
    dev_rec.copy_(rec.to(DEV))
    assert dev_rec.data_ptr() % 16 == shift
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.sparse_attn_decode(inp["q"].to(DEV), dev_rec, None, inp["idx"].to(DEV),
                                    scale=c.eff_scale(), window=c.window, n_rope=c.n_rope,
                                    err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.sparse_attention(inp["q"], inp["idx"], records=rec, n_rope=c.n_rope,
                                  scale=c.eff_scale(), window=c.window)
    assert_close(to64(y), ref, y.dtype, f"fp8 tc05 stride {stride} shift {shift}")


@pytest.mark.parametrize("over", [dict(B=16, T=3000, K=1000),   # 3 splits of 3 tiles
                                  dict(B=52, T=900, K=400)])    # 1 split of 5 tiles
def test_fp8_tc05_several_tiles_per_cta(cuda_lib, over):
    c = _fp8_case(Hq=128, **over)
    inp = synth.make_sparse_inputs(c, seed=98)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = _run_fp8(cuda_lib, c, inp, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = list(range(0, c.B * c.Hq, 5))
    ref = oracle.sparse_attention(inp["q"], inp["idx"], records=inp["kv_records"],
                                  n_rope=c.n_rope, scale=c.eff_scale(), window=c.window,
                                  rows=rows)
    assert_close(to64(y.reshape(-1, c.D)[rows]), ref, y.dtype, f"fp8 tc05 tiles {over}")


def test_fp8_tc05_options_kv_len_softcap_sink_and_query_positions(cuda_lib):
    c = _fp8_case(B=2, Hq=128, T=2500, K=400)
    inp = synth.make_sparse_inputs(c, seed=95)
    q2 = synth.normal((c.B, c.Hq, 2, c.D), "bf16", 96)
    idx2 = inp["idx"].repeat(1, 1, 2, 1)
    kv_len = torch.tensor([2500, 1300], dtype=torch.int64)
    sink = torch.linspace(-2.0, 1.0, c.Hq, dtype=torch.float32)
    inp2 = dict(inp, q=q2, idx=idx2)
    for softcap in (0.0, 4.0):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        y = _run_fp8(cuda_lib, c, inp2, kv_len=kv_len.to(DEV), softcap=softcap,
                     sink=sink.to(DEV), err_word=err)
        torch.cuda.synchronize()
        # indices at or past kv_len[1] are flagged (and masked), nothing else
        assert int(err.item()) == 4
        ref = oracle.sparse_attention(q2, idx2, records=inp["kv_records"], n_rope=c.n_rope,
                                      scale=c.eff_scale(), window=c.window, kv_len=kv_len,
                                      softcap=softcap, sink=sink.double())
        assert_close(to64(y), ref, y.dtype, f"fp8 tc05 options softcap={softcap}")


@pytest.mark.parametrize("past_len", [2400, 2450])
def test_fp8_tc05_causal_frontier_matches_oracle(cuda_lib, past_len):
    # Query position i sees keys <= past_len + i: the frontier cuts through the
    # 128-token window [2372, 2500) and through the selected indices.
    c = _fp8_case(B=2, Hq=128, T=2500, K=400)
    inp = synth.make_sparse_inputs(c, seed=99)
    q2 = synth.normal((c.B, c.Hq, 2, c.D), "bf16", 100)
    idx2 = inp["idx"].repeat(1, 1, 2, 1)
    inp2 = dict(inp, q=q2, idx=idx2)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = _run_fp8(cuda_lib, c, inp2, causal=True, past_len=past_len, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.sparse_attention(q2, idx2, records=inp["kv_records"], n_rope=c.n_rope,
                                  scale=c.eff_scale(), window=c.window, causal=True,
                                  past_len=past_len)
    assert_close(to64(y), ref, y.dtype, f"fp8 tc05 causal past_len={past_len}")


def test_fp8_tc05_is_deterministic(cuda_lib):
    c = _fp8_case(B=2, Hq=128, T=6000, K=1500)
    inp = synth.make_sparse_inputs(c, seed=97)
    y1 = _run_fp8(cuda_lib, c, inp)
    y2 = _run_fp8(cuda_lib, c, inp)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_full_size_fp8_sampled_rows(cuda_lib):
    """B16 Hq128 MQA D576 (648-byte records) T65536, window 128 + top-k 2048,
    the benchmark's launch configuration, checked on sampled batches."""
    c = synth.csa_fp8()
    inp = synth.make_sparse_inputs(c, seed=1, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.sparse_attn_decode(inp["q"], inp["kv_records"], None, inp["idx"],
                                    scale=c.eff_scale(), window=c.window, n_rope=c.n_rope,
                                    err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the sampled batches' rows hold selected entries inside the window, which
    # the union must count once
    inside = (inp["idx"][:, 0, 0] >= c.T - c.window).sum(dim=1).cpu()
    overlapping = [b for b in range(c.B) if int(inside[b]) > 0]
    assert overlapping
    for b in sorted({0, 11, overlapping[0]}):
        heads = list(range(0, c.Hq, 9))
        ref = oracle.sparse_attention(inp["q"][b:b + 1].cpu(), inp["idx"][b:b + 1].cpu(),
                                      records=inp["kv_records"][b:b + 1].cpu(), n_rope=c.n_rope,
                                      scale=c.eff_scale(), window=c.window, rows=heads)
        assert_close(to64(y[b, heads]), ref, y.dtype, f"fp8 full b={b}")
