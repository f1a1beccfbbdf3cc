"""Pins for the fp64 oracle, against facts fixed outside the oracle itself:
worked examples, closed forms, library decoders, invariants, and brute force
written here in a different form (whole score matrices with an explicit mask).

These run on the CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# brute force written in matrix form (independent of the oracle's loops)
# ---------------------------------------------------------------------------

def brute_attention(q, k, v, allowed, scale, softcap=0.0, sink=None):
    """q [D], k [N, D], v [N, Dv] float64, allowed [N] bool -> y [Dv]."""
    s = (k @ q) * scale
    if softcap:
        s = softcap * np.tanh(s / softcap)
    s = np.where(allowed, s, -np.inf)
    m = s.max() if allowed.any() else -np.inf
    if m == -np.inf:
        return np.zeros(v.shape[1])
    w = np.exp(s - m)
    den = w.sum() + (np.exp(sink - m) if sink is not None else 0.0)
    return (w / den) @ v


def as64(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# storage decoders
# ---------------------------------------------------------------------------

def test_f16_all_codes_match_library():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.float16).to(torch.float64).numpy()
    got = np.array([oracle.f16_to_double(c) for c in range(65536)])
    same = (ref == got) | (np.isnan(ref) & np.isnan(got))
    assert same.all()
    assert np.signbit(got[0x8000]) and got[0x8000] == 0.0


def test_bf16_all_codes_match_library():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(c) for c in range(65536)])
    same = (ref == got) | (np.isnan(ref) & np.isnan(got))
    assert same.all()


def test_e4m3fn_all_codes_match_library_and_spec_points():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3fn_to_double(c) for c in range(256)])
    same = (ref == got) | (np.isnan(ref) & np.isnan(got))
    assert same.all()
    # OCP E4M3FN spot values: max normal, min normal, min subnormal, -0, NaN.
    assert oracle.e4m3fn_to_double(0x7E) == 448.0
    assert oracle.e4m3fn_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3fn_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3fn_to_double(0x38) == 1.0
    z = oracle.e4m3fn_to_double(0x80)
    assert z == 0.0 and math.copysign(1.0, z) < 0
    assert math.isnan(oracle.e4m3fn_to_double(0x7F))
    assert math.isnan(oracle.e4m3fn_to_double(0xFF))
    # no infinity anywhere in the code space
    assert not np.isinf(got).any()


def test_e8m0_scale():
    assert oracle.e8m0_to_double(127) == 1.0
    assert oracle.e8m0_to_double(128) == 2.0
    assert oracle.e8m0_to_double(0) == 2.0 ** -127
    assert oracle.e8m0_to_double(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_to_double(255))


def test_fp8_record_hand_built():
    # two blocks (128 FP8 dims) + 2 RoPE dims; record = 2*65 + 4 bytes
    rec = np.zeros(2 * 65 + 4, dtype=np.uint8)
    rec[0] = 128            # block 0 scale 2
    rec[1:65] = 0x38        # 1.0 each -> 2.0
    rec[65] = 125           # block 1 scale 1/4
    rec[66:130] = 0xB8      # -1.0 each -> -0.25
    rec[66 + 5] = 0x7E      # 448 -> 112
    # RoPE tail: bf16 1.5 = 0x3FC0, bf16 -2.0 = 0xC000, little-endian
    rec[130:134] = [0xC0, 0x3F, 0x00, 0xC0]
    out = oracle.decode_fp8_record(rec, 128, 2)
    exp = np.concatenate([np.full(64, 2.0), np.full(64, -0.25), [1.5, -2.0]])
    exp[64 + 5] = 112.0
    assert np.array_equal(out, exp)


def test_fp8_quantizer_roundtrip_within_e4m3_half_ulp():
    nope = synth.normal((64, 512), "f32", 3)
    rope = synth.normal((64, 64), "bf16", 4)
    rec = synth.quantize_fp8_block64_records(nope, rope)
    assert rec.shape == (64, 648)
    for r in range(0, 64, 7):
        dec = oracle.decode_fp8_record(rec[r], 512, 64)
        x = nope[r].double().numpy()
        for blk in range(8):
            seg = x[blk * 64:(blk + 1) * 64]
            scale = 2.0 ** (int(rec[r, blk * 65]) - 127)
            assert np.abs(seg).max() / scale <= 448.0
            err = np.abs(dec[blk * 64:(blk + 1) * 64] - seg)
            # RNE to 3 mantissa bits: error <= 2^-4 relative for normals,
            # <= half the subnormal step 2^-10 * scale otherwise.
            bound = np.maximum(np.abs(seg) * 2.0 ** -4, 2.0 ** -10 * scale)
            assert (err <= bound * (1 + 1e-12)).all()
        assert np.array_equal(dec[512:], rope[r].double().numpy())


# ---------------------------------------------------------------------------
# index validation
# ---------------------------------------------------------------------------

def _independent_status(row, bound):
    """Second, differently organised statement of the row rules: locate the
    first column whose value breaks the rule set given all earlier columns
    passed; a row without any kept index is all padding."""
    first_pad = next((c for c, v in enumerate(row) if v == -1), len(row))
    for c, v in enumerate(row):
        if v == -1:
            continue
        if v <= -2:
            return 1, c
        if c > first_pad:
            return 2, c
        if not (0 <= v < bound):
            return 4, c
        if c > 0:
            p = row[c - 1]  # earlier columns passed and none is padding here
            if v == p:
                return 16, c
            if v < p:
                return 8, c
    if all(v == -1 for v in row):
        return 32, -1
    return 0, -1


def test_validation_brute_force_all_small_rows():
    values = list(range(-2, 6))
    bound = 4
    n = 0
    for width in range(1, 5):
        for row in itertools.product(values, repeat=width):
            code, col = oracle.validate_row(list(row), bound)
            assert (code, col) == _independent_status(list(row), bound), row
            n += 1
    assert n == 8 + 64 + 512 + 4096


def test_validation_messages_golden():
    path = os.path.join(GOLDEN, "validation_messages.txt")
    cases = 0
    with open(path) as f:
        text = f.read()
    for line in text.splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        name, bound, exp, col = parts[0], int(parts[1]), int(parts[2]), int(parts[3])
        row = [int(x) for x in parts[4:]]
        assert oracle.validate_row(row, bound) == (exp, col), name
        cases += 1
    assert cases == 10


def test_validation_tensor_status_and_error_word():
    idx = torch.tensor([[[[0, 1, 2, -1]], [[3, 3, -1, -1]]],
                        [[[-1, -1, -1, -1]], [[5, 4, 9, -1]]]], dtype=torch.int32)
    status, err = oracle.validate_indices(idx, bound=6)
    # [5, 4, 9]: column 1 (4 after 5) fails before column 2 (9 >= 6) is seen.
    assert status.tolist() == [0, 16, 32, 8]
    assert err == 16 | 32 | 8


def test_validation_first_column_wins():
    idx = torch.tensor([[[[5, 4, 9, -1]]]], dtype=torch.int64)
    status, err = oracle.validate_indices(idx, bound=6)
    assert status.tolist() == [8] and err == 8


def test_validation_per_batch_bound_and_or_word():
    idx = torch.tensor([[[[0, 7]]], [[[0, 7]]]], dtype=torch.int32)
    status, err = oracle.validate_indices(idx, bound=0, bound_per_batch=[8, 7])
    assert status.tolist() == [0, 4] and err == 4
    idx2 = torch.tensor([[[[0, 0]], [[-1, -1]]]], dtype=torch.int32)
    status, err = oracle.validate_indices(idx2, bound=8)
    assert status.tolist() == [16, 32] and err == 48


# ---------------------------------------------------------------------------
# present KV
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_present_concat_matches_cat(dt):
    past = synth.normal((2, 3, 5, 8), dt, 1)
    cur = synth.normal((2, 3, 2, 8), dt, 2)
    out = oracle.present_concat(past, cur)
    assert torch.equal(out.view(torch.uint8) if dt == "f32" else out,
                       torch.cat([past, cur], dim=2).view(torch.uint8)
                       if dt == "f32" else torch.cat([past, cur], dim=2))
    wide = oracle.present_concat(past, cur, out_stride=11)
    assert torch.equal(wide[:, :, :7], torch.cat([past, cur], dim=2))
    assert not wide[:, :, 7:].any()


def test_present_append_writes_only_the_slots():
    cache = synth.normal((2, 2, 16, 4), "bf16", 5)
    cur = synth.normal((2, 2, 1, 4), "bf16", 6)
    out = oracle.present_append(cache, cur, [3, 15])
    exp = cache.clone()
    exp[0, :, 3] = cur[0, :, 0]
    exp[1, :, 15] = cur[1, :, 0]
    assert torch.equal(out.view(torch.int16), exp.view(torch.int16))


# ---------------------------------------------------------------------------
# attention: worked examples and closed forms
# ---------------------------------------------------------------------------

def _one_row(q, k, v, keys, scale, softcap=0.0, **kw):
    """Single (b=0, h=0) row over the given key list, f32 storage."""
    D = len(q)
    qt = torch.tensor(q, dtype=torch.float32).reshape(1, 1, 1, D)
    kt = torch.tensor(k, dtype=torch.float32).reshape(1, 1, -1, D)
    vt = torch.tensor(v, dtype=torch.float32).reshape(1, 1, kt.shape[2], -1)
    idx = torch.tensor(keys, dtype=torch.int32).reshape(1, 1, 1, -1)
    return oracle.sparse_attention(qt, idx, kt, vt, scale=scale, softcap=softcap, **kw)[0]


def test_golden_two_token_examples():
    with open(os.path.join(GOLDEN, "two_token_softmax.txt")) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert [l[0] for l in lines] == ["plain", "softcap"]
    # plain: k1 = ln 3 as stored in f32; closed form with the stored value
    k1 = float(np.float32(math.log(3.0)))
    y = _one_row([1.0], [[0.0], [k1]], [[0.0], [4.0]], [0, 1], scale=1.0)
    assert abs(y[0] - 4.0 * math.exp(k1) / (1.0 + math.exp(k1))) < 1e-15
    assert abs(y[0] - 3.0) < 1e-6
    # softcap = 1: s = (0, tanh 1)
    y = _one_row([1.0], [[0.0], [1.0]], [[0.0], [1.0]], [0, 1], scale=1.0, softcap=1.0)
    e = math.exp(math.tanh(1.0))
    assert abs(y[0] - e / (1.0 + e)) < 1e-15


def test_single_selected_key_returns_its_value_row():
    k = synth.normal((1, 1, 9, 16), "bf16", 11)
    v = synth.normal((1, 1, 9, 16), "bf16", 12)
    q = synth.normal((1, 2, 1, 16), "bf16", 13)
    idx = torch.tensor([[[[4, -1, -1]]]], dtype=torch.int32)
    y = oracle.sparse_attention(q, idx, k, v, scale=0.25)
    assert np.array_equal(y[0], as64(v[0, 0, 4]))
    assert np.array_equal(y[1], as64(v[0, 0, 4]))


def test_equal_scores_give_mean_of_values_and_weights_sum_to_one():
    T, D = 12, 8
    k = synth.normal((1, 1, T, D), "f32", 21)
    v = synth.normal((1, 1, T, D), "f32", 22)
    q0 = torch.zeros((1, 1, 1, D), dtype=torch.float32)
    keys = [1, 4, 5, 9, 11]
    idx = torch.tensor([[[keys]]], dtype=torch.int32)
    y = oracle.sparse_attention(q0, idx, k, v, scale=1.0)
    assert np.allclose(y[0], as64(v[0, 0, keys]).mean(0), rtol=0, atol=1e-15)
    # constant value rows: y equals the constant for any scores (sum p = 1)
    q = synth.normal((1, 1, 1, D), "f32", 23)
    vc = torch.full((1, 1, T, D), 0.75, dtype=torch.float32)
    y = oracle.sparse_attention(q, idx, k, vc, scale=1.3)
    assert np.allclose(y[0], 0.75, rtol=0, atol=1e-15)


def test_fully_masked_rows_give_zero():
    k = synth.normal((1, 1, 8, 4), "f32", 31)
    v = synth.normal((1, 1, 8, 4), "f32", 32)
    q = synth.normal((1, 1, 1, 4), "f32", 33)
    idx = torch.tensor([[[[2, 5, 6]]]], dtype=torch.int32)
    y = oracle.sparse_attention(q, idx, k, v, scale=1.0, kv_len=[2])
    assert np.array_equal(y[0], np.zeros(4))
    y = oracle.sparse_attention(q, idx, k, v, scale=1.0, causal=True, past_len=1)
    assert np.array_equal(y[0], np.zeros(4))
    # a sink never revives a fully masked row
    y = oracle.sparse_attention(q, idx, k, v, scale=1.0, kv_len=[1], sink=[3.0])
    assert np.array_equal(y[0], np.zeros(4))


# ---------------------------------------------------------------------------
# attention: brute force (matrix form with a -inf mask)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("I_kind", ["hq", "hkv", "one"])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_sparse_matches_brute_force_masked_dense(I_kind, dt):
    B, Hq, Hkv, T, D, K = 2, 6, 2, 40, 16, 9
    I = {"hq": Hq, "hkv": Hkv, "one": 1}[I_kind]
    q = synth.normal((B, Hq, 1, D), dt, 41)
    k = synth.normal((B, Hkv, T, D), dt, 42)
    v = synth.normal((B, Hkv, T, D), dt, 43)
    idx = synth.sorted_sample_rows(B * I, 0, T, K, 44)
    idx = synth.pad_tails(idx, 45, prob=0.5, max_pad=4).reshape(B, I, 1, K)
    scale = 0.3
    y = oracle.sparse_attention(q, idx, k, v, scale=scale, softcap=2.5,
                                sink=[0.1 * h for h in range(Hq)])
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            ih = {"hq": h, "hkv": h // g, "one": 0}[I_kind]
            sel = [j for j in idx[b, ih, 0].tolist() if j >= 0]
            allowed = np.zeros(T, dtype=bool)
            allowed[sel] = True
            exp = brute_attention(as64(q[b, h, 0]), as64(k[b, h // g]), as64(v[b, h // g]),
                                  allowed, scale, 2.5, sink=0.1 * h)
            assert np.allclose(y[b * Hq + h], exp, rtol=1e-12, atol=1e-12)


def test_golden_bias_two_token_examples():
    with open(os.path.join(GOLDEN, "bias_two_token.txt")) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert [l[0] for l in lines] == ["plain", "softcap", "neginf"]
    ln3, ln2 = float(np.float32(math.log(3.0))), float(np.float32(math.log(2.0)))
    y = _one_row([1.0], [[0.0], [0.0]], [[0.0], [4.0]], [0, 1], scale=1.0,
                 bias=torch.tensor([0.0, ln3]))
    assert abs(y[0] - 4.0 * math.exp(ln3) / (1.0 + math.exp(ln3))) < 1e-15
    assert abs(y[0] - 3.0) < 1e-6
    # the bias comes after the softcap: tanh is not applied to it
    y = _one_row([1.0], [[0.0], [1.0]], [[0.0], [1.0]], [0, 1], scale=1.0, softcap=1.0,
                 bias=torch.tensor([ln2, 0.0]))
    e = math.exp(math.tanh(1.0))
    assert abs(y[0] - e / (math.exp(ln2) + e)) < 1e-15
    # a -inf entry masks its key
    y = _one_row([1.0], [[0.0], [5.0]], [[7.0], [4.0]], [0, 1], scale=1.0,
                 bias=torch.tensor([0.0, -math.inf]))
    assert y[0] == 7.0


def _broadcast_bias(shape, B, Hq, Sq, T, seed):
    """A float32 bias of the given shape and its numpy broadcast to [B, Hq, Sq, T]."""
    g = torch.Generator().manual_seed(seed)
    bias = (torch.randn(shape, generator=g) * 0.7).to(torch.float32)
    full = np.broadcast_to(bias.double().numpy(), (B, Hq, Sq, T))
    return bias, full


@pytest.mark.parametrize("shape_kind", ["full", "h1t", "b11t", "t", "st", "scalar1"])
def test_bias_broadcast_matches_brute_force(shape_kind):
    B, Hq, Hkv, Sq, T, D, K = 2, 4, 2, 2, 30, 8, 7
    shape = {"full": (B, Hq, Sq, T), "h1t": (Hq, 1, T), "b11t": (B, 1, 1, T), "t": (T,),
             "st": (Sq, T), "scalar1": (1, 1, 1, 1)}[shape_kind]
    q = synth.normal((B, Hq, Sq, D), "f32", 61)
    k = synth.normal((B, Hkv, T, D), "f32", 62)
    v = synth.normal((B, Hkv, T, D), "f32", 63)
    idx = synth.sorted_sample_rows(B * Hkv * Sq, 0, T, K, 64).reshape(B, Hkv, Sq, K)
    bias, full = _broadcast_bias(shape, B, Hq, Sq, T, 65)
    scale, cap = 0.4, 3.0
    y = oracle.sparse_attention(q, idx, k, v, scale=scale, softcap=cap, bias=bias)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                sel = idx[b, h // g, i].tolist()
                kk, vv = as64(k[b, h // g]), as64(v[b, h // g])
                s = cap * np.tanh((kk @ as64(q[b, h, i])) * scale / cap) + full[b, h, i]
                allowed = np.zeros(T, dtype=bool)
                allowed[sel] = True
                s = np.where(allowed, s, -np.inf)
                w = np.exp(s - s.max())
                exp = (w / w.sum()) @ vv
                row = (b * Hq + h) * Sq + i
                assert np.allclose(y[row], exp, rtol=1e-12, atol=1e-12)


def test_bias_neg_inf_equals_dropping_the_key_and_constant_bias_changes_nothing():
    B, Hq, T, D, K = 1, 3, 24, 8, 6
    q = synth.normal((B, Hq, 1, D), "bf16", 71)
    k = synth.normal((B, 1, T, D), "bf16", 72)
    v = synth.normal((B, 1, T, D), "bf16", 73)
    idx = torch.tensor([[[[1, 5, 8, 13, 20, 22]]]], dtype=torch.int32)
    base = oracle.sparse_attention(q, idx, k, v, scale=0.3)
    # the same bias for every key of a row is a shift: softmax is unchanged
    shift = torch.tensor([[[1.5]], [[-2.0]], [[0.25]]], dtype=torch.float32)  # [Hq, 1, 1]
    y = oracle.sparse_attention(q, idx, k, v, scale=0.3, bias=shift)
    assert np.allclose(y, base, rtol=0, atol=1e-14)
    # -inf at cache position 8 removes that key
    bias = torch.zeros(T, dtype=torch.float32)
    bias[8] = -math.inf
    y = oracle.sparse_attention(q, idx, k, v, scale=0.3, bias=bias)
    dropped = torch.tensor([[[[1, 5, 13, 20, 22, -1]]]], dtype=torch.int32)
    assert np.array_equal(y, oracle.sparse_attention(q, dropped, k, v, scale=0.3))
    # -inf everywhere: a fully masked row gives 0
    y = oracle.sparse_attention(q, idx, k, v, scale=0.3, bias=torch.full((T,), -math.inf))
    assert np.array_equal(y, np.zeros_like(y))


def test_bias_with_window_and_fp8_records_keys_by_cache_position():
    # window ∪ selected over FP8 records: brute force over the decoded cache
    B, Hq, T, W, K = 1, 2, 40, 6, 5
    nope = synth.normal((B, 1, T, 512), "f32", 81)
    rope = synth.normal((B, 1, T, 64), "bf16", 84)
    rec = synth.quantize_fp8_block64_records(nope, rope)
    q = synth.normal((B, Hq, 1, 576), "bf16", 82)
    idx = torch.tensor([[[[3, 9, 17, 35, 38]]]], dtype=torch.int32)
    bias, full = _broadcast_bias((Hq, 1, T), B, Hq, 1, T, 83)
    y = oracle.sparse_attention(q, idx, records=rec, n_rope=64, scale=0.05, window=W,
                                bias=bias)
    dec = np.stack([oracle.decode_fp8_record(rec[0, 0, t], 512, 64) for t in range(T)])
    keys = sorted(set(range(T - W, T)) | {3, 9, 17})
    for h in range(Hq):
        allowed = np.zeros(T, dtype=bool)
        allowed[keys] = True
        s = (dec @ as64(q[0, h, 0])) * 0.05 + full[0, h, 0]
        s = np.where(allowed, s, -np.inf)
        w = np.exp(s - s.max())
        assert np.allclose(y[h], (w / w.sum()) @ dec, rtol=1e-12, atol=1e-12)


def test_bias_shape_not_broadcastable_is_rejected():
    q = synth.normal((1, 2, 1, 4), "f32", 91)
    k = synth.normal((1, 1, 10, 4), "f32", 92)
    idx = torch.tensor([[[[1, 2]]]], dtype=torch.int32)
    with pytest.raises(ValueError):
        oracle.sparse_attention(q, idx, k, k, scale=1.0, bias=torch.zeros(9))
    with pytest.raises(ValueError):
        oracle.sparse_attention(q, idx, k, k, scale=1.0, bias=torch.zeros(3, 1, 10))


def test_prefill_mask_and_padding_golden():
    with open(os.path.join(GOLDEN, "prefill_mask_two_token.txt")) as f:
        rows = {l.split()[0]: (float(l.split()[1]), float(l.split()[2]))
                for l in f if l.strip() and not l.startswith("#")}
    ln3 = float(np.float32(math.log(3.0)))
    q = torch.tensor([1.0, 1.0], dtype=torch.float32).reshape(1, 1, 2, 1)
    k = torch.tensor([0.0, ln3], dtype=torch.float32).reshape(1, 1, 2, 1)
    v = torch.tensor([0.0, 4.0], dtype=torch.float32).reshape(1, 1, 2, 1)

    def run(**kw):
        return oracle.prefill(q, k, v, scale=1.0, **kw)[:, 0]

    cases = {
        "bool_full": run(causal=False, attn_mask=torch.tensor([[True, False], [True, True]])),
        "f32_full": run(causal=False, attn_mask=torch.tensor([[0.0, 0.0], [ln3, 0.0]])),
        "bool_short": run(causal=False, attn_mask=torch.tensor([[True], [True]])),
        "causal_nonpad1": run(causal=True, nonpad_kv_seqlen=[1]),
        "causal_nonpad2": run(causal=True, nonpad_kv_seqlen=[2]),
    }
    assert set(cases) == set(rows)
    for name, y in cases.items():
        assert np.allclose(y, rows[name], rtol=0, atol=1e-6), (name, y)


def _brute_prefill(q, k, v, scale, causal, softcap, mask_full, nonpad):
    """Masked dense attention in matrix form with numpy broadcasting."""
    B, Hq, S, D = q.shape
    g = Hq // k.shape[1]
    y = np.zeros((B, Hq, S, D))
    for b in range(B):
        for h in range(Hq):
            s = (as64(q[b, h]) @ as64(k[b, h // g]).T) * scale
            if softcap:
                s = softcap * np.tanh(s / softcap)
            allowed = np.ones((S, S), dtype=bool)
            off = 0
            if nonpad is not None:
                allowed[:, nonpad[b]:] = False
                off = nonpad[b] - S
            if causal:
                allowed &= np.arange(S)[None, :] <= np.arange(S)[:, None] + off
            if mask_full is not None:
                s = s + np.where(allowed, mask_full[b, h], 0.0)
            s = np.where(allowed, s, -np.inf)
            for i in range(S):
                if np.isneginf(s[i]).all():
                    continue
                w = np.exp(s[i] - s[i].max())
                y[b, h, i] = (w / w.sum()) @ as64(v[b, h // g])
    return y


@pytest.mark.parametrize("kind", ["bool_ss", "f32_b1ss", "bf16_hss", "f16_s", "none"])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_mask_and_padding_match_brute_force(kind, causal):
    B, Hq, Hkv, S, D = 2, 4, 2, 12, 8
    q = synth.normal((B, Hq, S, D), "f32", 101)
    k = synth.normal((B, Hkv, S, D), "f32", 102)
    v = synth.normal((B, Hkv, S, D), "f32", 103)
    g = torch.Generator().manual_seed(104)
    shape = {"bool_ss": (S, S), "f32_b1ss": (B, 1, S, S), "bf16_hss": (Hq, S, S),
             "f16_s": (S,), "none": None}[kind]
    mask = None
    full = None
    if shape is not None:
        if kind.startswith("bool"):
            mask = torch.rand(shape, generator=g) > 0.3
            full = np.broadcast_to(np.where(mask.numpy(), 0.0, -np.inf), (B, Hq, S, S))
        else:
            dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[
                kind.split("_")[0]]
            mask = (torch.randn(shape, generator=g) * 2.0).to(dt)
            full = np.broadcast_to(mask.double().numpy(), (B, Hq, S, S))
    nonpad = [9, 12]
    y = oracle.prefill(q, k, v, scale=0.35, causal=causal, softcap=4.0, attn_mask=mask,
                       nonpad_kv_seqlen=nonpad).reshape(B, Hq, S, D)
    exp = _brute_prefill(q, k, v, 0.35, causal, 4.0, full, nonpad)
    assert np.allclose(y, exp, rtol=1e-12, atol=1e-12)


def test_prefill_padding_to_full_length_and_zero_mask_change_nothing():
    B, Hq, Hkv, S, D = 2, 4, 2, 10, 8
    q = synth.normal((B, Hq, S, D), "bf16", 111)
    k = synth.normal((B, Hkv, S, D), "bf16", 112)
    v = synth.normal((B, Hkv, S, D), "bf16", 113)
    base = oracle.prefill(q, k, v, scale=0.3, causal=True)
    assert np.array_equal(oracle.prefill(q, k, v, scale=0.3, causal=True,
                                         nonpad_kv_seqlen=[S, S]), base)
    assert np.array_equal(oracle.prefill(q, k, v, scale=0.3, causal=True,
                                         attn_mask=torch.zeros(S, S)), base)


def test_window_union_matches_brute_force_and_counts_each_key_once():
    B, T, D, K, W = 2, 50, 8, 6, 10
    q = synth.normal((B, 3, 1, D), "f32", 51)
    k = synth.normal((B, 1, T, D), "f32", 52)
    v = synth.normal((B, 1, T, D), "f32", 53)
    # indices drawn from the whole cache: entries inside the window must not
    # be counted twice
    idx = synth.sorted_sample_rows(B, 0, T, K, 54).reshape(B, 1, 1, K)
    idx[0, 0, 0, -1] = T - 2  # force an overlap with the window
    idx[0, 0, 0] = torch.sort(idx[0, 0, 0]).values
    kv_len = [T, T - 7]
    y = oracle.sparse_attention(q, idx, k, v, scale=0.5, window=W, kv_len=kv_len)
    for b in range(B):
        L = kv_len[b]
        allowed = np.zeros(T, dtype=bool)
        allowed[max(0, L - W):L] = True
        for j in idx[b, 0, 0].tolist():
            if 0 <= j < L:
                allowed[j] = True
        for h in range(3):
            exp = brute_attention(as64(q[b, h, 0]), as64(k[b, 0]), as64(v[b, 0]), allowed,
                                  0.5)
            assert np.allclose(y[b * 3 + h], exp, rtol=1e-12, atol=1e-12)


def test_fp8_records_match_brute_force_on_library_decode():
    B, T, H = 2, 30, 4
    nope = synth.normal((B, T, 128), "f32", 61) * 3.0
    rope = synth.normal((B, T, 16), "bf16", 62)
    rec = synth.quantize_fp8_block64_records(nope, rope).reshape(B, 1, T, -1)
    q = synth.normal((B, H, 1, 144), "bf16", 63)
    idx = synth.sorted_sample_rows(B, 0, T - 5, 7, 64).reshape(B, 1, 1, 7)
    y = oracle.sparse_attention(q, idx, records=rec, n_rope=16, scale=1 / 12.0, window=5)
    # decode through the library (torch float8) rather than the oracle
    r = rec.reshape(B, T, -1)
    codes = r[:, :, :130].reshape(B, T, 2, 65)
    scl = torch.exp2(codes[:, :, :, 0].double() - 127)
    vals = codes[:, :, :, 1:].contiguous().view(torch.float8_e4m3fn).double() * scl[..., None]
    tail = r[:, :, 130:162].contiguous().view(torch.bfloat16).double()
    kv = torch.cat([vals.reshape(B, T, 128), tail], dim=2).numpy()
    for b in range(B):
        allowed = np.zeros(T, dtype=bool)
        allowed[T - 5:] = True
        allowed[[j for j in idx[b, 0, 0].tolist() if j >= 0]] = True
        for h in range(H):
            exp = brute_attention(as64(q[b, h, 0]), kv[b], kv[b], allowed, 1 / 12.0)
            assert np.allclose(y[b * H + h], exp, rtol=1e-12, atol=1e-12)


def test_gqa_equals_mha_with_replicated_kv_heads():
    B, Hq, Hkv, T, D = 1, 8, 2, 20, 8
    q = synth.normal((B, Hq, 1, D), "bf16", 71)
    k = synth.normal((B, Hkv, T, D), "bf16", 72)
    v = synth.normal((B, Hkv, T, D), "bf16", 73)
    idx = synth.sorted_sample_rows(1, 0, T, 6, 74).reshape(1, 1, 1, 6)
    y_gqa = oracle.sparse_attention(q, idx, k, v, scale=0.4)
    kr = k.repeat_interleave(Hq // Hkv, dim=1)
    vr = v.repeat_interleave(Hq // Hkv, dim=1)
    y_mha = oracle.sparse_attention(q, idx, kr, vr, scale=0.4)
    assert np.array_equal(y_gqa, y_mha)


def test_prefill_causal_softcap_matches_brute_force():
    B, Hq, Hkv, S, D = 1, 4, 2, 13, 8
    q = synth.normal((B, Hq, S, D), "bf16", 81)
    k = synth.normal((B, Hkv, S, D), "bf16", 82)
    v = synth.normal((B, Hkv, S, D), "bf16", 83)
    y = oracle.prefill(q, k, v, scale=0.35, causal=True, softcap=1.5)
    for h in range(Hq):
        for i in range(S):
            allowed = np.arange(S) <= i
            exp = brute_attention(as64(q[0, h, i]), as64(k[0, h // 2]), as64(v[0, h // 2]),
                                  allowed, 0.35, 1.5)
            assert np.allclose(y[h * S + i], exp, rtol=1e-12, atol=1e-12)
    yn = oracle.prefill(q, k, v, scale=0.35, causal=False)
    exp = brute_attention(as64(q[0, 3, 0]), as64(k[0, 1]), as64(v[0, 1]),
                          np.ones(S, dtype=bool), 0.35)
    assert np.allclose(yn[3 * S + 0], exp, rtol=1e-12, atol=1e-12)


def test_sparse_full_index_list_equals_last_prefill_row():
    B, Hq, Hkv, S, D = 1, 2, 1, 10, 8
    q = synth.normal((B, Hq, S, D), "f32", 91)
    k = synth.normal((B, Hkv, S, D), "f32", 92)
    v = synth.normal((B, Hkv, S, D), "f32", 93)
    yp = oracle.prefill(q, k, v, scale=0.5, causal=True)
    idx = torch.arange(S, dtype=torch.int32).reshape(1, 1, 1, S)
    ys = oracle.sparse_attention(q[:, :, S - 1:], idx, k, v, scale=0.5)
    for h in range(Hq):
        assert np.allclose(ys[h], yp[h * S + S - 1], rtol=0, atol=1e-15)


def test_paged_equals_contiguous_and_identity_table():
    c = synth.PagedCase("t", B=3, Hq=4, Hkv=2, D=8, ctx_low=5, ctx_high=40, page_tokens=4)
    inp = synth.make_paged_inputs(c, seed=5)
    y = oracle.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_table"],
                            inp["ctx_len"], page_tokens=4, scale=0.3)
    for b in range(3):
        n = int(inp["ctx_len"][b])
        pages = inp["block_table"][b, : (n + 3) // 4].long()
        kc = inp["k_pool"][pages].permute(1, 0, 2, 3).reshape(2, -1, 8)[:, :n]
        vc = inp["v_pool"][pages].permute(1, 0, 2, 3).reshape(2, -1, 8)[:, :n]
        for h in range(4):
            exp = brute_attention(as64(inp["q"][b, h, 0]), as64(kc[h // 2]), as64(vc[h // 2]),
                                  np.ones(n, dtype=bool), 0.3)
            assert np.allclose(y[b * 4 + h], exp, rtol=1e-12, atol=1e-12)
    # identity table over a contiguous cache equals the sparse path with all keys
    T = 12
    k = synth.normal((1, 1, T, 8), "f16", 6)
    v = synth.normal((1, 1, T, 8), "f16", 7)
    q = synth.normal((1, 2, 1, 8), "f16", 8)
    pool_k = k.reshape(1, 3, 4, 8).permute(1, 0, 2, 3).contiguous()
    pool_v = v.reshape(1, 3, 4, 8).permute(1, 0, 2, 3).contiguous()
    table = torch.tensor([[0, 1, 2]], dtype=torch.int32)
    yp = oracle.paged_decode(q, pool_k, pool_v, table, torch.tensor([T], dtype=torch.int32),
                             page_tokens=4, scale=0.7)
    ys = oracle.sparse_attention(q, torch.arange(T, dtype=torch.int32).reshape(1, 1, 1, T),
                                 k, v, scale=0.7)
    assert np.array_equal(yp, ys)


def test_rows_subset_matches_full_evaluation():
    c = synth.tiny_sparse()
    inp = synth.make_sparse_inputs(c, seed=1)
    full = oracle.sparse_attention(inp["q"], inp["idx"], inp["k_cache"], inp["v_cache"],
                                   scale=c.eff_scale())
    part = oracle.sparse_attention(inp["q"], inp["idx"], inp["k_cache"], inp["v_cache"],
                                   scale=c.eff_scale(), rows=[3, 0])
    assert np.array_equal(part, full[[3, 0]])
