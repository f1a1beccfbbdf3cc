"""Pins for the oracle's CSA compression stages (ratio 128, ratio 4 attention
records and index keys), checked against what the pages and the mathematics
fix rather than against the oracle itself:

* the FP8 block quantizer: E4M3FN codes against torch's float8_e4m3fn
  conversion (a library routine), the block-exponent rule on hand-worked
  blocks, the round trip within half an E4M3 step;
* softmax pooling: closed forms (equal scores give the mean, a dominant
  candidate gives its value, two candidates give the logistic function,
  -inf candidates drop out);
* the compressed RoPE: identity at position 0 and the YaRN-ramped
  frequencies of the pages (base 160000, factor 16, pairs 15..25) against a
  double evaluation;
* RMSNorm and the record layouts: constant and one-hot records worked by
  hand through to their stored bytes;
* the stream: every record equals the pooling of the tokens that the block
  formula names (ratio 4: the previous block's first source half and the
  current block's second half; ratio 128: the block's 128 tokens), with the
  carry mechanics left out, and chunked calls equal one call.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _torch_e4m3(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def _e4m3_values():
    return np.array([oracle.e4m3fn_to_double(c) for c in range(0x7F)], dtype=np.float64)


# -------------------------------------------------------------------- FP8 block


def test_fp8_codes_match_torch_on_grid_points_midpoints_and_random():
    grid = _e4m3_values()  # 0 .. 448, increasing
    mids = (grid[:-1] + grid[1:]) / 2  # ties: both sides must pick the even code
    rng = np.random.default_rng(5)
    rand = rng.uniform(-448, 448, size=4000)
    tiny = np.array([-0.0, 2.0 ** -12, -2.0 ** -12, 2.0 ** -10, -2.0 ** -10, 1.5 * 2.0 ** -10])
    pool = np.concatenate([grid, -grid, mids, -mids, rand, tiny]).astype(np.float32)
    n = (-len(pool)) % 63
    pool = np.concatenate([pool, np.zeros(n, np.float32)])
    for blk in pool.reshape(-1, 63):
        x = np.concatenate([[448.0], blk]).astype(np.float32)  # amax 448: exponent 0
        out = oracle.fp8_quantize_block(x)
        assert out[0] == 127
        np.testing.assert_array_equal(np.frombuffer(out[1:], np.uint8), _torch_e4m3(x))


@pytest.mark.parametrize("amax,byte", [
    (448.0, 127),          # 448 / 2^0 = 448 <= 448
    (449.0, 128),          # needs 2^1
    (896.0, 128),          # 896 / 2 = 448 exactly
    (1.0, 119),            # 1 / 2^-8 = 256 <= 448, 1 / 2^-9 = 512 > 448
    (1.75, 119),           # 1.75 * 256 = 448
    (1.8, 120),
    (0.0, 127),            # an all-zero block keeps exponent 0
    (2.0 ** -140, 0),      # clamped at 2^-127
])
def test_fp8_block_exponent_is_the_smallest_that_fits_448(amax, byte):
    x = np.zeros(64, np.float32)
    x[7] = -amax
    x[9] = amax / 3
    out = oracle.fp8_quantize_block(x)
    assert out[0] == byte
    e = byte - 127
    scaled = (x.astype(np.float64) / 2.0 ** e).astype(np.float32)
    np.testing.assert_array_equal(np.frombuffer(out[1:], np.uint8), _torch_e4m3(scaled))


def test_fp8_round_trip_within_half_a_step():
    rng = np.random.default_rng(11)
    for scale in (1e-3, 1.0, 37.0, 1e5):
        x = (rng.standard_normal(64) * scale).astype(np.float32)
        out = oracle.fp8_quantize_block(x)
        s = 2.0 ** (out[0] - 127)
        dec = np.array([oracle.e4m3fn_to_double(c) for c in out[1:]]) * s
        # an E4M3 normal has 3 mantissa bits: half a step is 2^-4 of the value;
        # below 2^-6 the step is 2^-9 (absolute, before the block scale)
        bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s)
        assert np.all(np.abs(dec - x) <= bound * (1 + 1e-12))


# -------------------------------------------------------------------- pooling


def test_pool_equal_scores_give_the_mean():
    value = np.array([[1.0], [2.0], [3.0], [4.0]], np.float32)
    score = np.full((4, 1), 0.37, np.float32)
    out, ok = oracle.pool_candidates(value, score)
    assert ok and out[0] == 2.5


def test_pool_dominant_candidate_and_minus_inf_candidates():
    rng = np.random.default_rng(2)
    value = rng.standard_normal((8, 16)).astype(np.float32)
    score = np.zeros((8, 16), np.float32)
    dom = np.arange(16) % 8
    score[dom, np.arange(16)] = 120.0  # the others weigh e^-120: below half an ulp
    out, ok = oracle.pool_candidates(value, score)
    assert ok
    np.testing.assert_array_equal(out, value[dom, np.arange(16)])
    # -inf candidates are skipped entirely: a lone finite candidate is exact
    score = np.full((8, 16), -np.inf, np.float32)
    score[dom, np.arange(16)] = -3.0
    out, ok = oracle.pool_candidates(value, score)
    assert ok
    np.testing.assert_array_equal(out, value[dom, np.arange(16)])


@pytest.mark.parametrize("t", [0.25, 1.0, 3.5, 9.0])
def test_pool_two_candidates_follow_the_logistic_function(t):
    # values 1 and 0 at scores 0 and -t: pooled = 1 / (1 + e^-t)
    value = np.array([[1.0], [0.0]], np.float32)
    score = np.array([[0.0], [-t]], np.float32)
    out, ok = oracle.pool_candidates(value, score)
    assert ok
    assert abs(out[0] - 1.0 / (1.0 + math.exp(-t))) <= 2 * np.spacing(np.float32(1.0))


def test_pool_rejects_a_dimension_with_no_finite_score():
    value = np.ones((8, 2), np.float32)
    score = np.zeros((8, 2), np.float32)
    score[:, 1] = -np.inf
    _, ok = oracle.pool_candidates(value, score)
    assert not ok


def test_pool_weight_is_the_exponential():
    assert oracle.pool_weight(0.0) == 1.0
    for t in (-1e-3, -0.5, -5.0, -50.0, -100.0):
        w = oracle.pool_weight(t)
        assert abs(w - math.exp(t)) <= np.spacing(np.float32(math.exp(t)))


# -------------------------------------------------------------------- RoPE


def _yarn_freq(pair, n_rope):
    # the pages' compressed RoPE: base 160000, factor 16, linear ramp over pairs 15..25
    base = 160000.0 ** (-(2.0 * pair) / n_rope)
    ramp = min(1.0, max(0.0, (pair - 15.0) / 10.0))
    return base * (1 - ramp) + base / 16 * ramp


def test_rope_rotation_is_identity_at_position_zero():
    cs, sn = oracle.rope_rotation(0, 64)
    assert np.all(cs == 1.0) and np.all(sn == 0.0)


@pytest.mark.parametrize("position", [1, 3, 1000, 65531])
def test_rope_rotation_follows_the_ramped_frequencies(position):
    cs, sn = oracle.rope_rotation(position, 64)
    for p in range(32):
        ang = position * _yarn_freq(p, 64)
        # binary32 angle: rounding of the frequency and of the product
        tol = 4e-7 * position * _yarn_freq(p, 64) + 1e-6
        assert abs(cs[p] - math.cos(ang)) <= tol
        assert abs(sn[p] - math.sin(ang)) <= tol


# -------------------------------------------------------------------- finalize


def test_attention_record_of_a_constant_vector():
    # pooled all 3.0, norm all 1: RMSNorm gives 1 - O(1e-7) -> bf16 1.0; at
    # block_start 0 the RoPE leaves the tail; every FP8 block has amax 1, so
    # exponent -8 (byte 119) and code 0x78 (256 = 2^8); the tail is bf16 1.0
    rec, byts, ok = oracle.finalize_record(np.full(512, 3.0, np.float32), np.ones(512),
                                           n_rope=64, kind=oracle.COMPRESS_ATTN, block_start=0)
    assert ok and len(byts) == 583
    assert np.all(rec == 1.0)
    for blk in range(7):
        assert byts[blk * 65] == 119
        assert set(byts[blk * 65 + 1: blk * 65 + 65]) == {0x78}
    assert byts[455:] == bytes([0x80, 0x3F]) * 64
    # a negative constant with norm 2 gives -2 everywhere
    rec, _, ok = oracle.finalize_record(np.full(512, -0.75, np.float32), np.full(512, 2.0),
                                        n_rope=64, kind=oracle.COMPRESS_ATTN, block_start=0)
    assert ok and np.all(rec == -2.0)


def test_attention_record_rms_and_rope_rotation():
    rng = np.random.default_rng(4)
    pooled = rng.standard_normal(512).astype(np.float32) * 5
    norm = (1 + rng.standard_normal(512) * 0.1).astype(np.float32)
    rec0, _, ok = oracle.finalize_record(pooled, norm, n_rope=64, kind=oracle.COMPRESS_ATTN,
                                         block_start=0)
    assert ok
    # RMSNorm: (value / rms) * norm, rms over the bf16-rounded pooled values
    pb = np.array([oracle.round_bf16(v) for v in pooled], np.float64)
    want = pb / math.sqrt(np.mean(pb * pb) + 1e-6) * norm
    np.testing.assert_allclose(rec0[448:], want[448:], rtol=2 ** -7, atol=0)
    # FP8 part within the E4M3 step
    np.testing.assert_allclose(rec0[:448], want[:448], rtol=2 ** -3, atol=2 ** -8)
    # at block_start P the tail pairs are rotated by P * frequency
    P = 4096
    recP, _, ok = oracle.finalize_record(pooled, norm, n_rope=64, kind=oracle.COMPRESS_ATTN,
                                         block_start=P)
    assert ok
    for p in range(32):
        re, im = rec0[448 + 2 * p], rec0[449 + 2 * p]
        a = P * _yarn_freq(p, 64)
        wre = re * math.cos(a) - im * math.sin(a)
        wim = re * math.sin(a) + im * math.cos(a)
        tol = 2 ** -7 * (abs(re) + abs(im)) + 1e-3 * P * _yarn_freq(p, 64) * 1e-3
        assert abs(recP[448 + 2 * p] - wre) <= tol
        assert abs(recP[449 + 2 * p] - wim) <= tol


def test_index_key_of_a_one_hot_vector():
    # pooled = 2 e_0, norm 1: RMSNorm gives bf16(2 * 5.6568) = 11.3125 in dim 0;
    # the Hadamard row 0 spreads it: 11.3125 / sqrt(128) = 0.99989 -> bf16 1.0
    # everywhere; FP4 blocks of amax 1 take scale 2^-2 (byte 125) and code 4.0
    # (nibble 6) -> packed 0x66
    pooled = np.zeros(128, np.float32)
    pooled[0] = 2.0
    rec, byts, ok = oracle.finalize_record(pooled, np.ones(128), n_rope=64,
                                           kind=oracle.COMPRESS_INDEX, block_start=0)
    assert ok and len(byts) == 68
    assert np.all(rec == 1.0)
    for blk in range(4):
        assert byts[blk * 17] == 125
        assert byts[blk * 17 + 1: blk * 17 + 17] == bytes([0x66]) * 16


def test_finalize_flags_non_finite_records():
    pooled = np.ones(512, np.float32)
    pooled[3] = 3e38  # its square overflows the binary32 sum
    rec, byts, ok = oracle.finalize_record(pooled, np.ones(512), n_rope=64,
                                           kind=oracle.COMPRESS_ATTN, block_start=0)
    assert not ok and not any(byts) and not rec.any()
    norm = np.ones(512, np.float32)
    norm[5] = np.inf
    _, _, ok = oracle.finalize_record(np.ones(512, np.float32), norm, n_rope=64,
                                      kind=oracle.COMPRESS_ATTN, block_start=0)
    assert not ok


# -------------------------------------------------------------------- stream


def _block_records(case, inp):
    """Every record of positions [start, total) by the block formula: the
    candidates are gathered directly from the tokens (input or carry), not
    through the carry's slot mechanics."""
    kv = inp["kv"].numpy()
    score = (inp["gate"] + inp["ape"][torch.arange(case.start, case.total) % case.ratio]
             [None]).numpy()
    carry = inp["carry"].numpy()
    D, R = case.D, case.ratio
    out = {}
    for b in range(case.B):
        def token(p):
            """(value row, score row) of absolute position p (full source width)."""
            if p < 0:
                return np.zeros(case.W, np.float32), np.full(case.W, -np.inf, np.float32)
            if p >= case.start:
                return kv[b, p - case.start], score[b, p - case.start]
            # before this call: the carry's slot of that position
            open_from = case.start - case.start % R
            if R == 128:
                sl = p % 128
            elif p >= open_from:
                sl = 4 + p % 4
            else:
                sl = p % 4  # the previous (closed) block
            return carry[b, sl, 0], carry[b, sl, 1]

        for k in range(case.start // R, case.total // R):
            if (k + 1) * R - 1 < case.start:
                continue
            vals, scs = [], []
            if R == 128:
                for j in range(128):
                    v, s = token(k * 128 + j)
                    vals.append(v)
                    scs.append(s)
            else:
                for c in range(4):
                    v, s = token(4 * k - 4 + c)
                    vals.append(v[:D])
                    scs.append(s[:D])
                for c in range(4):
                    v, s = token(4 * k + c)
                    vals.append(v[D:])
                    scs.append(s[D:])
            pooled, ok = oracle.pool_candidates(np.stack(vals), np.stack(scs))
            assert ok
            out[(b, k)] = oracle.finalize_record(pooled, inp["norm"].numpy(),
                                                 n_rope=case.n_rope, kind=case.kind,
                                                 block_start=k * R)
    return out


@pytest.mark.parametrize("case", [
    synth.compress_r4(0, B=2, S=23, total=23),          # from position 0
    synth.compress_r4(0, B=2, S=22, total=61),          # open block at the start
    synth.compress_r4(1, B=2, S=30, total=45),
    synth.compress_r4(1, B=1, S=5, total=8),            # one closed block before
    synth.compress_r128(B=1, S=300, total=300, D=128),
    synth.compress_r128(B=2, S=200, total=460, D=128),  # open block at the start
], ids=lambda c: f"r{c.ratio}k{c.kind}S{c.S}T{c.total}")
def test_stream_records_follow_the_block_formula(case):
    inp = synth.make_compress_inputs(case, seed=3)
    recs, logi, _, bad = oracle.csa_compress(inp["kv"], inp["gate"], inp["ape"], inp["norm"],
                                             inp["carry"], ratio=case.ratio, kind=case.kind,
                                             n_rope=case.n_rope, total=case.total, rows=case.R)
    assert bad == 0
    want = _block_records(case, inp)
    assert want
    for (b, k), (rec, byts, ok) in want.items():
        assert ok
        np.testing.assert_array_equal(logi[b, k], rec)
        assert bytes(recs[b, k]) == byts
    # records before this call are untouched (still zero)
    first = min(k for _, k in want)
    assert not recs[:, :first].any()


@pytest.mark.parametrize("ratio,kind", [(4, 0), (4, 1), (128, 0)])
def test_stream_chunked_calls_equal_one_call(ratio, kind):
    D = 128 if (kind == 1 or ratio == 128) else 512
    total = 700 if ratio == 128 else 83
    case = synth.CompressCase("chunks", B=2, S=total, D=D, n_rope=64, ratio=ratio, kind=kind,
                              total=total)
    inp = synth.make_compress_inputs(case, seed=9)
    args = (inp["ape"], inp["norm"])
    one = oracle.csa_compress(inp["kv"], inp["gate"], *args, inp["carry"], ratio=ratio,
                              kind=kind, n_rope=64, total=total, rows=case.R)
    cuts = [0, 1, 6, 7, 40, 41, 300, total] if ratio == 128 else [0, 1, 6, 7, 40, 41, 63, total]
    recs, logi, carry = None, None, np.zeros_like(inp["carry"].numpy())
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        recs, logi, carry, bad = oracle.csa_compress(
            inp["kv"][:, lo:hi], inp["gate"][:, lo:hi], *args, carry, ratio=ratio, kind=kind,
            n_rope=64, total=hi, rows=case.R, records=recs, logical=logi)
        assert bad == 0
    np.testing.assert_array_equal(recs, one[0])
    np.testing.assert_array_equal(logi, one[1])
    np.testing.assert_array_equal(carry, one[2])


def test_stream_stores_invalid_records_as_zeros():
    case = synth.compress_r4(0, B=2, S=12, total=12)
    inp = synth.make_compress_inputs(case, seed=1)
    inp["kv"][1, 5, 700] = float("nan")  # token 5, second half: record 1 of batch 1
    recs, logi, _, bad = oracle.csa_compress(inp["kv"], inp["gate"], inp["ape"], inp["norm"],
                                             inp["carry"], ratio=4, kind=0, n_rope=64,
                                             total=12, rows=3)
    assert bad == 1
    assert not recs[1, 1].any() and not logi[1, 1].any()
    assert recs[1, 0].any() and recs[1, 2].any() and recs[0].all(axis=1).any()
