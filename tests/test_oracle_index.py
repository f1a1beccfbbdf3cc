"""Pins for the oracle's ratio-4 index scoring and top-k selection, against
facts fixed outside the oracle: the OCP MX E2M1 table, hand-worked FP4
blocks, the Sylvester Hadamard matrix (scipy) with torch's bfloat16
rounding, float64 scores from an independent decode, numpy's stable sort,
and a hand-worked selection.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


# E2M1 magnitudes by code, for an independent numpy decode of index records
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def np_decode_records(rec, ID):
    """[..., stride] uint8 -> [..., ID] float64, written here from the record
    layout (blocks of [E8M0 scale, 16 bytes, low nibble first])."""
    rec = np.asarray(rec)
    nb = ID // 32
    blocks = rec[..., : nb * 17].reshape(*rec.shape[:-1], nb, 17)
    scale = np.exp2(blocks[..., 0].astype(np.float64) - 127.0)
    codes = np.stack([blocks[..., 1:] & 15, blocks[..., 1:] >> 4], axis=-1).reshape(
        *rec.shape[:-1], nb, 32)
    vals = _E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    return (vals * scale[..., None]).reshape(*rec.shape[:-1], ID)


def test_e2m1_codes_match_the_ocp_table():
    rows = _golden("e2m1_codes.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_to_double(int(code, 16))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_bf16_rounding_matches_torch_on_every_kind_of_value():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-140, 120, (20000,),
                                                                 generator=g).float())
    # exact ties (low half 0x8000) with even and odd neighbours, subnormals, specials
    ties = torch.from_numpy(np.array([0x3f808000, 0x3f818000, 0x00018000, 0x80028000,
                                      0x7f7f8000], dtype=np.uint32).view(np.float32))
    special = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), 1e-45, -3e-39])
    x = torch.cat([x, ties, special])
    ref = x.to(torch.bfloat16).to(torch.float32)
    got = torch.tensor([oracle.round_bf16(float(v)) for v in x], dtype=torch.float32)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    assert math.isnan(oracle.round_bf16(float("nan")))


def test_fp4_blocks_golden():
    for name, byte, inputs, expected in _golden("fp4_blocks.txt"):
        xs = [float(v) for v in inputs.split(",")]
        ex = [float(v) for v in expected.split(",")]
        block = np.zeros(32, dtype=np.float32)
        block[: len(xs)] = xs
        sb, packed, vals = oracle.fp4_quantize_block(block)
        assert sb == int(byte), name
        assert np.array_equal(vals[: len(ex)], np.array(ex, dtype=np.float32)), name
        assert not vals[len(ex):].any(), name


def test_fp4_round_trip_error_is_within_the_mx_step():
    g = torch.Generator().manual_seed(7)
    for t in range(300):
        x = (torch.randn(32, generator=g) * 10.0 ** float(torch.randint(-6, 6, (1,),
                                                                         generator=g))).numpy()
        sb, packed, vals = oracle.fp4_quantize_block(x)
        amax = np.abs(x).max()
        X = 2.0 ** (math.floor(math.log2(amax)) - 2)
        assert sb == math.floor(math.log2(amax)) - 2 + 127
        v = x.astype(np.float64) / X
        assert np.abs(v).max() >= 4.0 and np.abs(v).max() < 8.0
        err = np.abs(vals.astype(np.float64) - x.astype(np.float64))
        # spacing of E2M1 is at most 2 between neighbours below 6: error <= X;
        # values beyond 6 saturate: error < 2 X
        lim = np.where(np.abs(v) <= 6.0, X, 2.0 * X)
        assert (err <= lim + 1e-30).all()
        # decoded independently from the packed bytes
        rec = np.frombuffer(bytes([sb]) + packed, dtype=np.uint8)
        assert np.array_equal(np_decode_records(rec, 32), vals.astype(np.float64))


def test_hadamard_golden_width_four():
    # butterflies on (1, 2, 3, 4): span 1 -> (3, -1, 7, -1), span 2 ->
    # (10, -2, -4, 0), times 1/sqrt(4) -> (5, -1, -2, 0), exact in bfloat16
    assert np.array_equal(oracle.hadamard_bf16([1, 2, 3, 4]),
                          np.array([5, -1, -2, 0], dtype=np.float32))


@pytest.mark.parametrize("n", [32, 64, 128])
def test_hadamard_matches_the_sylvester_matrix(n):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(n)
    g = torch.Generator().manual_seed(n)
    for t in range(20):
        x = torch.randint(-50, 51, (n,), generator=g).numpy().astype(np.float32)
        exact = (H @ x.astype(np.int64)).astype(np.float32)  # integers: exact in f32
        scaled = exact * (np.float32(1.0) / np.sqrt(np.float32(n)))
        ref = torch.from_numpy(scaled).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(oracle.hadamard_bf16(x), ref)


def test_query_finalize_is_bf16_then_hadamard_then_fp4_round_trip():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(128, generator=g).numpy().astype(np.float32)
    out = oracle.index_query_finalize(x)
    # the steps one after another, each pinned above
    h = oracle.hadamard_bf16(torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    for b in range(4):
        _, _, vals = oracle.fp4_quantize_block(h[32 * b: 32 * b + 32])
        assert np.array_equal(out[32 * b: 32 * b + 32], vals)


def test_selection_golden():
    ID = 32
    q = np.zeros((1, 1, 1, ID), dtype=np.float32)
    q[0, 0, 0, 0] = 8.0
    w = np.ones((1, 1, 1), dtype=np.float32)
    keys = np.zeros((1, 5, 17), dtype=np.uint8)
    keys[:, :, 0] = 127

    def put(r, i, code):
        keys[0, r, 1 + i // 2] |= code << (4 * (i % 2))

    put(0, 3, 0x4)            # 2.0
    put(1, 7, 0x1)            # 0.5
    put(2, 0, 0x2)            # 1.0
    put(2, 9, 0x1)            # 0.5
    put(3, 5, 0xA)            # -1.0
    keys[0, 4] = keys[0, 2]
    assert np.array_equal(oracle.index_query_finalize(q[0, 0, 0]), np.full(ID, 1.5, np.float32))
    for pos, topk, exp, tie in _golden("index_topk_small.txt"):
        sel, st, err = oracle.index_select(q, w, keys, topk=int(topk), query_start=int(pos))
        assert sel[0, 0, 0].tolist() == [int(v) for v in exp.split(",")], (pos, topk)
        assert int(st[0]) == int(tie) * oracle.SEL_TIE and err == int(st[0])


def _small(seed, **over):
    kw = dict(B=3, S=2, IH=8, ID=128, R=300, topk=64, query_start=1000)
    kw.update(over)
    c = synth.IndexCase("t", **kw)
    return c, synth.make_index_inputs(c, seed)


def test_scores_match_float64_from_an_independent_decode():
    c, inp = _small(11)
    sel, st, err, scores = oracle.index_select(inp["query"], inp["weight"], inp["keys"],
                                               topk=c.topk, query_start=c.query_start,
                                               want_scores=True)
    keys = np_decode_records(inp["keys"].numpy(), c.ID)
    cst = 1.0 / math.sqrt(c.ID) / math.sqrt(c.IH)
    for b in range(c.B):
        for s in range(c.S):
            limit = min(c.R, (c.query_start + s + 1) // 4)
            qf = np.stack([oracle.index_query_finalize(inp["query"][b, s, h].numpy())
                           for h in range(c.IH)]).astype(np.float64)
            dots = keys[b, :limit] @ qf.T                       # [limit, IH]
            ref = (np.maximum(dots, 0.0) * inp["weight"][b, s].double().numpy()).sum(1) * cst
            got = scores[b, s, :limit].astype(np.float64)
            scale = (np.abs(np.maximum(dots, 0.0) * inp["weight"][b, s].double().numpy())
                     .sum(1) * cst)
            assert (np.abs(got - ref) <= 1e-5 * scale + 1e-30).all()
            assert not scores[b, s, limit:].any()


def test_selection_equals_a_stable_sort_of_the_scores():
    c, inp = _small(12, R=2000, topk=700, query_start=5000)
    for ascending in (False, True):
        sel, st, err, scores = oracle.index_select(inp["query"], inp["weight"], inp["keys"],
                                                   topk=c.topk, query_start=c.query_start,
                                                   out_heads=3, ascending=ascending,
                                                   want_scores=True)
        for b in range(c.B):
            for s in range(c.S):
                limit = min(c.R, (c.query_start + s + 1) // 4)
                sc = scores[b, s, :limit].astype(np.float64)
                order = np.argsort(-sc, kind="stable")[: c.topk]  # ties keep the lower record
                exp = np.full(c.topk, -1)
                exp[: len(order)] = np.sort(order) if ascending else order
                for o in range(3):
                    assert np.array_equal(sel[b, o, s], exp)
                tie = len(np.unique(sc)) < limit
                assert bool(st[b * c.S + s] & oracle.SEL_TIE) == tie


def test_causal_limit_padding_and_per_batch_positions():
    c, inp = _small(13, B=2, S=3, R=50, topk=40, query_start=0)
    starts = torch.tensor([100, 29], dtype=torch.int64)   # batch 1: positions 29, 30, 31
    sel, st, err = oracle.index_select(inp["query"], inp["weight"], inp["keys"], topk=c.topk,
                                       query_start_b=starts)
    for s, limit in enumerate([7, 7, 8]):                  # (29+1)//4, (30+1)//4, (31+1)//4
        row = sel[1, 0, s]
        assert (row[:limit] >= 0).all() and (row[limit:] == -1).all()
        assert sorted(row[:limit].tolist()) == list(range(limit))
    # batch 0: positions 100..102, (p + 1) // 4 = 25 records: 25 filled, 15 of -1
    assert (sel[0, 0, :, :25] >= 0).all() and (sel[0, 0, :, 25:] == -1).all()
