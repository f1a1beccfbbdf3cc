"""Pins for the oracle's compressed sparse attention (ratio 4) in the pages'
own form: a hand-worked example, and masked brute force in matrix form with
an independent record decode (torch's E4M3) and window logic written here.
CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_two_candidates():
    with open(os.path.join(GOLDEN, "csa_two_candidate.txt")) as f:
        rows = {l.split()[0]: (float(l.split()[1]), float(l.split()[2]))
                for l in f if l.strip() and not l.startswith("#")}
    ln3 = float(np.float32(math.log(3.0)))
    ln2 = float(np.float32(math.log(2.0)))
    q = torch.zeros((1, 1, 1, 64), dtype=torch.float32)
    q[0, 0, 0, 0] = ln3
    w = torch.zeros((1, 1, 64), dtype=torch.float32)
    w[0, 0, 0] = 1.0
    rec = torch.zeros((1, 2, 65), dtype=torch.uint8)
    rec[:, :, 0] = 127
    rec[0, 0, 1 + 1] = 0x40  # dim 1 = 2.0
    sel = torch.tensor([[[0]]], dtype=torch.int32)
    kw = dict(total=8, n_rope=0, scale=1.0)
    # position 7 > 0: 128 dense slots precede the record's slot 128
    slot_bias = torch.zeros(129)
    slot_bias[128] = ln2
    got = {
        "sink": oracle.csa_ratio4_attention(q, w, rec, sel, sink=[0.0], **kw)[0],
        "sink_bias": oracle.csa_ratio4_attention(q, w, rec, sel, sink=[0.0],
                                                 bias=slot_bias, **kw)[0],
        "nosink": oracle.csa_ratio4_attention(q, w, rec, sel, **kw)[0],
    }
    for name, y in got.items():
        assert np.allclose(y[0, 0, 0, :2], rows[name], rtol=0, atol=1e-6), (name, y[0, 0, 0, :2])
        assert not y[0, 0, 0, 2:].any()


def _decode_torch(rec, D, n_rope):
    """Records -> float64 rows via torch's E4M3 decode (independent of the oracle)."""
    nb = (D - n_rope) // 64
    blocks = rec[..., : nb * 65].reshape(*rec.shape[:-1], nb, 65)
    codes = blocks[..., 1:].contiguous().view(torch.float8_e4m3fn).double()
    scale = torch.exp2(blocks[..., 0].double() - 127.0)
    nope = (codes * scale[..., None]).reshape(*rec.shape[:-1], nb * 64)
    tail = rec[..., nb * 65: nb * 65 + 2 * n_rope].to(torch.int32)
    bits = (tail[..., 0::2] | (tail[..., 1::2] << 8)).to(torch.int16)
    rope = bits.view(torch.bfloat16).double()
    return torch.cat([nope, rope], dim=-1).numpy()


@pytest.mark.parametrize("case", ["mid", "start", "short_window", "bias"])
def test_matches_brute_force(case):
    over = {"mid": dict(total=600, L=128, S=3), "start": dict(total=40, L=40, S=40),
            "short_window": dict(total=900, L=50, S=2), "bias": dict(total=700, L=128, S=2)}[case]
    c = synth.CsaCase("t", B=2, H=4, D=128, n_rope=64, topk=30, dtype="f32", **over)
    inp = synth.make_csa_inputs(c, seed=7)
    dense = min(c.L, 128) if c.total - c.S == 0 else 128
    C = dense + c.topk
    bias = None
    full = None
    if case == "bias":
        g = torch.Generator().manual_seed(8)
        bias = torch.randn((c.H, 1, C), generator=g)
        full = np.broadcast_to(bias.double().numpy(), (c.B, c.H, c.S, C))
    sink = [0.3 * h - 0.5 for h in range(c.H)]
    y, bad = oracle.csa_ratio4_attention(inp["query"], inp["window"], inp["records"],
                                         inp["selected"], total=c.total, n_rope=c.n_rope,
                                         sink=sink, bias=bias)
    assert bad == 0
    dec = _decode_torch(inp["records"], c.D, c.n_rope)
    qs, ws = inp["query"].double().numpy(), inp["window"].double().numpy()
    base = c.total - c.L
    scale = 1.0 / math.sqrt(c.D)
    for b in range(c.B):
        for s in range(c.S):
            p = c.total - c.S + s
            start = max(base, max(0, p - 127))
            keys, slots = [], []
            for cnd in range(dense):          # window candidates (positions start + cnd)
                t = start + cnd
                if t <= p and t - base < c.L:
                    keys.append(ws[b, t - base])
                    slots.append(cnd)
            for k in range(c.topk):
                r = int(inp["selected"][b, s, k])
                if r >= 0:
                    keys.append(dec[b, r])
                    slots.append(dense + k)
            K = np.stack(keys)
            for h in range(c.H):
                sc = K @ qs[b, s, h] * scale
                if full is not None:
                    sc = sc + full[b, h, s, slots]
                m = sc.max()
                w = np.exp(sc - m)
                exp = (w @ K) / (w.sum() + math.exp(sink[h] - m))
                assert np.allclose(y[b, s, h], exp, rtol=1e-12, atol=1e-12)


def test_out_of_range_records_are_skipped_and_flagged():
    c = synth.CsaCase("t", B=1, S=1, H=2, D=64, n_rope=0, L=8, total=100, topk=6, dtype="f32")
    inp = synth.make_csa_inputs(c, seed=9)
    sel = inp["selected"].clone()
    y0, _ = oracle.csa_ratio4_attention(inp["query"], inp["window"], inp["records"], sel,
                                        total=c.total, n_rope=0)
    sel2 = sel.clone()
    sel2[0, 0, 5] = 25            # 25 >= 100 / 4: skipped, flagged
    sel3 = sel.clone()
    sel3[0, 0, 5] = -1
    y2, bad2 = oracle.csa_ratio4_attention(inp["query"], inp["window"], inp["records"], sel2,
                                           total=c.total, n_rope=0)
    y3, bad3 = oracle.csa_ratio4_attention(inp["query"], inp["window"], inp["records"], sel3,
                                           total=c.total, n_rope=0)
    assert bad2 == 1 and bad3 == 0
    assert np.array_equal(y2, y3) and not np.array_equal(y2, y0)
