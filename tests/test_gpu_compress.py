"""GPU parity of the CSA compression stages (onnx-runtime-ep-cpu
compressed_sparse_attention.rs compress_ratio4_stream / pool_ratio*_record /
finalize_attention_record / finalize_index_record; onnx-runtime-ep-cuda
csa_ratio128_compress, csa_ratio4_main_compress, csa_ratio4_index_compress)
against the oracle, through the C ABI.  The records are bytes that the pages
fix in binary32, so records, their dequantized values and the carry must
match bit for bit.  Cases span several records with ragged block edges at
both ends of a call, a stream starting at position 0, decode-sized calls,
chained calls, invalid records, extreme scores (the pool weight's subnormal
range and its double fallback), large positions (large RoPE angles), and
the full chunk the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"

_FN = {(4, 0): "csa_ratio4_main_compress", (4, 1): "csa_ratio4_index_compress",
       (128, 0): "csa_ratio128_compress"}


def _gpu(sa, c, inp, *, records=None, logical=None, carry=None, want=("records", "logical")):
    d = {k: v.to(DEV) for k, v in inp.items()}
    cy = (carry if carry is not None else inp["carry"]).to(DEV).clone()
    rec = None
    if "records" in want:
        rec = (records.to(DEV).clone() if records is not None
               else torch.zeros((c.B, c.R, c.width), dtype=torch.uint8, device=DEV))
    lg = None
    if "logical" in want:
        lg = (logical.to(DEV).clone() if logical is not None
              else torch.zeros((c.B, c.R, c.D), dtype=torch.float32, device=DEV))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    getattr(sa, _FN[(c.ratio, c.kind)])(d["kv"], d["gate"], d["ape"], d["norm"], cy,
                                        n_rope=c.n_rope, total=c.total, records=rec, logical=lg,
                                        err_word=err)
    torch.cuda.synchronize()
    return (None if rec is None else rec.cpu().numpy(), None if lg is None else lg.cpu().numpy(),
            cy.cpu().numpy(), int(err.item()))


def _ref(c, inp, *, records=None, logical=None, carry=None):
    return oracle.csa_compress(inp["kv"], inp["gate"], inp["ape"], inp["norm"],
                               inp["carry"] if carry is None else carry, ratio=c.ratio,
                               kind=c.kind, n_rope=c.n_rope, total=c.total, rows=c.R,
                               records=records, logical=logical)


def _same(got, ref, what):
    g_rec, g_log, g_cy, g_err = got
    r_rec, r_log, r_cy, r_bad = ref
    if g_rec is not None:
        bad = np.argwhere((g_rec != r_rec).any(axis=2))
        assert bad.size == 0, f"{what}: records differ at (b, k) {bad[:8].tolist()}"
    if g_log is not None:
        diff = g_log.view(np.uint32) != r_log.view(np.uint32)
        assert not diff.any(), f"{what}: logical differs at {np.argwhere(diff)[:8].tolist()}"
    assert np.array_equal(g_cy.view(np.uint32), r_cy.view(np.uint32)), f"{what}: carry differs"
    assert (g_err != 0) == (r_bad != 0), f"{what}: error bit {g_err} vs {r_bad} invalid records"


CASES = [
    # ratio 4 attention records (D 512 = 448 FP8 + 64 bf16 RoPE)
    ("r4_attn_from_zero", synth.compress_r4(0, B=3, S=37, total=37)),
    ("r4_attn_open_block", synth.compress_r4(0, B=3, S=37, total=102)),
    ("r4_attn_decode_close", synth.compress_r4(0, B=5, S=1, total=64)),
    ("r4_attn_decode_open", synth.compress_r4(0, B=5, S=1, total=66)),
    ("r4_attn_long", synth.compress_r4(0, B=9, S=301, total=1003)),
    ("r4_attn_d192_rope0", synth.compress_r4(0, B=2, S=21, total=50, D=192, n_rope=0)),
    ("r4_attn_d576_rope128", synth.compress_r4(0, B=2, S=40, total=90, D=576, n_rope=128)),
    # ratio 4 index keys (D 128, 64 RoPE, FP4)
    ("r4_index_from_zero", synth.compress_r4(1, B=3, S=37, total=37)),
    ("r4_index_open_block", synth.compress_r4(1, B=9, S=50, total=103)),
    ("r4_index_decode_close", synth.compress_r4(1, B=5, S=1, total=68)),
    ("r4_index_d256", synth.compress_r4(1, B=2, S=30, total=61, D=256)),
    ("r4_index_d32", synth.compress_r4(1, B=2, S=30, total=61, D=32, n_rope=16)),
    # ratio 128 (D 512)
    ("r128_from_zero", synth.compress_r128(B=2, S=300, total=300)),
    ("r128_open_block", synth.compress_r128(B=3, S=200, total=460)),
    ("r128_decode_close", synth.compress_r128(B=4, S=1, total=256)),
    ("r128_decode_open", synth.compress_r128(B=4, S=1, total=250)),
    ("r128_d128", synth.compress_r128(B=2, S=260, total=300, D=128, n_rope=64)),
]


@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_compress_matches_oracle(cuda_lib, name, case):
    inp = synth.make_compress_inputs(case, seed=17)
    _same(_gpu(cuda_lib, case, inp), _ref(case, inp), name)


def test_compress_one_output_at_a_time(cuda_lib):
    c = synth.compress_r4(0, B=2, S=33, total=70)
    inp = synth.make_compress_inputs(c, seed=5)
    ref = _ref(c, inp)
    rec, _, cy, _ = _gpu(cuda_lib, c, inp, want=("records",))
    _same((rec, None, cy, 0), ref, "records only")
    _, lg, cy, _ = _gpu(cuda_lib, c, inp, want=("logical",))
    _same((None, lg, cy, 0), ref, "logical only")


@pytest.mark.parametrize("ratio,kind", [(4, 0), (4, 1), (128, 0)])
def test_compress_chained_calls_match_one_oracle_stream(cuda_lib, ratio, kind):
    D = 512 if kind == 0 else 128
    total = 700 if ratio == 128 else 150
    full = synth.CompressCase("chain", B=3, S=total, D=D, n_rope=64, ratio=ratio, kind=kind,
                              total=total)
    inp = synth.make_compress_inputs(full, seed=23)
    ref = _ref(full, inp)
    cuts = ([0, 1, 2, 127, 128, 129, 300, 511, 512, 699, total] if ratio == 128
            else [0, 1, 2, 3, 4, 5, 9, 40, 41, 42, 43, 44, 120, total])
    rec = torch.zeros((full.B, full.R, full.width), dtype=torch.uint8)
    lg = torch.zeros((full.B, full.R, full.D), dtype=torch.float32)
    cy = torch.zeros_like(inp["carry"])
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        c = synth.CompressCase("chain", B=3, S=hi - lo, D=D, n_rope=64, ratio=ratio, kind=kind,
                               total=hi, rows=full.R)
        part = {"kv": inp["kv"][:, lo:hi].contiguous(), "gate": inp["gate"][:, lo:hi].contiguous(),
                "ape": inp["ape"], "norm": inp["norm"], "carry": cy}
        r, l_, cyn, err = _gpu(cuda_lib, c, part, records=rec, logical=lg, carry=cy)
        assert err == 0
        rec, lg, cy = torch.from_numpy(r), torch.from_numpy(l_), torch.from_numpy(cyn)
    _same((rec.numpy(), lg.numpy(), cy.numpy(), 0), ref, f"chained r{ratio} k{kind}")


@pytest.mark.parametrize("ratio,kind", [(4, 0), (4, 1), (128, 0)])
def test_compress_invalid_records_are_zero_and_flagged(cuda_lib, ratio, kind):
    c = (synth.compress_r128(B=2, S=300, total=300, D=128) if ratio == 128
         else synth.compress_r4(kind, B=2, S=30, total=30))
    inp = synth.make_compress_inputs(c, seed=2)
    inp["kv"][1, 9, 5] = float("nan")
    ref = _ref(c, inp)
    assert ref[3] >= 1
    got = _gpu(cuda_lib, c, inp)
    assert got[3] & cuda_lib.ERRBIT_COMPRESS
    _same(got, ref, "nan input")
    # a dimension with no finite score: gate -inf on every candidate of a record
    inp = synth.make_compress_inputs(c, seed=3)
    if ratio == 4:
        inp["gate"][0, 4:8, c.D + 3] = float("-inf")   # record 1's current half
        inp["gate"][0, 0:4, 3] = float("-inf")         # and its previous half
    else:
        inp["gate"][0, 128:256, 3] = float("-inf")
    ref = _ref(c, inp)
    assert ref[3] >= 1
    _same(_gpu(cuda_lib, c, inp), ref, "no finite score")


@pytest.mark.parametrize("ratio,kind", [(4, 0), (4, 1), (128, 0)])
def test_compress_extreme_scores(cuda_lib, ratio, kind):
    # score gaps of 80..110 put pool weights in the subnormal range and below
    c = (synth.compress_r128(B=2, S=256, total=256, D=128) if ratio == 128
         else synth.compress_r4(kind, B=3, S=64, total=64))
    inp = synth.make_compress_inputs(c, seed=8)
    g = torch.Generator().manual_seed(4)
    inp["gate"] = inp["gate"] * 40.0 + torch.randint(-2, 3, inp["gate"].shape, generator=g) * 45.0
    _same(_gpu(cuda_lib, c, inp), _ref(c, inp), "extreme scores")


@pytest.mark.parametrize("ratio,kind", [(4, 0), (4, 1), (128, 0)])
def test_compress_large_positions(cuda_lib, ratio, kind):
    total = (1 << 22) + 77 if ratio == 4 else (1 << 22) + 300
    S = 45 if ratio == 4 else 300
    c = synth.CompressCase("far", B=2, S=S, D=512 if kind == 0 else 128, n_rope=64, ratio=ratio,
                           kind=kind, total=total, rows=total // ratio)
    inp = synth.make_compress_inputs(c, seed=12)
    k0 = (total - S) // ratio
    got = _gpu(cuda_lib, c, inp)
    ref = _ref(c, inp)
    # compare the rows this call wrote (the rest are zero on both sides)
    sl = slice(k0, None)
    _same((got[0][:, sl], got[1][:, sl], got[2], got[3]),
          (ref[0][:, sl], ref[1][:, sl], ref[2], ref[3]), "large positions")


def test_pool_weight_is_correctly_rounded_on_every_binary32_input(cuda_lib):
    """Every binary32 t in [-104, 0] (about 1.1e9 values, in chunks) and a set
    of special values: the kernel's e^t against torch's double exponential
    rounded to binary32, bit for bit; and a random sample against the
    oracle's."""
    lo = np.array(-104.0, np.float32).view(np.uint32).item()
    top = 0x80000000
    chunk = 1 << 27
    mism = 0
    for start in range(top, lo + 1, chunk):
        n = min(chunk, lo + 1 - start)
        bits = torch.arange(start, start + n, dtype=torch.int64, device=DEV)
        t = (bits - (1 << 32)).to(torch.int32).view(torch.float32)
        w = cuda_lib.csa_pool_weight(t)
        want = torch.exp(t.double()).float()
        mism += int((w.view(torch.int32) != want.view(torch.int32)).sum().item())
        del bits, t, w, want
    assert mism == 0, f"{mism} inputs differ from the rounded double exponential"
    special = torch.tensor([0.0, -0.0, float("nan"), float("-inf"), 1.0, 10.0, 88.0, -87.0,
                            -87.3, -103.97, -103.98, -1e-30, -1e-7], device=DEV)
    w = cuda_lib.csa_pool_weight(special)
    want = torch.exp(special.double()).float()
    np.testing.assert_array_equal(w.cpu().numpy(), want.cpu().numpy())
    rng = np.random.default_rng(3)
    sample = np.concatenate([-rng.exponential(3.0, 20000), rng.uniform(-104, 0, 20000)])
    sample = sample.astype(np.float32)
    w = cuda_lib.csa_pool_weight(torch.from_numpy(sample).to(DEV)).cpu().numpy()
    want = np.array([oracle.pool_weight(float(x)) for x in sample], np.float32)
    np.testing.assert_array_equal(w.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("ratio,kind", [(4, 0), (4, 1), (128, 0)])
def test_compress_full_chunk_matches_oracle(cuda_lib, ratio, kind):
    """The benchmark's chunk (B 16, 4,096 tokens ending at 65,536), in the
    launch configuration it times: every record, the dequantized values and
    the carry."""
    c = synth.compress_r128() if ratio == 128 else synth.compress_r4(kind)
    inp = synth.make_compress_inputs(c, seed=1001)
    got = _gpu(cuda_lib, c, inp)
    ref = _ref(c, inp)
    k0 = c.start // c.ratio
    sl = slice(k0, None)
    _same((got[0][:, sl], got[1][:, sl], got[2], got[3]),
          (ref[0][:, sl], ref[1][:, sl], ref[2], ref[3]), "full chunk")
