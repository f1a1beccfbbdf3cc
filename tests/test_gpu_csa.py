"""GPU parity of compressed sparse attention (ratio 4) in the pages' own form
(onnx-runtime-ep-cpu compressed_sparse_attention.rs ratio4_attention;
onnx-runtime-ep-cuda csa_ratio4_sink_attention) against the fp64 oracle,
through the C ABI.  The op reads hybrid FP8 records, so its outputs are held
to the FP8/bf16 tolerance (2e-2 of the largest output magnitude)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL_REL_LOW

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _close(y, ref, what):
    got = y.detach().float().cpu().double().numpy()
    assert np.isfinite(got).all(), what
    tol = TOL_REL_LOW * float(np.abs(ref).max())
    err = float(np.abs(got - ref).max())
    assert err <= tol, f"{what}: max|got - oracle| = {err:.3e} > {tol:.3e}"


def _run(sa, c, inp, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkw = {n: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for n, t in kw.items()}
    y = sa.csa_ratio4_attention(inp["query"].to(DEV), inp["window"].to(DEV),
                                inp["records"].to(DEV), inp["selected"].to(DEV), total=c.total,
                                n_rope=c.n_rope, err_word=err, **gkw)
    torch.cuda.synchronize()
    return y, int(err.item())


def _ref(c, inp, **kw):
    okw = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in kw.items()}
    if "sink" in okw and okw["sink"] is not None:
        okw["sink"] = okw["sink"].double()
    return oracle.csa_ratio4_attention(inp["query"], inp["window"], inp["records"],
                                       inp["selected"], total=c.total, n_rope=c.n_rope, **okw)


CASES = [
    ("d512_mid", dict(B=2, S=1, H=64, D=512, n_rope=64, L=128, total=3000, topk=300)),
    ("d512_multi_query", dict(B=2, S=3, H=32, D=512, n_rope=64, L=128, total=2048, topk=100)),
    ("d512_short_window", dict(B=3, S=2, H=32, D=512, n_rope=64, L=40, total=900, topk=64)),
    ("d512_block_at_zero", dict(B=1, S=50, H=32, D=512, n_rope=64, L=50, total=50, topk=12)),
    ("d128", dict(B=2, S=2, H=32, D=128, n_rope=64, L=128, total=1500, topk=200)),
    ("d128_no_rope", dict(B=2, S=1, H=64, D=128, n_rope=0, L=100, total=800, topk=90)),
]


# 128-head blocks with bf16 queries run on the tcgen05 kernel (128-slot tiles,
# two CTAs per head block, key splits merged by the combine kernel); the
# f32 versions of the same shapes run on the warp-level MMA kernel.
CASES_TC = [
    ("tc_mid", dict(B=2, S=1, H=128, D=512, n_rope=64, L=128, total=3000, topk=300)),
    ("tc_multi_query", dict(B=2, S=3, H=128, D=512, n_rope=64, L=128, total=2048, topk=100)),
    ("tc_short_window_h256", dict(B=3, S=2, H=256, D=512, n_rope=64, L=40, total=900, topk=64)),
    ("tc_block_at_zero", dict(B=1, S=50, H=128, D=512, n_rope=64, L=50, total=50, topk=12)),
    ("tc_long_16_splits", dict(B=1, S=1, H=128, D=512, n_rope=64, L=128, total=40000,
                               topk=6000)),
    ("tc_one_tile", dict(B=2, S=20, H=128, D=512, n_rope=64, L=20, total=20, topk=4)),
]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("name,over", CASES + CASES_TC, ids=[c[0] for c in CASES + CASES_TC])
def test_csa_matches_oracle(cuda_lib, dt, name, over):
    c = synth.CsaCase(name, dtype=dt, **over)
    inp = synth.make_csa_inputs(c, seed=41)
    sink = torch.linspace(-1.0, 1.5, c.H, dtype=torch.float32)
    y, err = _run(cuda_lib, c, inp, sink=sink)
    ref, bad = _ref(c, inp, sink=sink)
    assert err == 0 and bad == 0
    _close(y, ref, f"{name} {dt}")


@pytest.mark.parametrize("H", [32, 128, 384])
@pytest.mark.parametrize("shape_kind", ["h1c", "b11c", "c", "full"])
def test_slot_bias(cuda_lib, shape_kind, H):
    c = synth.CsaCase("bias", B=2, S=2, H=H, D=512, n_rope=64, L=128, total=1200, topk=80)
    inp = synth.make_csa_inputs(c, seed=42)
    C = 128 + c.topk
    shape = {"h1c": (c.H, 1, C), "b11c": (c.B, 1, 1, C), "c": (C,),
             "full": (c.B, c.H, c.S, C)}[shape_kind]
    g = torch.Generator().manual_seed(43)
    bias = torch.randn(shape, generator=g) * 2.0
    bias.view(-1)[::17] = -float("inf")
    y, _ = _run(cuda_lib, c, inp, bias=bias)
    ref, _ = _ref(c, inp, bias=bias)
    _close(y, ref, f"bias {shape_kind}")


@pytest.mark.parametrize("H", [32, 128])
def test_invalid_records_are_skipped_and_flagged(cuda_lib, H):
    c = synth.CsaCase("bad", B=2, S=1, H=H, D=512, n_rope=64, L=128, total=1000, topk=40)
    inp = synth.make_csa_inputs(c, seed=44)
    sel = inp["selected"].clone()
    sel[0, 0, 5] = 250          # 250 >= 1000 / 4: skipped, flagged
    sel[1, 0, :10] = -1         # padding anywhere: no candidate
    inp = dict(inp, selected=sel)
    y, err = _run(cuda_lib, c, inp)
    ref, bad = _ref(c, inp)
    assert bad == 1 and err == cuda_lib.ERRBIT_RECORD
    _close(y, ref, "bad records")


@pytest.mark.parametrize("H", [64, 128])
def test_deterministic(cuda_lib, H):
    c = synth.CsaCase("det", B=2, S=1, H=H, D=512, n_rope=64, L=128, total=4000, topk=500)
    inp = synth.make_csa_inputs(c, seed=45, device=DEV)
    ys = [_run(cuda_lib, c, inp)[0] for _ in range(2)]
    assert torch.equal(ys[0], ys[1])


def test_full_size_csa_sampled_rows(cuda_lib):
    """B16 H128 D512 (583-byte records) L128 total 65,536 top-k 2,048: the
    benchmark's launch configuration, checked on sampled batches."""
    c = synth.csa_ratio4_ref()
    inp = synth.make_csa_inputs(c, seed=1, device=DEV)
    sink = torch.linspace(-1.0, 1.0, c.H, dtype=torch.float32, device=DEV)
    y, err = _run(cuda_lib, c, inp, sink=sink)
    assert err == 0
    for b in (0, 9):
        sub = {k: v[b:b + 1].cpu() for k, v in inp.items()}
        cb = synth.CsaCase("sub", B=1, S=c.S, H=c.H, D=c.D, n_rope=c.n_rope, L=c.L,
                           total=c.total, topk=c.topk)
        ref, _ = _ref(cb, sub, sink=sink)
        _close(y[b:b + 1], ref, f"full b={b}")
