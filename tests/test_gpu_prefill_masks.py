"""GPU parity of dense prefill with the ONNX Attention padding frontier and
attention mask (onnx-runtime-ep-cuda src/kernels/standard_attention.rs:
nonpad_kv_seqlen in attention_row -- keys j >= nonpad[b] masked, causal
offset nonpad[b] - S; mask_bias -- a float or bool mask broadcast against
[batch, head, query, key], a short key axis padding with -inf) against the
fp64 oracle, through the C ABI.  Present K/V stay exact copies."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(sa, c, inp, **kw):
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    pk, pv = torch.empty_like(k), torch.empty_like(v)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkw = {n: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for n, t in kw.items()}
    y = sa.attn_prefill(q, k, v, causal=c.causal, scale=c.eff_scale(), softcap=c.softcap,
                        present_k=pk, present_v=pv, err_word=err, **gkw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pk.cpu(), inp["k"]) and torch.equal(pv.cpu(), inp["v"])
    return y


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("softcap", [0.0, 50.0, 5.0])
def test_padding_frontier_on_the_tensor_core_kernel(cuda_lib, dt, causal, softcap):
    # per-batch valid lengths across tile boundaries; with causal the offset
    # nonpad - S leaves the first S - nonpad query rows with no key (output 0)
    c = synth.PrefillCase("pad", B=4, S=300, Hq=8, Hkv=2, D=128, causal=causal,
                          softcap=softcap, dtype=dt)
    inp = synth.make_prefill_inputs(c, seed=31)
    nonpad = torch.tensor([300, 257, 128, 1], dtype=torch.int64)
    y = _run(cuda_lib, c, inp, nonpad_kv_seqlen=nonpad)
    ref = oracle.prefill(inp["q"], inp["k"], inp["v"], scale=c.eff_scale(), causal=causal,
                         softcap=softcap, nonpad_kv_seqlen=nonpad)
    assert_close(to64(y), ref, y.dtype, f"pad {dt} causal={causal} cap={softcap}")
    if causal:
        # rows before S - nonpad see nothing: exact zeros
        y3 = y.reshape(c.B, c.Hq, c.S, c.D)[3, :, : c.S - 1].float()
        assert torch.count_nonzero(y3).item() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_padding_frontier_d64_and_negative_entries(cuda_lib, D):
    c = synth.PrefillCase("pad", B=3, S=200, Hq=4, Hkv=4, D=D, causal=True, softcap=0.0)
    inp = synth.make_prefill_inputs(c, seed=32)
    nonpad = torch.tensor([-1, 200, 77], dtype=torch.int64)  # -1: no padding frontier
    y = _run(cuda_lib, c, inp, nonpad_kv_seqlen=nonpad)
    ref = oracle.prefill(inp["q"], inp["k"], inp["v"], scale=c.eff_scale(), causal=True,
                         nonpad_kv_seqlen=nonpad)
    assert_close(to64(y), ref, y.dtype, f"pad D={D}")


def _mask(kind, B, Hq, S, seed):
    g = torch.Generator().manual_seed(seed)
    shape = {"bool_ss": (S, S), "f32_b1ss": (B, 1, S, S), "bf16_hss": (Hq, S, S),
             "f16_s": (S,), "bool_short": (1, S, S - 5), "f32_bhs1": (B, Hq, S, 1)}[kind]
    if kind.startswith("bool"):
        return torch.rand(shape, generator=g) > 0.25
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[kind.split("_")[0]]
    m = torch.randn(shape, generator=g) * 1.5
    m[torch.rand(shape, generator=g) < 0.1] = -float("inf")
    return m.to(dt)


@pytest.mark.parametrize("kind", ["bool_ss", "f32_b1ss", "bf16_hss", "f16_s", "bool_short",
                                  "f32_bhs1"])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_attention_mask(cuda_lib, kind, dt):
    # bf16 runs on the stream kernel's dense source, f32 on the split-K kernel
    c = synth.PrefillCase("mask", B=2, S=96, Hq=8, Hkv=2, D=64, causal=True, softcap=30.0,
                          dtype=dt)
    inp = synth.make_prefill_inputs(c, seed=33)
    mask = _mask(kind, c.B, c.Hq, c.S, 34)
    nonpad = torch.tensor([96, 80], dtype=torch.int64)
    y = _run(cuda_lib, c, inp, attn_mask=mask, nonpad_kv_seqlen=nonpad)
    ref = oracle.prefill(inp["q"], inp["k"], inp["v"], scale=c.eff_scale(), causal=True,
                         softcap=c.softcap, attn_mask=mask, nonpad_kv_seqlen=nonpad)
    assert_close(to64(y), ref, y.dtype, f"mask {kind} {dt}")


def test_attention_mask_d128_non_causal(cuda_lib):
    c = synth.PrefillCase("mask", B=1, S=150, Hq=4, Hkv=1, D=128, causal=False, softcap=0.0)
    inp = synth.make_prefill_inputs(c, seed=35)
    mask = _mask("bool_ss", c.B, c.Hq, c.S, 36)
    y = _run(cuda_lib, c, inp, attn_mask=mask)
    ref = oracle.prefill(inp["q"], inp["k"], inp["v"], scale=c.eff_scale(), causal=False,
                         attn_mask=mask)
    assert_close(to64(y), ref, y.dtype, "mask d128")
