"""GPU parity of ratio-4 index scoring and top-k selection
(onnx-runtime-ep-cpu compressed_sparse_attention.rs select_ratio4_topk;
onnx-runtime-ep-cuda csa_ratio4_index_select) against the oracle, through the
C ABI.  Selections, row statuses and error words are compared bit for bit:
both sides take every integer decision (FP4 codes, the order of scores) in
the pages' binary32 arithmetic."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(sa, c, inp, **kw):
    st = torch.full((c.B * c.S,), 77, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = sa.sparse_index_select(inp["query"].to(DEV), inp["weight"].to(DEV), inp["keys"].to(DEV),
                                 topk=c.topk, query_start=c.query_start, row_status=st,
                                 err_word=err, **kw)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), st.cpu().numpy(), int(err.item())


def _check(sa, c, inp, what, **kw):
    okw = dict(kw)
    if "query_start_b" in okw and okw["query_start_b"] is not None:
        okw["query_start_b"] = okw["query_start_b"].cpu()
    gkw = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    sel, st, err = _run(sa, c, inp, **gkw)
    ref, rst, rerr = oracle.index_select(inp["query"], inp["weight"], inp["keys"], topk=c.topk,
                                         query_start=c.query_start, **okw)
    assert np.array_equal(sel, ref), f"{what}: selection differs"
    assert np.array_equal(st, rst), f"{what}: row status differs"
    assert err == (rerr << 9), f"{what}: err_word {err:#x} vs {rerr << 9:#x}"
    return sel, st


def _case(**over):
    kw = dict(B=3, S=2, IH=8, ID=128, R=700, topk=150, query_start=2000)
    kw.update(over)
    return synth.IndexCase("t", **kw)


@pytest.mark.parametrize("ID", [32, 64, 128, 256])
@pytest.mark.parametrize("ascending", [False, True])
def test_index_select_bit_exact(cuda_lib, ID, ascending):
    c = _case(ID=ID)
    inp = synth.make_index_inputs(c, seed=ID)
    _check(cuda_lib, c, inp, f"ID {ID}", ascending=ascending, out_heads=2)


@pytest.mark.parametrize("over", [dict(IH=1, R=40, topk=16, query_start=100),     # one head
                                  dict(IH=64, R=3000, topk=2048, query_start=20000),
                                  dict(IH=3, R=257, topk=300, query_start=900),    # topk > limit
                                  dict(S=5, R=128, topk=33, query_start=200),       # several queries
                                  dict(IH=130, R=500, topk=1, query_start=10000),   # topk 1
                                  dict(IH=8, R=5000, topk=4096, query_start=40000)])  # largest k
def test_index_select_shapes(cuda_lib, over):
    c = _case(**over)
    inp = synth.make_index_inputs(c, seed=21)
    _check(cuda_lib, c, inp, str(over))


def test_causal_limits_per_batch_and_empty_rows(cuda_lib):
    c = _case(B=4, S=3, R=400, topk=120)
    inp = synth.make_index_inputs(c, seed=22)
    starts = torch.tensor([-5, 2, 450, 5000], dtype=torch.int64)  # limits 0, 0/0/1, ~113, 400
    sel, st = _check(cuda_lib, c, inp, "per-batch starts", query_start_b=starts)
    assert (sel[0] == -1).all()


def test_equal_scores_are_flagged_and_ranked_by_record(cuda_lib):
    c = _case(B=2, S=1, R=600, topk=200)
    inp = synth.make_index_inputs(c, seed=23)
    keys = inp["keys"].clone()
    keys[:, 300:400] = keys[:, 100:200]  # 100 duplicated records per batch: equal scores
    inp = dict(inp, keys=keys)
    sel, st = _check(cuda_lib, c, inp, "duplicates")
    assert (st & cuda_lib.SEL_TIE).all()


def test_wide_scale_spreads_take_the_serial_path(cuda_lib):
    # block scales 2^+-12 apart in a record: the exact integer path does not
    # apply, the serial binary32 loop runs (and must still match bit for bit)
    c = _case(B=2, S=2, R=500, topk=100)
    inp = synth.make_index_inputs(c, seed=24)
    keys = inp["keys"].clone()
    keys[:, ::3, 0] = 127 + 12
    keys[:, ::3, 17] = 127 - 12
    keys[:, 1::7, 34] = 4           # tiny scale: subnormal products
    inp = dict(inp, keys=keys)
    _check(cuda_lib, c, inp, "spread scales")


def test_nonfinite_key_scales(cuda_lib):
    c = _case(B=2, S=1, R=300, topk=64)
    inp = synth.make_index_inputs(c, seed=25)
    keys = inp["keys"].clone()
    keys[0, 10, 0] = 0xFF           # NaN scale: the head's dot is NaN, relu gives 0
    keys[1, 20, 17] = 254           # 2^126 * codes up to 12: infinite products
    inp = dict(inp, keys=keys)
    _check(cuda_lib, c, inp, "non-finite scales")


def test_long_rows(cuda_lib):
    # 20,000 records: a hash set of 65,536 slots in 8 parts, a large threshold bin
    c = _case(B=2, S=1, IH=4, ID=32, R=20000, topk=1000, query_start=100000)
    inp = synth.make_index_inputs(c, seed=26)
    _check(cuda_lib, c, inp, "long rows", ascending=True)


def test_deterministic_and_independent_of_workspace_contents(cuda_lib):
    c = _case(IH=16, R=2000, topk=500, query_start=9000)
    inp = synth.make_index_inputs(c, seed=27)
    need = cuda_lib.sparse_index_select_workspace(inp["query"].to(DEV), inp["weight"].to(DEV),
                                                  inp["keys"].to(DEV), topk=c.topk)
    outs = []
    for fill in (0, 0xFF, 0x5A):
        ws = torch.full((need,), fill, dtype=torch.uint8, device=DEV)
        outs.append(_run(cuda_lib, c, inp, workspace=ws))
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])


def test_full_size_index_select(cuda_lib):
    """B16 decode rows at position 65,535: 16,384 records of 128 FP4 dims, 64
    index heads, top-k 2,048 -- the benchmark's launch configuration; every
    row checked bit for bit."""
    c = synth.index_select_fp4()
    inp = synth.make_index_inputs(c, seed=1)
    _check(cuda_lib, c, inp, "full size")
