"""The seeded input recipe: index rows, padding tails, page tables and FP8
records have the structure the workloads state (CPU only)."""
import numpy as np
import torch

import oracle
import synth


def test_sorted_sample_rows_are_distinct_sorted_and_in_range():
    idx = synth.sorted_sample_rows(64, 100, 900, 300, seed=3)
    assert idx.shape == (64, 300) and idx.dtype == torch.int64
    assert bool((idx[:, 1:] > idx[:, :-1]).all())
    assert int(idx.min()) >= 100 and int(idx.max()) < 900
    # uniform over the range: the mean of 19,200 draws sits near the middle
    assert abs(float(idx.double().mean()) - 499.5) < 10.0
    assert torch.equal(idx, synth.sorted_sample_rows(64, 100, 900, 300, seed=3))
    assert not torch.equal(idx, synth.sorted_sample_rows(64, 100, 900, 300, seed=4))


def test_padded_rows_follow_the_recipe_and_stay_valid():
    # the bf16 decode workload's index rows: 256 rows of 2,048 over 8,192
    # positions, a row padded with probability 0.05 by a tail of U[1, 256]
    rows, K, T = 256, 2048, 8192
    idx = synth.sorted_sample_rows(rows, 0, T, K, seed=11)
    pad = synth.pad_tails(idx, seed=12, prob=0.05, max_pad=256)
    n_pad = (pad == -1).sum(dim=1)
    padded = n_pad > 0
    assert 2 <= int(padded.sum()) <= 35          # about 13 of 256 expected
    assert int(n_pad[padded].min()) >= 1 and int(n_pad[padded].max()) <= 256
    for r in torch.nonzero(padded).flatten().tolist():
        k = K - int(n_pad[r])
        assert bool((pad[r, k:] == -1).all())     # a trailing tail only
        assert torch.equal(pad[r, :k], idx[r, :k])  # the largest indices were dropped
    status, err = oracle.validate_indices(pad.reshape(1, rows, 1, K), bound=T)
    assert err == 0 and not status.any()


def test_page_tables_map_every_sequence_onto_distinct_pages():
    ctx, table, num_pages = synth.paged_layout(B=40, ctx_low=1, ctx_high=300, page_tokens=16,
                                               seed=5)
    assert int(ctx.min()) >= 1 and int(ctx.max()) <= 300
    assert table.shape == (40, 19)                 # ceil(300 / 16) slots per sequence
    used = []
    for b in range(40):
        n = (int(ctx[b]) + 15) // 16
        assert bool((table[b, :n] >= 0).all()) and bool((table[b, n:] == -1).all())
        used += table[b, :n].tolist()
    assert sorted(used) == list(range(num_pages))  # a permutation of one shared pool


def test_fp8_records_layout_and_block_exponents():
    nope = synth.normal((5, 512), "f32", seed=21)
    nope[1, 64:128] = 0.0                          # an all-zero block
    nope[2, :64] *= 1.0e4                          # a large block
    rope = synth.normal((5, 64), "bf16", seed=22)
    rec = synth.quantize_fp8_block64_records(nope, rope)
    assert rec.shape == (5, 648) and rec.dtype == torch.uint8
    x = nope.reshape(5, 8, 64).double()
    amax = x.abs().amax(dim=2)
    e = rec[:, : 8 * 65].reshape(5, 8, 65)[:, :, 0].to(torch.int64) - 127
    nz = amax > 0
    assert bool((amax[nz] / torch.exp2(e[nz].double()) <= 448.0).all())
    assert bool((amax[nz] / torch.exp2(e[nz].double() - 1) > 448.0).all())  # smallest e
    assert int(e[1, 1]) == 0                        # zero block: byte 127
    # RoPE tail: 64 little-endian bf16 values from byte 520
    tail = rec[:, 520:648].to(torch.int32)
    bits = (tail[:, 0::2] | (tail[:, 1::2] << 8)).to(torch.int16)
    assert torch.equal(bits.view(torch.bfloat16), rope)
    # the codes decode back to the inputs within E4M3's half-ULP (relative 2^-4)
    codes = rec[:, : 8 * 65].reshape(5, 8, 65)[:, :, 1:].contiguous()
    vals = codes.view(torch.float8_e4m3fn).double() * torch.exp2(e.double())[:, :, None]
    err = (vals - x).abs()
    assert bool((err <= x.abs() * 2.0 ** -4 + torch.exp2(e.double() - 9)[:, :, None]).all())
    assert np.isfinite(vals.numpy()).all()


def test_window_workload_index_rows_overlap_the_window():
    # The FP8 latent workload unites a 128-token window with 2,048 indices
    # drawn from all 65,536 positions: about 2048 * 128 / 65536 = 4 selected
    # entries per row fall inside the window and must be counted once.
    c = synth.csa_fp8()
    idx = synth.sorted_sample_rows(c.B * c.I, 0, c.T, c.K, seed=1 * 7919 + 4)
    inside = (idx >= c.T - c.window).sum(dim=1)
    assert int(inside.sum()) > 0
    assert 1.0 <= float(inside.double().mean()) <= 10.0
    # make_sparse_inputs draws them that way
    small = synth.csa_fp8(B=4, T=600, K=300)
    inp = synth.make_sparse_inputs(small, seed=2)
    assert int((inp["idx"] >= small.T - small.window).sum()) > 0
