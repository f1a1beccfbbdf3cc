"""The bounded-wait timeout path, run on purpose without a GPU fault.

Every pipelined kernel of the library waits on its shared-memory barriers
for a bounded number of cycles, then records SA_ERRBIT_TIMEOUT in the
caller's error word and returns.  sa_check_wait_timeout makes one warp wait
on a barrier that nothing arrives on (no copy or MMA in flight): the wait must
give up after its limit, report the bit, make a second wait return at once,
and leave the context usable for the next call.
"""
import pytest
import torch

import oracle
import synth
from helpers import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
WAIT_CYCLES = 2_000_000_000  # the library's per-wait limit, in SM cycles


def test_wait_gives_up_reports_and_context_stays_usable(cuda_lib):
    err, out = cuda_lib.check_wait_timeout(DEV)
    torch.cuda.synchronize()
    o = [int(v) & 0xFFFFFFFF for v in out.cpu()]
    assert int(err.item()) == cuda_lib.ERRBIT_TIMEOUT
    assert o[0] == 1, "the first wait did not give up"
    assert o[1] == 1, "the second wait did not return at once on the abort flag"
    cycles = o[2] | (o[3] << 32)
    assert WAIT_CYCLES <= cycles < 10 * WAIT_CYCLES
    # the context still runs a call, and its result matches the oracle
    c = synth.sparse_bf16(B=2, Hq=16, Hkv=2, T=512, K=100, I=2)
    inp = synth.make_sparse_inputs(c, seed=5)
    d = {k: v.to(DEV) for k, v in inp.items()}
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = cuda_lib.sparse_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["idx"],
                                    scale=c.eff_scale(), err_word=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    ref = oracle.sparse_attention(inp["q"], inp["idx"], inp["k_cache"], inp["v_cache"],
                                  scale=c.eff_scale())
    assert_close(to64(y), ref, y.dtype, "decode after a timeout")


def test_wait_timeout_argument_checks(cuda_lib):
    L = cuda_lib.load()
    buf = torch.zeros(8, dtype=torch.int32, device=DEV)
    assert L.sa_check_wait_timeout(None, buf.data_ptr(), None) == -1
    assert L.sa_check_wait_timeout(buf.data_ptr(), None, None) == -1
    assert L.sa_check_wait_timeout(buf.data_ptr() + 2, buf.data_ptr() + 8, None) < 0
