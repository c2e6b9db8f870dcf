"""ar_allreduce_noalloc: the all-reduce entry point that allocates nothing.

It serves callers that cannot allocate device memory when they reduce (their
memory belongs to another library's pool or arena, or cudaMalloc is off limits
on their latency-critical path).  This file runs last, so that a failure here
leaves every other test already run.  It checks, on two calls in a row, that
the entry point's outputs match the handle-based ar_allreduce bit for bit
(the tolerance every all-reduce test here uses) and the CPU oracle.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(R, dtype_code, ins, outs, numel, stream):
    """Through the C ABI, with R device pointers per side."""
    import tensor_decode_all_gb300 as tda
    return tda.ar_allreduce_noalloc(R, dtype_code, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs],
                                    numel, stream.cuda_stream)


@pytest.mark.parametrize("R,dtype,numel,slots", [(2, "f16", 131072, "pinned"), (8, "bf16", 393216, "hbm"),
                                                 (3, "f16", 4099, "hbm")])
def test_noalloc_matches_handle_path_two_calls_in_a_row(R, dtype, numel, slots):
    import tensor_decode_all_gb300 as tda
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    code = {"f16": tda.AR_F16, "bf16": tda.AR_BF16}[dtype]
    h = tda.Handle(R, tdt, numel, slots)
    streams = rank_streams(R)
    s = torch.cuda.Stream()
    for call in range(2):
        xs = inputs.allreduce_inputs(5, R, numel, dtype, "uniform", 40 + call)
        ins = [to_dev(x, dtype) for x in xs]
        ref = [torch.empty_like(t) for t in ins]
        enqueue(h, "allreduce", ins, ref, streams)
        got = [torch.full_like(t, float("nan")) for t in ins]
        s.wait_stream(torch.cuda.current_stream())
        assert _noalloc(R, code, ins, got, numel, s) == 0
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        h.check()
        want = oracle.allreduce(xs, dtype, ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(got[r]), to_bits(ref[r]), dtype, f"call {call} rank {r} vs ar_allreduce")
            assert_bits_equal(to_bits(got[r]), want, dtype, f"call {call} rank {r} vs oracle")
    h.destroy()


def test_noalloc_rejects_oversize_and_bad_arguments():
    import tensor_decode_all_gb300 as tda
    t = torch.zeros(16, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    assert _noalloc(2, tda.AR_F16, [t, t], [t, t], (1 << 19) + 1, s) == tda.ar.AR_ETOOBIG
    assert _noalloc(9, tda.AR_F16, [t] * 9, [t] * 9, 8, s) == tda.ar.AR_EINVAL
    assert _noalloc(2, tda.AR_C64, [t, t], [t, t], 8, s) == tda.ar.AR_EINVAL
