"""ar_allreduce_noalloc: the all-reduce entry point that allocates nothing.

It serves callers that cannot allocate device memory when they reduce (their
memory belongs to another library's pool or arena, or cudaMalloc is off limits
on their latency-critical path).  This file runs last, so that a failure here
leaves every other test already run.  It checks, on two calls in a row, that
the entry point's outputs match the handle-based ar_allreduce bit for bit
(the tolerance every all-reduce test here uses) and the CPU oracle, and that
the array's error record reads OK after them.  It also checks the status
plumbing (a record planted from the host is reported, and the next call
clears it) and first calls from several host threads at once.
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
        status, info = tda.ar.ar_noalloc_status()
        assert status == tda.ar.AR_OK and info.code == tda.ar.AR_OK, f"call {call}: {status}"
    h.destroy()


def test_noalloc_status_reports_a_record_until_the_next_call_clears_it():
    """A block whose wait ran out writes an error record into the array and
    leaves; the caller reads it with ar_noalloc_status after synchronising.
    The record is planted from the host (no wait is made to run out), then the
    next call must clear it and still compute the right bits."""
    import tensor_decode_all_gb300 as tda
    ar = tda.ar
    R, numel = 2, 4096
    s = torch.cuda.Stream()
    planted = ar.ErrorInfo(ar.AR_ETIMEOUT, 1, 3, 0, 7, 5)
    assert ar.ar_noalloc_debug_record(planted) == ar.AR_OK
    code, info = ar.ar_noalloc_status()
    assert code == ar.AR_ETIMEOUT
    assert (info.code, info.rank, info.block, info.peer, info.want, info.seen) == (ar.AR_ETIMEOUT, 1, 3, 0, 7, 5)
    xs = inputs.allreduce_inputs(1, R, numel, "f16", "uniform", 77)
    ins = [to_dev(x, "f16") for x in xs]
    got = [torch.empty_like(t) for t in ins]
    s.wait_stream(torch.cuda.current_stream())
    assert _noalloc(R, tda.AR_F16, ins, got, numel, s) == 0
    s.synchronize()
    code, info = ar.ar_noalloc_status()
    assert code == ar.AR_OK and info.code == ar.AR_OK and info.rank == 0 and info.want == 0
    want = oracle.allreduce(xs, "f16", ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(got[r]), want, "f16", f"rank {r} after a planted record")


def test_noalloc_first_calls_from_several_threads():
    """First calls made by several host threads at once share one set-up of the
    device (a lock guards it); every thread's results are right."""
    import threading

    import tensor_decode_all_gb300 as tda
    R, numel = 2, 2048
    n = 4
    xs = [inputs.allreduce_inputs(1, R, numel, "bf16", "uniform", 90 + i) for i in range(n)]
    ins = [[to_dev(x, "bf16") for x in xi] for xi in xs]
    outs = [[torch.empty_like(t) for t in ii] for ii in ins]
    streams = [torch.cuda.Stream() for _ in range(n)]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    rcs = [None] * n
    lock = threading.Lock()

    def run(i):
        torch.cuda.set_device(0)
        rc = _noalloc(R, tda.AR_BF16, ins[i], outs[i], numel, streams[i])
        with lock:
            rcs[i] = rc
        # calls on different streams share the array and race: keep them apart
        streams[i].synchronize()

    # the threads start together (the set-up races), but each call runs alone:
    # thread i waits for thread i-1's call before it enqueues its own
    gate = [threading.Event() for _ in range(n + 1)]
    gate[0].set()

    def ordered(i):
        torch.cuda.set_device(0)
        tda.ar.ar_noalloc_status()          # first use of the device from this thread
        gate[i].wait()
        run(i)
        gate[i + 1].set()

    threads = [threading.Thread(target=ordered, args=(i,)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert rcs == [0] * n, rcs
    torch.cuda.synchronize()
    for i in range(n):
        want = oracle.allreduce(xs[i], "bf16", ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[i][r]), want, "bf16", f"thread {i} rank {r}")


def test_noalloc_rejects_oversize_and_bad_arguments():
    import tensor_decode_all_gb300 as tda
    t = torch.zeros(16, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    assert _noalloc(2, tda.AR_F16, [t, t], [t, t], (1 << 19) + 1, s) == tda.ar.AR_ETOOBIG
    assert _noalloc(9, tda.AR_F16, [t] * 9, [t] * 9, 8, s) == tda.ar.AR_EINVAL
    assert _noalloc(2, tda.AR_C64, [t, t], [t, t], 8, s) == tda.ar.AR_EINVAL
