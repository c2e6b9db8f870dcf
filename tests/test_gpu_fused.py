"""GPU parity of the single-launch form (ar_allreduce_fused / ar_allgather_fused).

One cooperative launch plays all R ranks of a call (block (b, r) is block b of
rank r), on the same handle state as the per-rank calls.  Every output must
match the CPU oracle bit for bit, as for the per-rank form, and the two forms
must interleave on one handle.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "c64": torch.complex64}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle(R, dtype, max_numel, slots):
    import tensor_decode_all_gb300 as tda
    return tda.Handle(R, TORCH[dtype], max_numel, slots)


def _fused_allreduce(h, xs, dtype, stream):
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    stream.wait_stream(torch.cuda.current_stream())
    h.allreduce_fused(ins, outs, stream)
    torch.cuda.current_stream().wait_stream(stream)
    return ins, outs


def _check_allreduce(outs, xs, dtype, what):
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, dtype, f"{what} rank {r}")


@pytest.mark.parametrize("R,dtype,n,slots,algo", [
    (2, "f16", 4096, "pinned", None),          # one decode token
    (2, "f16", 131072, "pinned", None),        # the 256 KiB host all-reduce cap
    (8, "bf16", 393216, "hbm", None),          # 48 rows x hidden 8192 (two-shot)
    (8, "bf16", 393216, "hbm", "oneshot"),
    (4, "bf16", (3 << 20) + 5, "hbm", None),   # two-shot, several stages, ragged tail
    (4, "f16", (1 << 18) + 3, "pinned", "twoshot"),
    (3, "bf16", 100003, "hbm", None),
    (1, "f16", 777, "hbm", None),
])
def test_fused_allreduce_matches_oracle(R, dtype, n, slots, algo):
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 7)
    h = _handle(R, dtype, n, slots)
    if algo:
        h.set_algo(algo)
    _, outs = _fused_allreduce(h, xs, dtype, torch.cuda.Stream())
    torch.cuda.synchronize()
    h.check()
    _check_allreduce(outs, xs, dtype, f"fused R={R} {dtype} n={n} {slots} {algo}")
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
def test_fused_and_per_rank_calls_alternate(slots):
    """A fused call counts as one call of every rank: per-rank and fused calls
    interleave on one handle, across both slot parities, and all stay exact."""
    R, n, dtype = 4, 70001, "bf16"
    h = _handle(R, dtype, n, slots)
    streams = rank_streams(R)
    fstream = torch.cuda.Stream()
    for call, kind in enumerate(["fused", "rank", "rank", "fused", "fused", "rank", "fused"]):
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 100 + call)
        if kind == "fused":
            _, outs = _fused_allreduce(h, xs, dtype, fstream)
        else:
            ins = [to_dev(x, dtype) for x in xs]
            outs = [torch.empty_like(t) for t in ins]
            enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        h.check()
        _check_allreduce(outs, xs, dtype, f"call {call} ({kind}) {slots}")
    h.destroy()


def test_fused_graph_replay_fresh_inputs():
    """Fused calls captured in a graph (C calls), replayed with refilled inputs."""
    R, n, dtype, C = 8, 393216, "bf16", 6
    h = _handle(R, dtype, n, "hbm")
    ins = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(C)]
    outs = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(C)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for c in range(C):
                h.allreduce_fused(ins[c], outs[c], torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(3):
        xs_all = []
        for c in range(C):
            xs = inputs.allreduce_inputs(3, R, n, dtype, "normal", rep * C + c)
            for r in range(R):
                ins[c][r].copy_(to_dev(xs[r], dtype))
            xs_all.append(xs)
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in (0, C - 1):
            _check_allreduce(outs[c], xs_all[c], dtype, f"rep {rep} call {c}")
    del g
    h.destroy()


@pytest.mark.parametrize("pdl", [True, False])
def test_fused_pdl_on_and_off(pdl):
    R, n, dtype = 2, 131072, "f16"
    h = _handle(R, dtype, n, "pinned")
    h.set_pdl(pdl)
    s = torch.cuda.Stream()
    for call in range(5):
        xs = inputs.allreduce_inputs(2, R, n, dtype, "normal4", call)
        _, outs = _fused_allreduce(h, xs, dtype, s)
        torch.cuda.synchronize()
        h.check()
        _check_allreduce(outs, xs, dtype, f"pdl={pdl} call {call}")
    h.destroy()


@pytest.mark.parametrize("R,slots,n", [(4, "hbm", 1000 * 500), (8, "pinned", 4096), (8, "hbm", 4097), (3, "hbm", 17)])
def test_fused_allgather_matches_oracle(R, slots, n):
    zs = inputs.allgather_inputs(4, R, n, 11)
    h = _handle(R, "c64", n, slots)
    ins = [to_dev(z, "c64") for z in zs]
    outs = [torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    h.allgather_fused(ins, outs, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    h.check()
    want = oracle.allgather(zs, ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, "c64", f"fused allgather R={R} {slots} n={n} rank {r}")
    h.destroy()


def test_fused_declines():
    """Each decline returns its code and enqueues nothing."""
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    R, n = 2, 1024
    h = _handle(R, "f16", n, "hbm")
    s = torch.cuda.Stream()
    ins = [torch.zeros(n, dtype=torch.float16, device="cuda") for _ in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    p_in = [t.data_ptr() for t in ins]
    p_out = [t.data_ptr() for t in outs]
    assert ar.ar_allreduce_fused(h.ptr, p_in, p_out, n + 1, s.cuda_stream) == ar.AR_ETOOBIG
    assert ar.ar_allreduce_fused(h.ptr, [p_in[0], 0], p_out, n, s.cuda_stream) == ar.AR_EINVAL
    assert ar.ar_allreduce_fused(h.ptr, [p_in[0], p_in[1] + 2], p_out, n - 1, s.cuda_stream) == ar.AR_EINVAL
    assert ar.ar_allreduce_fused(h.ptr, p_in, p_out, n, 0) == ar.AR_ESTREAM
    assert ar.ar_allreduce_fused(h.ptr, p_in, p_out, 0, s.cuda_stream) == ar.AR_OK
    # A per-rank sequence left half-issued: rank 0 has one call more than rank 1.
    streams = rank_streams(R)
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    h.allreduce(0, ins[0], outs[0], streams[0])
    assert ar.ar_allreduce_fused(h.ptr, p_in, p_out, n, s.cuda_stream) == ar.AR_EINVAL
    h.allreduce(1, ins[1], outs[1], streams[1])   # completes rank 0's call
    torch.cuda.synchronize()
    h.check()
    # an all-reduce on a complex64 handle is refused
    g = tda.Handle(R, torch.complex64, 8, "hbm")
    assert ar.ar_allreduce_fused(g.ptr, p_in, p_out, 8, s.cuda_stream) == ar.AR_EINVAL
    g.destroy()
    h.destroy()
