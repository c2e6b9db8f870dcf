"""GPU parity of the cluster form (AR_ALGO_CLUSTER) and of ar_allreduce_all.

In a launch of every rank at once, block b of every rank forms one
thread-block cluster and the hardware cluster barrier stands in for the
per-block flags; the data still moves through the handle's slots.  Every
output must match the CPU oracle bit for bit, whatever the variant (one-shot,
two-shot with each sub-tile size), slot kind, rank count, size or ragged
tail, and the form must share one handle with the flag forms in any order.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, enqueue, generate, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}
NEVER = (1 << 64) - 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle(R, dtype, n, slots, **tactics):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, TORCH[dtype], n, slots)
    assert h.info().cluster_form >= 1, "cluster launches unavailable on this GPU"
    h.set_algo("cluster")
    if tactics:
        h.set_tactics(**tactics)
    return h


def _fused(h, ins, outs, stream):
    stream.wait_stream(torch.cuda.current_stream())
    h.allreduce_fused(ins, outs, stream)
    torch.cuda.current_stream().wait_stream(stream)


def _check(outs, xs, dtype, what):
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, dtype, f"{what} rank {r}")


@pytest.mark.parametrize("variant", ["oneshot", "sub64", "sub128", "sub256"])
@pytest.mark.parametrize("R,dtype,slots", [(1, "f16", "hbm"), (2, "f16", "pinned"), (2, "bf16", "hbm"),
                                           (3, "bf16", "pinned"), (4, "f16", "hbm"), (5, "bf16", "hbm"),
                                           (8, "bf16", "hbm"), (8, "f16", "pinned")])
@pytest.mark.parametrize("n", [1, 7, 4099, 65536 + 9, 393216])
def test_cluster_variants_match_oracle(variant, R, dtype, slots, n):
    """Every variant at sizes from one element to the decode-sized 393216,
    with ragged tails; the block cap (3 clusters) makes the larger calls run
    several stages per cluster."""
    sub = {"oneshot": 0, "sub64": 64, "sub128": 128, "sub256": 256}[variant]
    h = _handle(R, dtype, n, slots, cluster_twoshot_min_bytes=NEVER if sub == 0 else 0, twoshot_sub=sub,
                max_blocks=3 if n > 4099 else 0)
    p = h.plan("allreduce_fused", n)
    assert p.algo == 3 and p.subtile_vecs == sub
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", n % 97)
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.full_like(t, float("nan")) for t in ins]
    _fused(h, ins, outs, torch.cuda.Stream())
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs, dtype, f"{variant} R={R} n={n} {slots}")
    h.destroy()


def test_auto_picks_the_cluster_form_for_launches_of_every_rank():
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(8, torch.bfloat16, 393216, "hbm")
    if h.info().cluster_form < 1:
        pytest.skip("cluster launches unavailable")
    t = h.tactics()
    assert t["cluster_max_bytes"] >= 393216 * 2 and t["all_fused"] == 1
    p = h.plan("allreduce_fused", 393216)
    assert p.algo == 3 and p.flag_rounds == 2 and p.subtile_vecs == 64 and p.max_stages == 1
    assert h.plan("allreduce", 393216).algo in (0, 1)        # a rank's own launch keeps the flag forms
    h.set_tactics(cluster_max_bytes=0)
    assert h.plan("allreduce_fused", 393216).algo in (0, 1)
    h.set_tactics(cluster_max_bytes=393216 * 2 - 1)          # the limit is per rank, inclusive
    assert h.plan("allreduce_fused", 393216).algo in (0, 1)
    h.set_tactics(cluster_max_bytes=393216 * 2)
    assert h.plan("allreduce_fused", 393216).algo == 3
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
def test_config3_through_allreduce_all_1000_calls(slots):
    """Workload 3 (R=8 bf16 N=393216) through the default entry for a caller
    that drives all ranks, ar_allreduce_all, which fuses the ranks into one
    launch (a cluster launch in HBM; over the host link, above the cluster
    form's limit, one cooperative launch of the flag forms): a graph of 100
    calls replayed 10 times with fresh inputs, every call checked on every
    rank (1000 calls)."""
    import tensor_decode_all_gb300 as tda
    R, n, C, REPLAYS, dtype = 8, 393216, 100, 10, "bf16"
    h = tda.Handle(R, torch.bfloat16, n, slots)
    if h.info().cluster_form < 1:
        pytest.skip("cluster launches unavailable")
    streams = rank_streams(R)
    ins = torch.empty((C, R, n), dtype=torch.bfloat16, device="cuda")
    outs = torch.empty((C, R, n), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            for s in streams:
                s.wait_stream(cap)
            for c in range(C):
                h.allreduce_all([ins[c, r] for r in range(R)], [outs[c, r] for r in range(R)], streams)
            for s in streams:
                cap.wait_stream(s)
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(REPLAYS):
        xs_all = generate(inputs.allreduce_inputs, [(3, R, n, dtype, "normal", rep * C + c) for c in range(C)])
        ins.copy_(torch.from_numpy(np.stack([np.stack(xs) for xs in xs_all]).view(np.int16)).view(torch.bfloat16))
        outs.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        want = generate(lambda xs: oracle.allreduce(xs, dtype, ranks=[0])[0], [(xs,) for xs in xs_all])
        got = to_bits(outs)
        for c in range(C):
            if not np.array_equal(got[c], np.broadcast_to(want[c], (R, n))):
                for r in range(R):
                    assert_bits_equal(got[c, r], want[c], dtype, f"replay {rep} call {c} rank {r}")
    del g
    h.destroy()


def test_every_form_interleaves_on_one_handle():
    """Per-rank flag calls (one-shot, two-shot, tagged), fused flag calls and
    cluster calls, with changing sizes and grids, in one sequence on one
    handle and then in one captured graph: the call counts (slot parity) and
    the stage counts (flags, tags) stay consistent across the forms."""
    import tensor_decode_all_gb300 as tda
    R, dtype = 4, "bf16"
    nmax = 1 << 20
    h = tda.Handle(R, torch.bfloat16, nmax, "hbm")
    if h.info().cluster_form < 1:
        pytest.skip("cluster launches unavailable")
    streams = rank_streams(R)
    one = torch.cuda.Stream()
    # (form, launch, numel)
    seq = [("oneshot", "rank", 4096), ("cluster", "fused", 8195), ("tagged", "rank", 1024),
           ("cluster", "fused", 700001), ("twoshot", "rank", 300007), ("oneshot", "fused", 5000),
           ("cluster", "fused", 77), ("tagged", "fused", 2048), ("twoshot", "fused", 600000),
           ("cluster", "fused", 393216), ("oneshot", "rank", 9), ("cluster", "fused", 131072)]
    for rnd in range(2):
        for i, (form, launch, n) in enumerate(seq):
            xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 100 * rnd + i)
            ins = [to_dev(x, dtype) for x in xs]
            outs = [torch.full_like(t, float("nan")) for t in ins]
            h.set_algo(form)
            if launch == "rank":
                enqueue(h, "allreduce", ins, outs, streams)
            else:
                _fused(h, ins, outs, one)
            torch.cuda.synchronize()
            h.check()
            _check(outs, xs, dtype, f"round {rnd} step {i} {form}/{launch} n={n}")
    # the same mix inside one graph (forms and grids frozen at capture)
    xs_all, ins_all, outs_all = [], [], []
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            for i, (form, launch, n) in enumerate(seq):
                xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 500 + i)
                ins = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
                outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
                xs_all.append(xs)
                ins_all.append(ins)
                outs_all.append(outs)
                h.set_algo(form)
                if launch == "rank":
                    for s in streams:
                        s.wait_stream(cap)
                    for r in range(R):
                        h.allreduce(r, ins[r], outs[r], streams[r])
                    for s in streams:
                        cap.wait_stream(s)
                else:
                    h.allreduce_fused(ins, outs, cap)
    torch.cuda.current_stream().wait_stream(side)
    for i in range(len(seq)):
        for r in range(R):
            ins_all[i][r].copy_(to_dev(xs_all[i][r], dtype))
    for rep in range(3):
        for o in outs_all:
            for t in o:
                t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for i, (form, launch, n) in enumerate(seq):
            _check(outs_all[i], xs_all[i], dtype, f"graph replay {rep} step {i} {form}/{launch}")
    del g
    h.destroy()


@pytest.mark.parametrize("all_fused", [0, 1])
def test_allreduce_all_orders_each_output_on_its_own_stream(all_fused):
    """Whether it fuses or not, each rank's output is ready on that rank's
    stream: work enqueued on streams[r] after the call sees rank r's result."""
    import tensor_decode_all_gb300 as tda
    R, n, dtype = 4, 262147, "f16"
    h = tda.Handle(R, torch.float16, n, "hbm")
    h.set_tactics(all_fused=all_fused)
    streams = rank_streams(R)
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 3)
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    copies = [torch.empty_like(t) for t in ins]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(5):
        h.allreduce_all(ins, outs, streams)
        for r in range(R):
            with torch.cuda.stream(streams[r]):
                copies[r].copy_(outs[r])         # ordered by streams[r] alone
    for s in streams:
        s.synchronize()
    h.check()
    _check(copies, xs, dtype, f"all_fused={all_fused}")
    h.destroy()


def test_allreduce_all_declines():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    R, n = 2, 64
    h = tda.Handle(R, torch.float16, n, "hbm")
    a = torch.zeros(n, dtype=torch.float16, device="cuda")
    s0, s1 = rank_streams(2)
    p = [a.data_ptr()] * 2
    assert ar.ar_allreduce_all(h.ptr, p, p, n + 1, [s0.cuda_stream, s1.cuda_stream]) == ar.AR_ETOOBIG
    assert ar.ar_allreduce_all(h.ptr, p, p, n, [s0.cuda_stream, s0.cuda_stream]) == ar.AR_ESTREAM
    assert ar.ar_allreduce_all(h.ptr, p, p, n, [s0.cuda_stream, 0]) == ar.AR_ESTREAM
    assert ar.ar_allreduce_all(h.ptr, [a.data_ptr() + 2, a.data_ptr()], p, n,
                               [s0.cuda_stream, s1.cuda_stream]) == ar.AR_EINVAL
    # one stream capturing, the other not: refused, nothing enqueued
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s0):
        rc = ar.ar_allreduce_all(h.ptr, p, p, n, [s0.cuda_stream, s1.cuda_stream])
    assert rc == ar.AR_ESTREAM
    del g
    torch.cuda.synchronize()
    hc = tda.Handle(2, torch.complex64, 16, "hbm")
    assert ar.ar_allreduce_all(hc.ptr, p, p, 16, [s0.cuda_stream, s1.cuda_stream]) == ar.AR_EINVAL
    hc.destroy()
    # the handle is still in step: a normal call completes
    xs = inputs.allreduce_inputs(5, R, n, "f16", "uniform", 1)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    for s in (s0, s1):
        s.wait_stream(torch.cuda.current_stream())
    h.allreduce_all(ins, outs, [s0, s1])
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs, "f16", "after declines")
    h.destroy()


def test_cluster_trace_records():
    """Traced cluster calls write one record per (rank, block) with the
    cluster form's code, and every cluster's blocks overlap in time."""
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import trace
    R, n, dtype = 8, 393216, "bf16"
    h = _handle(R, dtype, n, "hbm")
    buf = trace.start(h, 4)
    xs = inputs.allreduce_inputs(3, R, n, dtype, "normal", 0)
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    one = torch.cuda.Stream()
    for _ in range(3):
        _fused(h, ins, outs, one)
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs, dtype, "traced cluster")
    rec = trace.records(buf)
    live = rec[rec["t_end_ns"] != 0]
    blocks = h.plan("allreduce_fused", n).blocks
    assert len(live) == 3 * R * blocks
    assert (live["algo"] == 3).all()
    summary = trace.summarize(rec, 2000.0)
    assert summary["overlap_violations"] == 0
    h.destroy()


@pytest.mark.parametrize("pdl", [False, True])
def test_cluster_with_and_without_programmatic_launch(pdl):
    R, n, dtype, C = 8, 50001, "bf16", 6
    h = _handle(R, dtype, n, "hbm", cluster_twoshot_min_bytes=0)
    h.set_pdl(pdl)
    xs_all = [inputs.allreduce_inputs(5, R, n, dtype, "uniform", 300 + c) for c in range(C)]
    ins = [[to_dev(x, dtype) for x in xs] for xs in xs_all]
    outs = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(C)]
    one = torch.cuda.Stream()
    one.wait_stream(torch.cuda.current_stream())
    for c in range(C):
        h.allreduce_fused(ins[c], outs[c], one)
    torch.cuda.current_stream().wait_stream(one)
    torch.cuda.synchronize()
    h.check()
    for c in range(C):
        _check(outs[c], xs_all[c], dtype, f"pdl={pdl} call {c}")
    h.destroy()
