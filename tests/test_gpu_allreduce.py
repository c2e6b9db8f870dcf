"""GPU parity of the all-reduce against the CPU oracle (bit-exact).

The oracle's result is unique (fixed rank order, one rounding), so every
element of every rank must match its bits; only NaN payloads are exempt.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, enqueue, generate, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle(R, dtype, max_numel, slots):
    import tensor_decode_all_gb300 as tda
    return tda.Handle(R, {"f16": torch.float16, "bf16": torch.bfloat16}[dtype], max_numel, slots)


def _run_once(R, dtype, numel, slots, dist="uniform", config=5, call=0, h=None, algo=None):
    xs = inputs.allreduce_inputs(config, R, numel, dtype, dist, call)
    own = h is None
    h = h or _handle(R, dtype, max(numel, 1), slots)
    if algo is not None:
        h.set_algo(algo)
    streams = rank_streams(R)
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    enqueue(h, "allreduce", ins, outs, streams)
    torch.cuda.synchronize()
    h.check()
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, dtype, f"R={R} {dtype} n={numel} {slots} rank {r}")
    if own:
        h.destroy()


def test_config1_r2_fp16_4096_pinned_fresh_inputs_every_call():
    """Workload 1: 100 eager calls, fresh inputs each call; every call, both
    ranks equal the oracle, which equals RNE16(a + b) (the two-rank closed form)."""
    R, n = 2, 4096
    h = _handle(R, "f16", n, "pinned")
    streams = rank_streams(R)
    for call in range(100):
        xs = inputs.allreduce_inputs(1, R, n, "f16", "uniform", call)
        ins = [to_dev(x, "f16") for x in xs]
        outs = [torch.empty_like(t) for t in ins]
        enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        want = oracle.allreduce(xs, "f16", ranks=[0])[0]
        closed = (xs[0].view(np.float16).astype(np.float64)
                  + xs[1].view(np.float16).astype(np.float64)).astype(np.float16).view(np.uint16)
        assert np.array_equal(want, closed)
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, "f16", f"call {call} rank {r}")
    h.check()
    h.destroy()


@pytest.mark.parametrize("slots", ["pinned", "hbm"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 8])
def test_ranks_dtypes_slots(R, dtype, slots):
    # several tiles per block, plus a ragged tail of 5 elements
    _run_once(R, dtype, 256 * 8 * 2 * 7 + 5, slots)


@pytest.mark.parametrize("numel", [1, 2, 7, 8, 9, 15, 2047, 2048, 2049, 4095, 65536 + 3, 1000003])
def test_edge_sizes(numel):
    _run_once(4, "bf16", numel, "hbm")
    _run_once(2, "f16", numel, "pinned")
    _run_once(8, "bf16", numel, "hbm", algo="twoshot")
    _run_once(5, "f16", numel, "pinned", algo="twoshot")


@pytest.mark.parametrize("slots", ["pinned", "hbm"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 6, 8])
def test_twoshot_forced(R, dtype, slots):
    """The two-shot form reduces each sub-tile once, in rank order, on one
    rank: the same bits as the oracle (several stages, ragged tail)."""
    _run_once(R, dtype, 256 * 8 * R * 5 + 3, slots, algo="twoshot")


def test_auto_picks_twoshot_at_16MiB_r8():
    import tensor_decode_all_gb300 as tda
    R, n = 8, 8 << 20
    h = _handle(R, "bf16", n, "hbm")
    assert h.plan("allreduce", n).algo == tda.ar.AR_ALGO_TWOSHOT
    assert h.plan("allreduce", 4096).algo == tda.ar.AR_ALGO_ONESHOT
    _run_once(R, "bf16", n, "hbm", h=h)
    h.destroy()


def test_oneshot_then_twoshot_on_one_handle():
    """Switching forms between calls keeps the counters and flags consistent."""
    R, n = 4, 300001
    h = _handle(R, "f16", n, "hbm")
    for k, algo in enumerate(["oneshot", "twoshot", "twoshot", "oneshot", "twoshot"]):
        _run_once(R, "f16", n, "hbm", call=k, h=h, algo=algo)
    h.destroy()


def test_max_numel_exactly_and_one_over():
    import tensor_decode_all_gb300 as tda
    n = 12345
    h = _handle(2, "f16", n, "hbm")
    _run_once(2, "f16", n, "hbm", h=h)
    t = torch.zeros(n + 8, dtype=torch.float16, device="cuda")
    s = rank_streams(2)
    rc = tda.ar_allreduce(h.ptr, 0, t.data_ptr(), t.data_ptr(), n + 1, s[0].cuda_stream)
    assert rc == tda.ar.AR_ETOOBIG
    h.destroy()


def _graph_run(R, dtype, n, slots, config, dist, C, REPLAYS, label):
    """C calls of all R ranks captured once (every call with its own input and
    output buffers, ranks on forked streams), replayed REPLAYS times with fresh
    inputs each replay; every call of every replay compared with the oracle,
    bit for bit, on every rank (C * REPLAYS calls)."""
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    h = _handle(R, dtype, n, slots)
    streams = rank_streams(R)
    ins = torch.empty((C, R, n), dtype=tdt, device="cuda")
    outs = torch.empty((C, R, n), dtype=tdt, device="cuda")
    g = capture(h, "allreduce", [[ins[c, r] for r in range(R)] for c in range(C)],
                [[outs[c, r] for r in range(R)] for c in range(C)], streams)
    for rep in range(REPLAYS):
        xs_all = generate(inputs.allreduce_inputs, [(config, R, n, dtype, dist, rep * C + c) for c in range(C)])
        host = np.stack([np.stack(xs) for xs in xs_all]).view(np.int16)
        ins.copy_(torch.from_numpy(host).view(tdt))
        outs.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        want = generate(lambda xs: oracle.allreduce(xs, dtype, ranks=[0])[0], [(xs,) for xs in xs_all])
        got = to_bits(outs)
        for c in range(C):
            if not np.array_equal(got[c], np.broadcast_to(want[c], (R, n))):
                for r in range(R):
                    assert_bits_equal(got[c, r], want[c], dtype, f"{label} replay {rep} call {c} rank {r}")
    del g
    h.destroy()
    return C * REPLAYS


def test_config2_graph_1000_calls_double_buffered():
    """Workload 2: R=2 fp16 N=131072 pinned-host; a graph of 100 calls, each
    with its own input and output buffers, replayed 10 times with the inputs
    refilled between replays: 1000 calls, every one of them compared with the
    oracle on both ranks (both parities see different data)."""
    assert _graph_run(2, "f16", 131072, "pinned", 2, "normal4", 100, 10, "config 2") == 1000


def test_config3_r8_bf16_hbm_graph_1000_calls():
    """Workload 3: R=8, bf16, N=393216, HBM slots; a graph of 100 calls
    replayed 10 times with fresh inputs each replay: 1000 calls, every one
    compared with the oracle on all eight ranks."""
    assert _graph_run(8, "bf16", 393216, "hbm", 3, "normal", 100, 10, "config 3") == 1000


@pytest.mark.parametrize("algo", ["oneshot", "twoshot"])
def test_in_place(algo):
    R, n, dtype = 4, 70001, "bf16"
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 7)
    h = _handle(R, dtype, n, "hbm")
    h.set_algo(algo)
    bufs = [to_dev(x, dtype) for x in xs]
    enqueue(h, "allreduce", bufs, bufs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(bufs[r]), want, dtype, f"in place rank {r}")
    h.destroy()


def test_every_output_element_is_written():
    """Outputs pre-filled with a NaN sentinel; inputs hold no NaN, so no NaN may
    remain (a slot path that dropped data would also fail the oracle check)."""
    R, n = 2, 100003
    xs = inputs.allreduce_inputs(5, R, n, "f16", "uniform", 3)
    h = _handle(R, "f16", n, "pinned")
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.full((n,), float("nan"), dtype=torch.float16, device="cuda") for _ in range(R)]
    enqueue(h, "allreduce", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    for r in range(R):
        assert not torch.isnan(outs[r]).any()
    want = oracle.allreduce(xs, "f16", ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, "f16", f"rank {r}")
    h.destroy()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_special_values(dtype):
    """Random bit patterns: subnormals, infinities, NaNs, overflow."""
    R, n = 3, 50000
    rng = np.random.default_rng(99)
    xs = [rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16) for _ in range(R)]
    h = _handle(R, dtype, n, "hbm")
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    enqueue(h, "allreduce", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, dtype, f"rank {r}")
    h.destroy()


@pytest.mark.parametrize("slots", ["pinned", "hbm"])
def test_programmatic_dependent_launch_on_and_off_agree(slots):
    """A graph of back-to-back calls with each rank's kernels launched as
    programmatic dependents (the default) and without: same bits, equal to the
    oracle on every call."""
    R, n, C = 4, 50001, 12
    outs_by_mode = {}
    xs_all = [inputs.allreduce_inputs(5, R, n, "bf16", "uniform", 200 + c) for c in range(C)]
    for pdl in (True, False):
        h = _handle(R, "bf16", n, slots)
        h.set_pdl(pdl)
        streams = rank_streams(R)
        ins = [[to_dev(x, "bf16") for x in xs] for xs in xs_all]
        outs = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(C)]
        g = capture(h, "allreduce", ins, outs, streams)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        h.check()
        outs_by_mode[pdl] = [[to_bits(t) for t in row] for row in outs]
        del g
        h.destroy()
    for c in range(C):
        want = oracle.allreduce(xs_all[c], "bf16", ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(outs_by_mode[True][c][r], want, "bf16", f"pdl on, call {c} rank {r}")
            assert_bits_equal(outs_by_mode[False][c][r], want, "bf16", f"pdl off, call {c} rank {r}")


@pytest.mark.parametrize("sub", [64, 128, 256])
@pytest.mark.parametrize("R,slots", [(3, "hbm"), (4, "pinned"), (8, "hbm"), (8, "pinned")])
def test_twoshot_subtile_sizes(sub, R, slots, monkeypatch):
    """Every two-shot sub-tile size gives the oracle's bits (several stages,
    partial last tile, ragged tail)."""
    monkeypatch.setenv("AR_TWOSHOT_SUB", str(sub))
    n = 8 * sub * R * 7 + 8 * 37 + 5
    h = _handle(R, "bf16", n, slots)
    h.set_algo("twoshot")
    assert h.plan("allreduce", n).subtile_vecs == sub
    _run_once(R, "bf16", n, slots, h=h)
    h.destroy()
