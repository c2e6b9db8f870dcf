"""Declines, the bounded device wait, reset, and long call sequences.

The timeout test launches only one rank of a two-rank handle: its kernel
waits on a flag that nothing raises, gives up after a short limit, records
AR_ETIMEOUT and returns.  The GPU stays usable; nothing traps or hangs.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import BlockingStream, assert_bits_equal, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _tda():
    import tensor_decode_all_gb300 as tda
    return tda


def test_declines_enqueue_nothing_and_return_codes():
    tda = _tda()
    ar = tda.ar
    n = 1024
    h = tda.Handle(2, torch.float16, n, "hbm")
    a = torch.zeros(n + 64, dtype=torch.float16, device="cuda")
    b = torch.zeros(n + 64, dtype=torch.float16, device="cuda")
    s0, s1 = rank_streams(2)
    p, q = a.data_ptr(), b.data_ptr()
    assert tda.ar_allreduce(h.ptr, 0, p, q, n + 1, s0.cuda_stream) == ar.AR_ETOOBIG
    assert tda.ar_allreduce(h.ptr, 2, p, q, n, s0.cuda_stream) == ar.AR_EINVAL
    assert tda.ar_allreduce(h.ptr, -1, p, q, n, s0.cuda_stream) == ar.AR_EINVAL
    assert tda.ar_allreduce(h.ptr, 0, p + 2, q, n, s0.cuda_stream) == ar.AR_EINVAL   # misaligned
    assert tda.ar_allreduce(h.ptr, 0, p, q + 8, n, s0.cuda_stream) == ar.AR_EINVAL
    assert tda.ar_allreduce(h.ptr, 0, 0, q, n, s0.cuda_stream) == ar.AR_EINVAL
    assert tda.ar_allreduce(h.ptr, 0, p, q, n, 0) == ar.AR_ESTREAM                   # legacy default
    assert tda.ar_allreduce(h.ptr, 0, p, q, n, 1) == ar.AR_ESTREAM                   # cudaStreamLegacy
    assert tda.ar_allreduce(h.ptr, 0, p, q, n, 2) == ar.AR_ESTREAM                   # per-thread default
    assert tda.ar_allreduce(0, 0, p, q, n, s0.cuda_stream) == ar.AR_EINVAL
    assert tda.ar_allreduce(h.ptr, 0, p, q, 0, s0.cuda_stream) == ar.AR_OK           # nothing to do
    assert tda.ar_allgather(h.ptr, 0, p, q, 0, s0.cuda_stream) == ar.AR_OK
    torch.cuda.synchronize()
    assert h.status().code == 0
    # a complex64 handle has no all-reduce
    hc = tda.Handle(2, torch.complex64, 16, "hbm")
    assert tda.ar_allreduce(hc.ptr, 0, p, q, 16, s0.cuda_stream) == ar.AR_EINVAL
    hc.destroy()
    # the handle still works after all the declines
    xs = inputs.allreduce_inputs(5, 2, n, "f16", "uniform", 1)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    enqueue(h, "allreduce", ins, outs, [s0, s1])
    torch.cuda.synchronize()
    want = oracle.allreduce(xs, "f16", ranks=[0])[0]
    for r in range(2):
        assert_bits_equal(to_bits(outs[r]), want, "f16")
    h.destroy()


def test_same_stream_for_two_ranks_is_refused():
    tda = _tda()
    n = 256
    h = tda.Handle(2, torch.float16, n, "hbm")
    a = torch.zeros(n, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    # rank 0's call would wait for rank 1, which would sit behind it on s
    # forever; a bounded wait would end it, but the library refuses up front.
    h.set_timeout(20_000_000)
    assert tda.ar_allreduce(h.ptr, 0, a.data_ptr(), a.data_ptr(), n, s.cuda_stream) == 0
    assert tda.ar_allreduce(h.ptr, 1, a.data_ptr(), a.data_ptr(), n, s.cuda_stream) == tda.ar.AR_ESTREAM
    torch.cuda.synchronize()
    # rank 0 waited for a rank-1 call that never came: the bounded wait ended it
    assert h.status().code == tda.ar.AR_ETIMEOUT
    h.reset()
    h.destroy()


def test_blocking_stream_is_refused():
    """A blocking stream serialises with the legacy stream, which can hold back
    a peer rank while this rank's kernel waits for it ("fix(group): run each
    rank on a non-blocking stream", sections "What" and "Why"): refused, with
    nothing enqueued, for the per-rank and the fused calls alike."""
    tda = _tda()
    bs = BlockingStream()
    try:
        assert bs.flags() & 1 == 0          # cudaStreamNonBlocking not set
        h = tda.Handle(2, torch.float16, 64, "hbm")
        a = torch.zeros(64, dtype=torch.float16, device="cuda")
        assert tda.ar_allreduce(h.ptr, 0, a.data_ptr(), a.data_ptr(), 64, bs.handle) == tda.ar.AR_ESTREAM
        assert tda.ar_allgather(h.ptr, 0, a.data_ptr(), a.data_ptr(), 32, bs.handle) == tda.ar.AR_ESTREAM
        assert tda.ar.ar_allreduce_fused(h.ptr, [a.data_ptr()] * 2, [a.data_ptr()] * 2, 64,
                                         bs.handle) == tda.ar.AR_ESTREAM
        torch.cuda.synchronize()
        assert h.status().code == tda.ar.AR_OK
        # nothing was counted: a normal call pair still completes
        s0, s1 = rank_streams(2)
        xs = inputs.allreduce_inputs(5, 2, 64, "f16", "uniform", 3)
        ins = [to_dev(x, "f16") for x in xs]
        outs = [torch.empty_like(t) for t in ins]
        enqueue(h, "allreduce", ins, outs, [s0, s1])
        torch.cuda.synchronize()
        h.check()
        want = oracle.allreduce(xs, "f16", ranks=[0])[0]
        for r in range(2):
            assert_bits_equal(to_bits(outs[r]), want, "f16")
        h.destroy()
    finally:
        bs.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
def test_missing_peer_times_out_and_reset_restores(slots):
    tda = _tda()
    ar = tda.ar
    R, n = 2, 8192
    h = tda.Handle(R, torch.float16, n, slots)
    h.set_timeout(50_000_000)  # 50 ms
    streams = rank_streams(R)
    xs = inputs.allreduce_inputs(5, R, n, "f16", "uniform", 11)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h.allreduce(0, ins[0], outs[0], streams[0])      # rank 1 never called
    streams[0].synchronize()
    dt = time.perf_counter() - t0
    st = h.status()
    assert st.code == ar.AR_ETIMEOUT
    assert st.rank == 0 and st.peer == 1
    assert st.want >= 1 and st.seen == 0
    assert 0.04 < dt < 5.0, dt
    # the handle refuses work until reset
    assert tda.ar_allreduce(h.ptr, 1, ins[1].data_ptr(), outs[1].data_ptr(), n,
                            streams[1].cuda_stream) == ar.AR_ESTATE
    h.reset()
    assert h.status().code == ar.AR_OK
    enqueue(h, "allreduce", ins, outs, streams)
    torch.cuda.synchronize()
    h.check()
    want = oracle.allreduce(xs, "f16", ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, "f16", f"after reset rank {r}")
    h.destroy()


def test_ten_thousand_calls_rotating_buffers():
    """10^4 back-to-back eager calls; inputs and outputs rotate over 7 buffer
    sets (7 is odd, so each set meets both slot parities)."""
    tda = _tda()
    R, n, K, CALLS = 3, 3000, 7, 10000
    h = tda.Handle(R, torch.bfloat16, n, "hbm")
    streams = rank_streams(R)
    xs = [inputs.allreduce_inputs(5, R, n, "bf16", "uniform", 100 + k) for k in range(K)]
    ins = [[to_dev(x, "bf16") for x in xk] for xk in xs]
    outs = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(K)]
    cur = torch.cuda.current_stream()
    for s in streams:
        s.wait_stream(cur)
    for c in range(CALLS):
        k = c % K
        for r in range(R):
            h.allreduce(r, ins[k][r], outs[k][r], streams[r])
    for s in streams:
        cur.wait_stream(s)
    torch.cuda.synchronize()
    h.check()
    for k in range(K):
        want = oracle.allreduce(xs[k], "bf16", ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[k][r]), want, "bf16", f"set {k} rank {r}")
    h.destroy()


def test_query_and_plan():
    tda = _tda()
    h = tda.Handle(8, torch.bfloat16, 393216, "hbm")
    info = h.info()
    assert info.R == 8 and info.max_blocks >= 1
    bps = (info.blocks_per_sm, info.blocks_per_sm_twoshot, info.blocks_per_sm_allgather)
    assert min(bps) >= 1
    assert info.max_blocks * 8 <= info.sm_count * max(bps)
    assert info.slot_bytes == 393216 * 2
    assert info.total_slot_bytes == 2 * 8 * info.slot_bytes
    p = h.plan("allreduce", 393216)
    assert p.algo == tda.ar_choose_algo(8, 393216 * 2, tda.AR_SLOT_HBM)
    h.set_algo("oneshot")
    p = h.plan("allreduce", 393216)
    assert p.algo == 0 and 1 <= p.blocks and p.blocks * 8 <= info.sm_count * info.blocks_per_sm
    assert p.tiles * p.tile_bytes >= 393216 * 2
    h.set_algo("twoshot")
    p = h.plan("allreduce", 393216)
    assert p.algo == 1 and p.flag_rounds == 2 and p.blocks * 8 <= info.sm_count * info.blocks_per_sm_twoshot
    # HBM slots: 128-vector sub-tiles when 256-vector ones would fill under half the blocks
    nv = 393216 // 8
    tiles256 = -(-nv // (256 * 8))
    bmax = info.sm_count * info.blocks_per_sm_twoshot // 8
    assert p.subtile_vecs == (128 if 2 * tiles256 < bmax else 256)
    h.destroy()
    # pinned-host slots: 64-vector sub-tiles while 256-vector ones make fewer than 8 tiles
    g = tda.Handle(8, torch.bfloat16, 1 << 20, "pinned")
    g.set_algo("twoshot")
    for n, sub in ((16384, 64), (65536, 64), (114688, 64), (114688 + 8, 256), (1 << 20, 256)):
        assert g.plan("allreduce", n).subtile_vecs == sub, n
    g.destroy()


def test_probes_run():
    tda = _tda()
    link = tda.ar_probe_host_link(64 << 20, 5)
    assert all(v > 1.0 for v in link.values()), link
    # both directions at once: each below its solo rate (with some slack for
    # noise), together above either alone
    assert link["bidir_write_gbs"] < 1.1 * link["write_gbs"], link
    assert link["bidir_read_gbs"] < 1.1 * link["read_gbs"], link
    assert link["bidir_write_gbs"] + link["bidir_read_gbs"] > max(link["write_gbs"], link["read_gbs"]), link
    assert tda.ar_probe_hbm_copy(1 << 30, 5) > 100.0


def test_link_latency_probe_is_ordered():
    """The latency probe's figures are positive and keep the order the
    hardware implies: an HBM flag at GPU scope is faster than a host-memory
    flag at system scope, a host round trip is slower than nothing, and the
    probe rejects nonsense repetition counts."""
    from tensor_decode_all_gb300 import ar
    tda = _tda()
    lat = tda.ar_probe_host_link_latency(100)
    assert all(20.0 < v < 1e6 for v in lat.values()), lat
    assert lat["flag_hbm_gpu_one_way_ns"] < lat["flag_host_sys_one_way_ns"], lat
    assert set(lat) == {"host_load_rtt_ns", "store_4KiB_fence_sys_ns", "flag_host_sys_one_way_ns",
                        "flag_hbm_gpu_one_way_ns", "store_4KiB_fence_gpu_ns"}, lat
    with pytest.raises(ar.ArError):
        tda.ar_probe_host_link_latency(0)


def test_one_host_thread_per_rank():
    """Each rank's calls enqueued from its own host thread, as separate
    processes would: the C ABI's host-side bookkeeping is thread-safe and every
    call still matches the oracle."""
    import threading
    tda = _tda()
    R, n, CALLS = 4, 20001, 50
    h = tda.Handle(R, torch.bfloat16, n, "hbm")
    streams = rank_streams(R)
    xs = [inputs.allreduce_inputs(5, R, n, "bf16", "uniform", 300 + c) for c in range(CALLS)]
    ins = [[to_dev(x, "bf16") for x in xc] for xc in xs]
    outs = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(CALLS)]
    torch.cuda.synchronize()
    errors = []

    def rank_thread(r):
        try:
            for c in range(CALLS):
                h.allreduce(r, ins[c][r], outs[c][r], streams[r])
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=rank_thread, args=(r,)) for r in range(R)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    h.check()
    for c in (0, CALLS // 2, CALLS - 1):
        want = oracle.allreduce(xs[c], "bf16", ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[c][r]), want, "bf16", f"call {c} rank {r}")
    h.destroy()


def test_allreduce_and_allgather_interleaved_on_one_handle():
    """The two operations share a handle's counters and flags."""
    tda = _tda()
    R, n = 3, 10007
    h = tda.Handle(R, torch.float16, n, "pinned")
    streams = rank_streams(R)
    for k in range(6):
        xs = inputs.allreduce_inputs(5, R, n, "f16", "uniform", 400 + k)
        ins = [to_dev(x, "f16") for x in xs]
        if k % 2 == 0:
            outs = [torch.empty_like(t) for t in ins]
            enqueue(h, "allreduce", ins, outs, streams)
            want = oracle.allreduce(xs, "f16", ranks=[0])[0]
        else:
            outs = [torch.empty(R * n, dtype=torch.float16, device="cuda") for _ in range(R)]
            enqueue(h, "allgather", ins, outs, streams)
            want = oracle.allgather(xs, ranks=[0])[0].view(np.uint16)
        torch.cuda.synchronize()
        h.check()
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, "f16", f"step {k} rank {r}")
    h.destroy()
