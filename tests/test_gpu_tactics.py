"""Per-handle tactics, ar_supports, and the tuner, on the GPU."""
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


def test_supports_matches_what_the_enqueue_calls_accept():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    n = 4096
    h = tda.Handle(2, torch.float16, n, "hbm")
    a = torch.zeros(n, dtype=torch.float16, device="cuda")
    b = torch.empty_like(a)
    assert h.supports("allreduce", a, b) == ar.AR_OK
    assert h.supports("allgather", a, torch.empty(2 * n, dtype=torch.float16, device="cuda")) == ar.AR_OK
    big = torch.zeros(n + 8, dtype=torch.float16, device="cuda")
    assert h.supports("allreduce", big, torch.empty_like(big)) == ar.AR_ETOOBIG
    assert ar.ar_supports(h.ptr, 0, n - 1, a.data_ptr() + 2, b.data_ptr()) == ar.AR_EINVAL
    assert ar.ar_supports(h.ptr, 0, n, 0, b.data_ptr()) == ar.AR_EINVAL
    assert ar.ar_supports(h.ptr, 0, 0, 0, 0) == ar.AR_OK
    assert ar.ar_supports(h.ptr, 2, n, a.data_ptr(), b.data_ptr()) == ar.AR_EINVAL
    assert ar.ar_supports(0, 0, n, a.data_ptr(), b.data_ptr()) == ar.AR_EINVAL
    g = tda.Handle(2, torch.complex64, 16, "hbm")
    assert ar.ar_supports(g.ptr, 0, 16, a.data_ptr(), b.data_ptr()) == ar.AR_EINVAL
    assert ar.ar_supports(g.ptr, 1, 16, a.data_ptr(), b.data_ptr()) == ar.AR_OK
    g.destroy()
    h.destroy()


def test_tactics_default_to_the_builtin_table_and_steer_auto():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    n = 4 << 20
    h = tda.Handle(8, torch.bfloat16, n, "hbm")
    t = h.tactics()
    assert t["twoshot_min_bytes"] == 512 << 10 and t["twoshot_sub"] == 0 and t["max_blocks"] == 0
    assert h.plan("allreduce", 128 << 10).algo == ar.AR_ALGO_ONESHOT       # 256 KiB per rank
    assert h.plan("allreduce", 256 << 10).algo == ar.AR_ALGO_TWOSHOT       # 512 KiB per rank
    h.set_tactics(twoshot_min_bytes=2 << 20)
    assert h.plan("allreduce", 512 << 10).algo == ar.AR_ALGO_ONESHOT       # 1 MiB per rank
    assert h.plan("allreduce", 1 << 20).algo == ar.AR_ALGO_TWOSHOT         # 2 MiB per rank
    h.set_tactics(twoshot_sub=64)
    assert h.plan("allreduce", 1 << 20).subtile_vecs == 64
    h.set_tactics(max_blocks=5)
    p = h.plan("allreduce", 1 << 20)
    assert p.blocks == 5 and p.max_stages == (p.tiles + 4) // 5
    with pytest.raises(ar.ArError):
        h.set_tactics(twoshot_sub=96)
    with pytest.raises(ar.ArError):
        h.set_tactics(max_blocks=-1)
    h.destroy()
    assert tda.Handle(2, torch.float16, 64, "pinned").tactics()["twoshot_min_bytes"] == (1 << 64) - 1


@pytest.mark.parametrize("R,slots,algo", [(8, "hbm", "twoshot"), (4, "pinned", "oneshot"), (3, "hbm", "oneshot")])
def test_capped_grid_stays_exact(R, slots, algo):
    """A block cap forces many stages per block; the bits do not change."""
    import tensor_decode_all_gb300 as tda
    n = (1 << 19) + 7
    xs = inputs.allreduce_inputs(5, R, n, "bf16", "uniform", 3)
    h = tda.Handle(R, torch.bfloat16, n, slots)
    h.set_algo(algo)
    h.set_tactics(max_blocks=3)
    assert h.plan("allreduce", n).blocks == 3
    ins = [to_dev(x, "bf16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    for _ in range(2):   # both slot parities
        enqueue(h, "allreduce", ins, outs, rank_streams(R))
        torch.cuda.synchronize()
        h.check()
        want = oracle.allreduce(xs, "bf16", ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, "bf16", f"capped R={R} {slots} {algo} rank {r}")
    h.destroy()


def test_tune_sets_a_measured_threshold_and_the_file_applies_it(tmp_path):
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import tune
    h = tda.Handle(8, torch.bfloat16, 1 << 20, "hbm")
    out = tune.tune(h, sizes=[64 << 10, 256 << 10, 1 << 20], tagged_sizes=[4 << 10, 16 << 10],
                    cluster_sizes=[8 << 10, 512 << 10, 2 << 20], replays=3)
    thr = out["tactics"]["twoshot_min_bytes"]
    assert thr in (64 << 10, 256 << 10, 1 << 20, tune.NEVER)
    assert thr == tune.crossover({int(k): v for k, v in out["times_us"].items()})
    lim = out["tactics"]["tagged_max_bytes"]
    assert lim in (0, 4 << 10, 16 << 10)
    assert lim == tune.tagged_limit({int(k): v for k, v in out["tagged_times_us"].items()})
    assert h.tactics()["twoshot_min_bytes"] == thr
    if h.info().cluster_form > 0:
        ct = {int(k): v for k, v in out["cluster_times_us"].items()}
        assert sorted(ct) == [8 << 10, 512 << 10, 2 << 20]
        tw, cl = tune.cluster_tactics(ct)
        assert (out["tactics"]["cluster_twoshot_min_bytes"], out["tactics"]["cluster_max_bytes"]) == (tw, cl)
    assert h.info().algo == -1                       # the forced form was restored to AUTO
    path = str(tmp_path / "tactics.json")
    tune.save(path, tune.handle_key(h), h.tactics())
    g = tda.Handle(8, torch.bfloat16, 1 << 20, "hbm")
    g.set_tactics(twoshot_min_bytes=12345 * 16, tagged_max_bytes=16)
    assert tune.load(path, g) and g.tactics()["twoshot_min_bytes"] == thr
    assert g.tactics()["tagged_max_bytes"] == lim
    k = tda.Handle(4, torch.bfloat16, 1 << 20, "hbm")
    assert not tune.load(path, k)
    for x in (h, g, k):
        x.destroy()


def test_tune_measures_the_pace_of_a_pinned_handle():
    """Over the host link the tuner also times each pace on a call of one
    stage per block and on one of several, and keeps the fastest of each."""
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import tune
    h = tda.Handle(2, torch.float16, 2 << 20, "pinned")
    out = tune.tune(h, sizes=[256 << 10, 1 << 20], tagged_sizes=[4 << 10], cluster_sizes=[], replays=3)
    pt = out["pace_times_us"]
    assert set(pt) == {"single", "multi"}
    assert pt["single"]["bytes"] == 1 << 20 and pt["multi"]["bytes"] == 2 << 20
    for kind, field in (("single", "pace_mbs"), ("multi", "pace_multi_mbs")):
        us = {int(k): v for k, v in pt[kind]["us"].items()}
        assert sorted(us) == sorted(tune.PACES) and all(v > 0 for v in us.values())
        assert out["tactics"][field] == tune.best_pace(us) == h.tactics()[field]
    h.destroy()


def test_settings_are_refused_while_a_call_is_half_issued():
    """Between the ranks' halves of one call the form, the tactics and the
    trace setting stay as they are (changed there, the ranks of the call
    would run different kernels); once the call is complete they change
    again.  Everything is allocated before rank 0's kernel is enqueued, so
    nothing on the host waits for it while rank 1's half is outstanding."""
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar, trace
    R, n = 2, 65536
    xs = inputs.allreduce_inputs(5, R, n, "f16", "uniform", 8)
    h = tda.Handle(R, torch.float16, n, "hbm")
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    info = h.info()
    depth = 2
    buf = torch.zeros(depth * R * info.max_blocks * trace.RECORD_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    streams = rank_streams(R)
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    before = h.tactics()
    h.allreduce(0, ins[0], outs[0], streams[0])
    assert ar.ar_set_algo(h.ptr, ar.AR_ALGO_TWOSHOT) == ar.AR_EINVAL
    t = ar.ar_get_tactics(h.ptr)
    t.max_blocks = 2
    assert ar.ar_set_tactics(h.ptr, t) == ar.AR_EINVAL
    assert ar.lib().ar_set_trace(h.ptr, buf.data_ptr(), depth * R * info.max_blocks) == ar.AR_EINVAL
    h.allreduce(1, ins[1], outs[1], streams[1])   # completes the call
    for s in streams:
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    h.check()
    want = oracle.allreduce(xs, "f16", ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, "f16", f"rank {r}")
    assert h.tactics() == before and h.info().algo == ar.AR_ALGO_AUTO
    assert (buf == 0).all()
    h.set_algo("twoshot")
    h.set_tactics(max_blocks=2)
    h.set_trace(buf, depth * R * info.max_blocks)
    h.set_trace(None, 0)
    h.destroy()
