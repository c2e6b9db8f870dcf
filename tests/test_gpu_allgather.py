"""GPU parity of the allgather against the CPU oracle (byte-exact)."""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle(R, n, slots, dtype=torch.complex64):
    import tensor_decode_all_gb300 as tda
    return tda.Handle(R, dtype, n, slots)


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("R", [4, 8])
def test_config4_c64_1000x500_graph(R, slots):
    """Workload 4: complex64 1000x500 shards, graph-replayed, refilled inputs."""
    n, C, REPLAYS = 1000 * 500, 4, 3
    h = _handle(R, n, slots)
    streams = rank_streams(R)
    ins = [[torch.empty(n, dtype=torch.complex64, device="cuda") for _ in range(R)] for _ in range(C)]
    outs = [[torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)] for _ in range(C)]
    g = capture(h, "allgather", ins, outs, streams)
    for rep in range(REPLAYS):
        zs_all = []
        for c in range(C):
            zs = inputs.allgather_inputs(4, R, n, rep * C + c)
            for r in range(R):
                ins[c][r].copy_(to_dev(zs[r], "c64"))
            zs_all.append(zs)
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            want = oracle.allgather(zs_all[c], ranks=[0])[0]
            for r in range(R):
                assert_bits_equal(to_bits(outs[c][r]), want, "c64", f"rep {rep} call {c} rank {r}")
    del g
    h.destroy()


@pytest.mark.parametrize("R", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 2, 3, 17, 4096 + 1, 250001])
def test_odd_sizes(R, n):
    """Odd element counts make shard p start at an 8-byte (not 16-byte) offset."""
    zs = inputs.allgather_inputs(4, R, n, 5)
    h = _handle(R, n, "hbm")
    ins = [to_dev(z, "c64") for z in zs]
    outs = [torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)]
    enqueue(h, "allgather", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    want = oracle.allgather(zs, ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, "c64", f"rank {r}")
    h.destroy()


@pytest.mark.parametrize("n", [1, 3, 5, 1001])
def test_fp16_allgather_narrow_vectors(n):
    """A 2-byte dtype with odd numel takes the 2-byte vector path."""
    R = 3
    rng = np.random.default_rng(n)
    xs = [rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16) for _ in range(R)]
    h = _handle(R, n, "pinned", torch.float16)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty(R * n, dtype=torch.float16, device="cuda") for _ in range(R)]
    enqueue(h, "allgather", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    want = oracle.allgather(xs, ranks=[0])[0].view(np.uint16)
    for r in range(R):
        assert np.array_equal(to_bits(outs[r]), want)
    h.destroy()
