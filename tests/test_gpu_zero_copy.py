"""Inputs and outputs in pinned host memory (zero copy through ar_allreduce).

Mapped pinned host memory is device-accessible, so a caller may hand the
library host tensors directly: each rank's kernel then reads its input from
and writes its output to host memory.  Every form must still give the
oracle's bits.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, enqueue, rank_streams

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _host(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH[dtype]).pin_memory()


@pytest.mark.parametrize("R,dtype,n,slots,algo,fused", [
    (2, "f16", 131072, "pinned", None, False),
    (2, "f16", 4096, "pinned", None, False),        # tagged words
    (4, "bf16", 300001, "hbm", None, False),
    (8, "bf16", 393216, "hbm", None, False),        # two-shot
    (8, "bf16", 393216, "hbm", None, True),
    (3, "bf16", 65536, "pinned", "oneshot", True),
])
def test_host_buffers_directly(R, dtype, n, slots, algo, fused):
    import tensor_decode_all_gb300 as tda
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 21)
    h = tda.Handle(R, TORCH[dtype], n, slots)
    if algo:
        h.set_algo(algo)
    ins = [_host(x, dtype) for x in xs]
    outs = [torch.empty(n, dtype=TORCH[dtype]).pin_memory() for _ in range(R)]
    if fused:
        s = torch.cuda.Stream()
        h.allreduce_fused(ins, outs, s)
        s.synchronize()
    else:
        enqueue(h, "allreduce", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r in range(R):
        got = outs[r].view(torch.int16).numpy().view(np.uint16)
        assert_bits_equal(got, want, dtype, f"zero copy R={R} {dtype} n={n} {slots} rank {r}")
    h.destroy()


@pytest.mark.parametrize("launch", ["rank", "all"])
@pytest.mark.parametrize("R,dtype,n", [(2, "f16", 131072), (4, "bf16", 262144 + 3)])
def test_host_buffers_in_a_graph(launch, R, dtype, n):
    """Zero-copy calls of a size the handle paces, captured in a CUDA graph
    (the library asks the runtime whether the pointers are host memory, and
    runs such calls unpaced) and replayed with new inputs: the capture stays
    valid and every call of every replay equals the oracle."""
    import tensor_decode_all_gb300 as tda
    C = 4
    h = tda.Handle(R, TORCH[dtype], n, "pinned")
    assert h.plan("allreduce", n).pace_cycles > 0          # device pointers would be paced
    streams = rank_streams(R)
    ins = [[torch.empty(n, dtype=TORCH[dtype]).pin_memory() for _ in range(R)] for _ in range(C)]
    outs = [[torch.empty(n, dtype=TORCH[dtype]).pin_memory() for _ in range(R)] for _ in range(C)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            for s in streams:
                s.wait_stream(cap)
            for c in range(C):
                if launch == "all":
                    h.allreduce_all(ins[c], outs[c], streams)
                else:
                    for r in range(R):
                        h.allreduce(r, ins[c][r], outs[c][r], streams[r])
            for s in streams:
                cap.wait_stream(s)
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(2):
        xs = [inputs.allreduce_inputs(5, R, n, dtype, "uniform", 100 * rep + c) for c in range(C)]
        for c in range(C):
            for r in range(R):
                ins[c][r].copy_(torch.from_numpy(np.ascontiguousarray(xs[c][r]).view(np.int16)).view(TORCH[dtype]))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            want = oracle.allreduce(xs[c], dtype, ranks=[0])[0]
            for r in range(R):
                got = outs[c][r].view(torch.int16).numpy().view(np.uint16)
                assert_bits_equal(got, want, dtype, f"zero copy graph {launch} R={R} replay {rep} call {c} rank {r}")
    del g
    h.destroy()
