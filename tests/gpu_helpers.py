"""Helpers for the GPU tests: device buffers, rank streams, graph capture.

Nothing here computes the operation: expected values always come from the
CPU oracle (oracle/), inputs from tensor_decode_all_gb300.inputs.
"""
import ctypes
import ctypes.util
import glob
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "c64": torch.complex64}


def to_dev(bits_or_values, dtype):
    """numpy uint16 bit patterns (f16/bf16) or complex64 values -> CUDA tensor."""
    a = np.ascontiguousarray(bits_or_values)
    if dtype == "c64":
        return torch.from_numpy(a).cuda()
    return torch.from_numpy(a.view(np.int16)).view(TORCH_DT[dtype]).cuda()


def to_bits(t):
    """CUDA tensor -> numpy uint16 bit patterns (or uint8 bytes for complex64)."""
    t = t.detach().cpu()
    if t.dtype == torch.complex64:
        return t.numpy().view(np.uint8)
    return t.view(torch.int16).numpy().view(np.uint16)


def rank_streams(R):
    return [torch.cuda.Stream() for _ in range(R)]


def enqueue(h, op, ins, outs, streams):
    """Enqueue all R ranks, ordered after the current stream and joined back."""
    cur = torch.cuda.current_stream()
    for s in streams:
        s.wait_stream(cur)
    for r in range(len(streams)):
        getattr(h, op)(r, ins[r], outs[r], streams[r])
    for s in streams:
        cur.wait_stream(s)


def capture(h, op, ins_per_call, outs_per_call, streams):
    """One CUDA graph holding len(ins_per_call) calls of all R ranks, each rank
    on its own forked stream (fork from the capture stream, join back)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            for s in streams:
                s.wait_stream(cap)
            for ins, outs in zip(ins_per_call, outs_per_call):
                for r in range(len(streams)):
                    getattr(h, op)(r, ins[r], outs[r], streams[r])
            for s in streams:
                cap.wait_stream(s)
    torch.cuda.current_stream().wait_stream(side)
    return g


def nan_mask(bits, dtype):
    if dtype == "f16":
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def assert_bits_equal(got, want, dtype, what=""):
    """Bit-exact, except that NaN payloads are not compared (NaN-ness is)."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if dtype == "c64":
        assert np.array_equal(got, want), f"{what}: bytes differ"
        return
    gn, wn = nan_mask(got, dtype), nan_mask(want, dtype)
    bad = (gn != wn) | (~gn & (got != want))
    if bad.any():
        i = np.flatnonzero(bad)[:8]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first at {i.tolist()}: "
                             f"got {[hex(int(x)) for x in got[i]]} want {[hex(int(x)) for x in want[i]]}")


def cudart():
    """The CUDA runtime library through ctypes (the toolkit's, or the one the
    torch wheel ships), for the few runtime calls torch does not expose."""
    cands = [ctypes.util.find_library("cudart"), "libcudart.so.13", "libcudart.so",
             "/usr/local/cuda/lib64/libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"]
    torch_dir = os.path.dirname(torch.__file__)
    cands += sorted(glob.glob(os.path.join(os.path.dirname(torch_dir), "nvidia", "cu*", "lib", "libcudart.so*")))
    cands += sorted(glob.glob(os.path.join(os.path.dirname(torch_dir), "nvidia", "cuda_runtime", "lib",
                                           "libcudart.so*")))
    cands += sorted(glob.glob(os.path.join(torch_dir, "lib", "libcudart*.so*")))
    for c in cands:
        if not c:
            continue
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    raise RuntimeError("libcudart not found")


class BlockingStream:
    """A stream created with cudaStreamDefault flags (blocking: it serialises
    with the legacy default stream), which torch's stream pool never hands out."""

    def __init__(self):
        self.rt = cudart()
        self.rt.cudaStreamCreateWithFlags.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint]
        self.rt.cudaStreamCreateWithFlags.restype = ctypes.c_int
        self.rt.cudaStreamGetFlags.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint)]
        self.rt.cudaStreamGetFlags.restype = ctypes.c_int
        self.rt.cudaStreamDestroy.argtypes = [ctypes.c_void_p]
        self.rt.cudaStreamDestroy.restype = ctypes.c_int
        h = ctypes.c_void_p()
        rc = self.rt.cudaStreamCreateWithFlags(ctypes.byref(h), 0)
        if rc != 0:
            raise RuntimeError(f"cudaStreamCreateWithFlags: {rc}")
        self.handle = int(h.value)

    def flags(self) -> int:
        f = ctypes.c_uint()
        rc = self.rt.cudaStreamGetFlags(ctypes.c_void_p(self.handle), ctypes.byref(f))
        if rc != 0:
            raise RuntimeError(f"cudaStreamGetFlags: {rc}")
        return int(f.value)

    def destroy(self):
        if self.handle:
            self.rt.cudaStreamDestroy(ctypes.c_void_p(self.handle))
            self.handle = 0


def generate(fn, args_list, workers=8):
    """[fn(*a) for a in args_list], drawn on a thread pool (numpy's generators
    and torch's casts release the GIL): inputs of many calls in seconds."""
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda a: fn(*a), args_list))


def assert_device_equal(got, want_dev, what=""):
    """Bytes of a device tensor equal the bytes of the oracle's result (uploaded
    to the device): for outputs too large to copy back call by call."""
    g = got.reshape(-1).view(torch.uint8)
    w = want_dev.reshape(-1).view(torch.uint8)
    assert g.numel() == w.numel(), (what, g.numel(), w.numel())
    if not torch.equal(g, w):
        bad = torch.nonzero(g != w)[:8].reshape(-1).tolist()
        raise AssertionError(f"{what}: bytes differ from the oracle's at {bad}")
