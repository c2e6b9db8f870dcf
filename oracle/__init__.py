"""CPU oracle for the logical-rank all-reduce and allgather.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The CUDA
library (``tensor_decode_all_gb300``) never imports it, and it never imports
the CUDA library; the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, built here with gcc).  This
module only compiles it and marshals numpy arrays through ctypes.

What the oracle computes is stated in ``oracle.c``: the fp32 rank-order sum
with one round-to-nearest-even rounding to fp16/bf16 ("[Kernel] Two-rank FP16
all-reduce through pinned host memory for GPUs without P2P", section
"Purpose"), and the rank-major concatenation for allgather ("fix(group): run
each rank on a non-blocking stream", section "What").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16 = 1
BF16 = 2
_FMT = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (IEEE-exact flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no libgomp: the single-threaded oracle is still complete
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp = ctypes.c_void_p
            lib.oracle_allreduce.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp),
                                             ctypes.POINTER(vp), ctypes.c_size_t, ctypes.c_int]
            lib.oracle_allreduce.restype = ctypes.c_int
            lib.oracle_allgather.argtypes = [ctypes.c_int, ctypes.POINTER(vp),
                                             ctypes.POINTER(vp), ctypes.c_size_t]
            lib.oracle_allgather.restype = ctypes.c_int
            lib.oracle_widen_array.argtypes = [ctypes.c_int, vp, vp, ctypes.c_size_t]
            lib.oracle_narrow_array.argtypes = [ctypes.c_int, vp, vp, ctypes.c_size_t]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def fmt_code(fmt) -> int:
    if isinstance(fmt, int):
        return fmt
    return _FMT[str(fmt).lower()]


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data if a is not None else None for a in arrs])


def allreduce(ins, fmt, nthreads: int = 1, ranks=None):
    """Rank-order fp32 sum with one rounding.

    ``ins``: list of R uint16 arrays (bit patterns), all of one length n.
    Returns a list of uint16 arrays, one per rank in ``ranks`` (default: every
    rank); by the definition they are identical, and each is computed on its own.
    """
    lib = _load()
    ins = [np.ascontiguousarray(a, dtype=np.uint16).reshape(-1) for a in ins]
    R = len(ins)
    n = ins[0].size
    if any(a.size != n for a in ins):
        raise ValueError("all ranks must hold the same number of elements")
    ranks = list(range(R)) if ranks is None else list(ranks)
    outs = [np.empty(n, np.uint16) if r in ranks else None for r in range(R)]
    rc = lib.oracle_allreduce(R, fmt_code(fmt), _ptrs(ins), _ptrs(outs), n, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_allreduce rejected its arguments")
    return [outs[r] for r in ranks]


def allgather(ins, ranks=None):
    """Rank-major concatenation of R shards of equal byte size (any dtype)."""
    lib = _load()
    ins = [np.ascontiguousarray(a).reshape(-1).view(np.uint8) for a in ins]
    R = len(ins)
    nbytes = ins[0].size
    if any(a.size != nbytes for a in ins):
        raise ValueError("all shards must have the same size")
    ranks = list(range(R)) if ranks is None else list(ranks)
    outs = [np.empty(R * nbytes, np.uint8) if r in ranks else None for r in range(R)]
    rc = lib.oracle_allgather(R, _ptrs(ins), _ptrs(outs), nbytes)
    if rc != 0:
        raise ValueError("oracle_allgather rejected its arguments")
    return [outs[r] for r in ranks]


def widen(fmt, bits):
    """16-bit patterns -> float32 values, by the oracle's own conversion."""
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16).reshape(-1)
    out = np.empty(bits.size, np.float32)
    lib.oracle_widen_array(fmt_code(fmt), bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def narrow(fmt, values):
    """float32 values -> 16-bit patterns, by the oracle's own RNE conversion."""
    lib = _load()
    values = np.ascontiguousarray(values, dtype=np.float32).reshape(-1)
    out = np.empty(values.size, np.uint16)
    lib.oracle_narrow_array(fmt_code(fmt), values.ctypes.data, out.ctypes.data, values.size)
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())
