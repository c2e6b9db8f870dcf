"""Python binding of include/ar.h (ctypes; argument marshalling only).

Every step of the exchange runs in libtda_ar.so.  PyTorch is used only to hand
over device pointers (``tensor.data_ptr()``) and streams
(``torch.cuda.Stream.cuda_stream``).  If the library is not built, every call
raises: there is no CPU path.

Module-level functions carry the C names (``ar_create``, ``ar_allreduce``, ...)
and take raw pointers / stream handles as ints.  ``Handle`` wraps one
``ar_handle*`` for tensor arguments.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import builder as _build

AR_F16, AR_BF16, AR_C64 = 1, 2, 3
AR_SLOT_PINNED_HOST, AR_SLOT_HBM = 0, 1
AR_ALGO_AUTO, AR_ALGO_ONESHOT, AR_ALGO_TWOSHOT, AR_ALGO_TAGGED, AR_ALGO_CLUSTER, AR_ALGO_PUSH = -1, 0, 1, 2, 3, 4
ALGOS = {"auto": AR_ALGO_AUTO, "oneshot": AR_ALGO_ONESHOT, "twoshot": AR_ALGO_TWOSHOT, "tagged": AR_ALGO_TAGGED,
         "cluster": AR_ALGO_CLUSTER, "push": AR_ALGO_PUSH}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
AR_OK, AR_EINVAL, AR_ETOOBIG, AR_ESTREAM, AR_ENOMEM, AR_ECUDA, AR_ETIMEOUT, AR_ESTATE = range(8)
CODE_NAMES = {0: "AR_OK", 1: "AR_EINVAL", 2: "AR_ETOOBIG", 3: "AR_ESTREAM", 4: "AR_ENOMEM",
              5: "AR_ECUDA", 6: "AR_ETIMEOUT", 7: "AR_ESTATE"}
ITEMSIZE = {AR_F16: 2, AR_BF16: 2, AR_C64: 8}
SLOT_KINDS = {"pinned": AR_SLOT_PINNED_HOST, "pinned_host": AR_SLOT_PINNED_HOST, "host": AR_SLOT_PINNED_HOST,
              "hbm": AR_SLOT_HBM, "device": AR_SLOT_HBM}


class ArError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = int(code)
        super().__init__(f"{what}: {strerror(code)}" if what else strerror(code))


class ErrorInfo(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("rank", ctypes.c_int32), ("block", ctypes.c_int32),
                ("peer", ctypes.c_int32), ("want", ctypes.c_uint64), ("seen", ctypes.c_uint64)]


class Info(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("dtype", ctypes.c_int32), ("slot_kind", ctypes.c_int32),
                ("device", ctypes.c_int32), ("threads", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("blocks_per_sm", ctypes.c_int32),
                ("blocks_per_sm_twoshot", ctypes.c_int32), ("blocks_per_sm_allgather", ctypes.c_int32),
                ("algo", ctypes.c_int32), ("pdl", ctypes.c_int32),
                ("max_numel", ctypes.c_uint64), ("slot_bytes", ctypes.c_uint64),
                ("total_slot_bytes", ctypes.c_uint64), ("timeout_ns", ctypes.c_uint64),
                ("tagged_capacity_bytes", ctypes.c_uint64), ("blocks_per_sm_tagged", ctypes.c_int32),
                ("cluster_form", ctypes.c_int32)]


class Tactics(ctypes.Structure):
    _fields_ = [("twoshot_min_bytes", ctypes.c_uint64), ("twoshot_sub", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("tagged_max_bytes", ctypes.c_uint64),
                ("cluster_twoshot_min_bytes", ctypes.c_uint64), ("cluster_max_bytes", ctypes.c_uint64),
                ("all_fused", ctypes.c_int32), ("pace_mbs", ctypes.c_int32),
                ("pace_min_bytes", ctypes.c_uint64), ("pace_multi_mbs", ctypes.c_int32),
                ("gpu_scope", ctypes.c_int32)]


TACTIC_FIELDS = [name for name, _ in Tactics._fields_]


class Plan(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_int32), ("threads", ctypes.c_int32), ("vec_bytes", ctypes.c_int32),
                ("unroll", ctypes.c_int32), ("algo", ctypes.c_int32), ("flag_rounds", ctypes.c_int32),
                ("subtile_vecs", ctypes.c_int32), ("pace_cycles", ctypes.c_int32),
                ("tile_bytes", ctypes.c_uint64), ("tiles", ctypes.c_uint64),
                ("max_stages", ctypes.c_uint64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libtda_ar.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "tensor_decode_all_gb300.build() (there is no CPU fallback)")
            L = ctypes.CDLL(path)
            vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
            L.ar_create.argtypes = [i32, i32, sz, i32]
            L.ar_create.restype = vp
            L.ar_last_error.restype = i32
            for name in ("ar_allreduce", "ar_allgather"):
                f = getattr(L, name)
                f.argtypes = [vp, i32, vp, vp, sz, vp]
                f.restype = i32
            L.ar_status.argtypes = [vp, ctypes.POINTER(ErrorInfo)]
            L.ar_reset.argtypes = [vp]
            L.ar_destroy.argtypes = [vp]
            L.ar_set_timeout.argtypes = [vp, u64]
            L.ar_query.argtypes = [vp, ctypes.POINTER(Info)]
            L.ar_plan_for.argtypes = [vp, i32, sz, ctypes.POINTER(Plan)]
            L.ar_plan_compute.argtypes = [i32, u64, i32, i32, i32, i32, i32, ctypes.POINTER(Plan)]
            L.ar_choose_algo.argtypes = [i32, u64, i32]
            L.ar_set_algo.argtypes = [vp, i32]
            L.ar_set_pdl.argtypes = [vp, i32]
            L.ar_get_tactics.argtypes = [vp, ctypes.POINTER(Tactics)]
            L.ar_set_tactics.argtypes = [vp, ctypes.POINTER(Tactics)]
            L.ar_supports.argtypes = [vp, i32, sz, vp, vp]
            L.ar_set_trace.argtypes = [vp, vp, u64]
            L.ar_debug_seed_stages.argtypes = [vp, u64]
            L.ar_allreduce_noalloc.argtypes = [i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, vp]
            L.ar_allreduce_noalloc.restype = i32
            L.ar_noalloc_status.argtypes = [ctypes.POINTER(ErrorInfo)]
            L.ar_noalloc_status.restype = i32
            L.ar_noalloc_debug_record.argtypes = [ctypes.POINTER(ErrorInfo)]
            L.ar_noalloc_debug_record.restype = i32
            for name in ("ar_allreduce_fused", "ar_allgather_fused"):
                f = getattr(L, name)
                f.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, vp]
                f.restype = i32
            L.ar_allreduce_all.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, ctypes.POINTER(vp)]
            L.ar_allreduce_all.restype = i32
            L.ar_strerror.argtypes = [i32]
            L.ar_strerror.restype = ctypes.c_char_p
            L.ar_probe_host_link.argtypes = [u64, i32, ctypes.POINTER(ctypes.c_double)]
            L.ar_probe_hbm_copy.argtypes = [u64, i32, ctypes.POINTER(ctypes.c_double)]
            L.ar_probe_host_link_latency.argtypes = [i32, ctypes.POINTER(ctypes.c_double)]
            L.ar_probe_host_link_latency.restype = i32
            _lib = L
    return _lib


def declared_symbols(header: str | None = None):
    """Names of the entry points include/ar.h declares."""
    header = header or os.path.join(_build.INCLUDE, "ar.h")
    text = open(header).read()
    return sorted(set(re.findall(r"AR_API\s+[^;(]*?\b(ar_\w+)\s*\(", text)))


# ---------------------------------------------------------------- C names

def ar_create(R: int, dtype: int, max_numel: int, slot_kind: int) -> int:
    return lib().ar_create(R, dtype, max_numel, slot_kind) or 0


def ar_last_error() -> int:
    return lib().ar_last_error()


def ar_allreduce(h: int, rank: int, inp: int, out: int, numel: int, stream: int) -> int:
    return lib().ar_allreduce(h, rank, inp, out, numel, stream)


def ar_allgather(h: int, rank: int, inp: int, out: int, numel: int, stream: int) -> int:
    return lib().ar_allgather(h, rank, inp, out, numel, stream)


def ar_allreduce_noalloc(R: int, dtype: int, ins, outs, numel: int, stream: int) -> int:
    """All R ranks in one call, with no allocation (ins/outs: R device pointers)."""
    arr_in = (ctypes.c_void_p * R)(*[int(p) for p in ins])
    arr_out = (ctypes.c_void_p * R)(*[int(p) for p in outs])
    return lib().ar_allreduce_noalloc(R, dtype, arr_in, arr_out, numel, stream)


def ar_noalloc_status():
    """(code, ErrorInfo) of ar_allreduce_noalloc's error record on the current device."""
    info = ErrorInfo()
    rc = lib().ar_noalloc_status(ctypes.byref(info))
    return rc, info


def ar_noalloc_debug_record(info: ErrorInfo) -> int:
    """Test hook: write an error record into ar_allreduce_noalloc's array."""
    return lib().ar_noalloc_debug_record(ctypes.byref(info))


def ar_get_tactics(h: int) -> Tactics:
    t = Tactics()
    rc = lib().ar_get_tactics(h, ctypes.byref(t))
    if rc:
        raise ArError(rc, "ar_get_tactics")
    return t


def ar_set_tactics(h: int, t: Tactics) -> int:
    return lib().ar_set_tactics(h, ctypes.byref(t))


def ar_supports(h: int, op: int, numel: int, inp: int, out: int) -> int:
    return lib().ar_supports(h, op, numel, inp, out)


def _ptr_array(ptrs):
    ptrs = [int(p) for p in ptrs]
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


def ar_allreduce_fused(h: int, ins, outs, numel: int, stream: int) -> int:
    """Every rank's call at once, one cooperative launch (ins/outs: R device pointers)."""
    return lib().ar_allreduce_fused(h, _ptr_array(ins), _ptr_array(outs), numel, stream)


def ar_allgather_fused(h: int, ins, outs, numel: int, stream: int) -> int:
    return lib().ar_allgather_fused(h, _ptr_array(ins), _ptr_array(outs), numel, stream)


def ar_allreduce_all(h: int, ins, outs, numel: int, streams) -> int:
    """Every rank's call, rank r's on streams[r] (R device pointers per side, R stream handles)."""
    return lib().ar_allreduce_all(h, _ptr_array(ins), _ptr_array(outs), numel, _ptr_array(streams))


def ar_status(h: int) -> ErrorInfo:
    info = ErrorInfo()
    lib().ar_status(h, ctypes.byref(info))
    return info


def ar_reset(h: int) -> int:
    return lib().ar_reset(h)


def ar_destroy(h: int) -> int:
    return lib().ar_destroy(h)


def ar_set_timeout(h: int, ns: int) -> int:
    return lib().ar_set_timeout(h, ns)


def ar_query(h: int) -> Info:
    info = Info()
    rc = lib().ar_query(h, ctypes.byref(info))
    if rc:
        raise ArError(rc, "ar_query")
    return info


def ar_plan_for(h: int, op: int, numel: int) -> Plan:
    p = Plan()
    rc = lib().ar_plan_for(h, op, numel, ctypes.byref(p))
    if rc:
        raise ArError(rc, "ar_plan_for")
    return p


def ar_plan_compute(R, nbytes, vec_bytes, algo, threads, sm_count, blocks_per_sm) -> Plan:
    p = Plan()
    rc = lib().ar_plan_compute(R, nbytes, vec_bytes, algo, threads, sm_count, blocks_per_sm, ctypes.byref(p))
    if rc:
        raise ArError(rc, "ar_plan_compute")
    return p


def ar_choose_algo(R: int, nbytes: int, slot_kind: int) -> int:
    return lib().ar_choose_algo(R, nbytes, slot_kind)


def ar_set_algo(h: int, algo: int) -> int:
    return lib().ar_set_algo(h, algo)


def ar_set_pdl(h: int, enable: bool) -> int:
    return lib().ar_set_pdl(h, 1 if enable else 0)


def strerror(code: int) -> str:
    try:
        return lib().ar_strerror(int(code)).decode()
    except RuntimeError:
        return CODE_NAMES.get(int(code), f"code {code}")


ar_strerror = strerror


def ar_probe_host_link(nbytes: int, reps: int):
    out = (ctypes.c_double * 5)()
    rc = lib().ar_probe_host_link(nbytes, reps, out)
    if rc:
        raise ArError(rc, "ar_probe_host_link")
    return {"write_gbs": out[0], "read_gbs": out[1], "bidir_write_gbs": out[2], "bidir_read_gbs": out[3]}


def ar_probe_host_link_latency(reps: int = 200):
    out = (ctypes.c_double * 5)()
    rc = lib().ar_probe_host_link_latency(int(reps), out)
    if rc:
        raise ArError(rc, "ar_probe_host_link_latency")
    return {"host_load_rtt_ns": out[0], "store_4KiB_fence_sys_ns": out[1], "flag_host_sys_one_way_ns": out[2],
            "flag_hbm_gpu_one_way_ns": out[3], "store_4KiB_fence_gpu_ns": out[4]}


def ar_probe_hbm_copy(nbytes: int, reps: int) -> float:
    out = ctypes.c_double()
    rc = lib().ar_probe_hbm_copy(nbytes, reps, ctypes.byref(out))
    if rc:
        raise ArError(rc, "ar_probe_hbm_copy")
    return out.value


# ------------------------------------------------------------- tensor API

def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    import torch
    table = {torch.float16: AR_F16, torch.bfloat16: AR_BF16, torch.complex64: AR_C64}
    if dtype in table:
        return table[dtype]
    return {"f16": AR_F16, "fp16": AR_F16, "bf16": AR_BF16, "c64": AR_C64, "complex64": AR_C64}[str(dtype)]


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class Handle:
    """One ar_handle: R logical ranks, one dtype, fixed max_numel, one slot kind."""

    def __init__(self, R: int, dtype, max_numel: int, slot_kind="hbm"):
        self.R = int(R)
        self.dtype = _dtype_code(dtype)
        self.slot_kind = SLOT_KINDS[slot_kind] if isinstance(slot_kind, str) else int(slot_kind)
        self.max_numel = int(max_numel)
        self._h = ar_create(self.R, self.dtype, self.max_numel, self.slot_kind)
        if not self._h:
            raise ArError(ar_last_error(), "ar_create")

    @property
    def ptr(self) -> int:
        if not self._h:
            raise RuntimeError("handle destroyed")
        return self._h

    def _check_tensors(self, name: str, inp, out, out_factor: int) -> None:
        """What the C ABI cannot see through raw pointers: both tensors dense,
        of the handle's dtype, and `out` large enough for the call (numel
        elements for an all-reduce, R * numel for an allgather), so that a
        wrong tensor is refused here instead of being read or written past
        its end on the device."""
        for what, t in (("input", inp), ("output", out)):
            if not t.is_contiguous():
                raise ValueError(f"{name}: {what} tensor is not contiguous")
            try:
                code = _dtype_code(t.dtype)
            except KeyError:
                code = None
            if code != self.dtype:
                raise ValueError(f"{name}: {what} dtype {t.dtype} does not match the handle's")
        if out.numel() < out_factor * inp.numel():
            raise ValueError(f"{name}: output holds {out.numel()} elements, the call writes {out_factor * inp.numel()}")

    def allreduce(self, rank: int, inp, out, stream=None) -> None:
        self._check_tensors("ar_allreduce", inp, out, 1)
        rc = ar_allreduce(self.ptr, rank, inp.data_ptr(), out.data_ptr(), inp.numel(), _stream_handle(stream))
        if rc:
            raise ArError(rc, f"ar_allreduce(rank={rank})")

    def allgather(self, rank: int, inp, out, stream=None) -> None:
        self._check_tensors("ar_allgather", inp, out, self.R)
        rc = ar_allgather(self.ptr, rank, inp.data_ptr(), out.data_ptr(), inp.numel(), _stream_handle(stream))
        if rc:
            raise ArError(rc, f"ar_allgather(rank={rank})")

    def allreduce_all(self, ins, outs, streams) -> None:
        """Enqueue all R ranks' calls, rank r's output ready on streams[r]
        (ar_allreduce_all: R per-rank launches or one launch of every rank,
        by the handle's all_fused tactic)."""
        if len(ins) != self.R or len(outs) != self.R or len(streams) != self.R:
            raise ValueError(f"ar_allreduce_all: need {self.R} inputs, outputs and streams")
        for r in range(self.R):
            if ins[r].numel() != ins[0].numel():
                raise ValueError(f"ar_allreduce_all: rank {r}'s input has {ins[r].numel()} elements, "
                                 f"rank 0's {ins[0].numel()}")
            self._check_tensors("ar_allreduce_all", ins[r], outs[r], 1)
        rc = ar_allreduce_all(self.ptr, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], ins[0].numel(),
                              [_stream_handle(s) for s in streams])
        if rc:
            raise ArError(rc, "ar_allreduce_all")

    def allreduce_each(self, ins, outs, streams) -> None:
        """Enqueue all R ranks' calls as R separate ar_allreduce calls (rank r on streams[r])."""
        for r in range(self.R):
            self.allreduce(r, ins[r], outs[r], streams[r])

    def allgather_all(self, ins, outs, streams) -> None:
        for r in range(self.R):
            self.allgather(r, ins[r], outs[r], streams[r])

    def allreduce_fused(self, ins, outs, stream=None) -> None:
        """All R ranks' calls as one launch on one stream (ins[r], outs[r]: rank r's tensors)."""
        self._fused(ar_allreduce_fused, "ar_allreduce_fused", ins, outs, stream)

    def allgather_fused(self, ins, outs, stream=None) -> None:
        self._fused(ar_allgather_fused, "ar_allgather_fused", ins, outs, stream)

    def _fused(self, fn, name, ins, outs, stream) -> None:
        if len(ins) != self.R or len(outs) != self.R:
            raise ValueError(f"{name}: need {self.R} inputs and outputs")
        factor = self.R if fn is ar_allgather_fused else 1
        for r in range(self.R):
            if ins[r].numel() != ins[0].numel():
                raise ValueError(f"{name}: rank {r}'s input has {ins[r].numel()} elements, rank 0's {ins[0].numel()}")
            self._check_tensors(name, ins[r], outs[r], factor)
        rc = fn(self.ptr, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], ins[0].numel(),
                _stream_handle(stream))
        if rc:
            raise ArError(rc, name)

    def status(self) -> ErrorInfo:
        return ar_status(self.ptr)

    def check(self) -> None:
        st = self.status()
        if st.code:
            raise ArError(st.code, f"device (rank {st.rank} block {st.block} waited on peer {st.peer}: "
                                   f"want {st.want} seen {st.seen})")

    def reset(self) -> None:
        rc = ar_reset(self.ptr)
        if rc:
            raise ArError(rc, "ar_reset")

    def set_timeout(self, ns: int) -> None:
        rc = ar_set_timeout(self.ptr, int(ns))
        if rc:
            raise ArError(rc, "ar_set_timeout")

    def set_algo(self, algo) -> None:
        """'auto', 'oneshot', 'twoshot', 'tagged', 'cluster' or 'push' (or an AR_ALGO_* code)."""
        code = ALGOS[algo] if isinstance(algo, str) else int(algo)
        rc = ar_set_algo(self.ptr, code)
        if rc:
            raise ArError(rc, "ar_set_algo")

    def set_pdl(self, enable: bool) -> None:
        rc = ar_set_pdl(self.ptr, enable)
        if rc:
            raise ArError(rc, "ar_set_pdl")

    def info(self) -> Info:
        return ar_query(self.ptr)

    def tactics(self) -> dict:
        t = ar_get_tactics(self.ptr)
        return {name: int(getattr(t, name)) for name in TACTIC_FIELDS}

    def set_tactics(self, **changes) -> None:
        """Replace some or all of the handle's tactics (see ar_tactics in ar.h);
        keyword names are the struct's fields, None keeps a field."""
        unknown = set(changes) - set(TACTIC_FIELDS)
        if unknown:
            raise TypeError(f"unknown tactics {sorted(unknown)}")
        cur = self.tactics()
        cur.update({k: v for k, v in changes.items() if v is not None})
        t = Tactics(**{name: int(cur[name]) for name in TACTIC_FIELDS})
        rc = ar_set_tactics(self.ptr, t)
        if rc:
            raise ArError(rc, "ar_set_tactics")

    def set_trace(self, buf, capacity: int) -> None:
        """Trace into `buf` (device memory of `capacity` records), or stop (buf None)."""
        rc = lib().ar_set_trace(self.ptr, buf.data_ptr() if buf is not None else None, int(capacity))
        if rc:
            raise ArError(rc, "ar_set_trace")

    def debug_seed_stages(self, stages: int) -> None:
        """Test hook: set every block's stage count (see ar_debug_seed_stages)."""
        rc = lib().ar_debug_seed_stages(self.ptr, int(stages))
        if rc:
            raise ArError(rc, "ar_debug_seed_stages")

    def supports(self, op: str, inp, out) -> int:
        """AR_OK if ar_allreduce / ar_allgather would accept these tensors, else its code."""
        return ar_supports(self.ptr, 0 if op == "allreduce" else 1, inp.numel(), inp.data_ptr(), out.data_ptr())

    def plan(self, op: str, numel: int) -> Plan:
        """op: 'allreduce' (one rank's launch), 'allgather', or 'allreduce_fused'
        (every rank in one launch)."""
        return ar_plan_for(self.ptr, {"allreduce": 0, "allgather": 1, "allreduce_fused": 2}[op], numel)

    def destroy(self) -> None:
        if self._h:
            h, self._h = self._h, 0
            rc = ar_destroy(h)
            if rc:
                raise ArError(rc, "ar_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass
