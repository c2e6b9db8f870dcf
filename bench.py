#!/usr/bin/env python3
"""Benchmark of the logical-rank all-reduce on one GB300 (one JSON line).

Headline workload: R=2 logical ranks, fp16, N=131072 elements per rank (256 KiB,
the host all-reduce's payload cap), pinned-host slots, calls replayed from a
CUDA graph.  A step is one graph replay of C calls (every call of the step has
its own input and output buffers, so inputs are fresh each call); L2 is
flushed (a 256 MiB write) before every step, outside the timed events.

value = algbw = S / (time per call), S = per-rank payload bytes (GB/s, 1e9).
Also reported: us/call, the host-link roofline of the exchange kernel (with
the link bandwidth measured in the same run by the library's probe kernels),
an end-to-end figure through the C ABI with host buffers, the HBM-slot
workloads (R=8 bf16, 16/64 MiB), the complex64 allgather, and the CPU oracle
timed on the host's cores.

--impl reference runs the CPU oracle instead (the reference arm of this
build): the same metric, config and unit, each step a bounded sample.

--gpus N (under torchrun) runs N independent replicas, one per GPU: the
all-reduce's ranks are logical ranks on one GPU, so there is nothing to shard
across GPUs.  The step time is the max over GPUs; value sums the replicas.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "all-reduce us/call and algbw GB/s vs payload, R logical ranks on 1 GB300 (graph)"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--calls", type=int, default=100, help="all-reduce calls per step (graph length)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", default=None, help="run the payload sweep; write JSON lines to this file")
    ap.add_argument("--sweep-calls", type=int, default=1000)
    ap.add_argument("--sweep-both", action="store_true",
                    help="in the sweep, run both all-reduce forms where they compete (R >= 3, 64 KiB..8 MiB)")
    ap.add_argument("--sweep-slots", default="hbm,pinned")
    ap.add_argument("--sweep-dtypes", default="f16,bf16")
    ap.add_argument("--sweep-ranks", default="2,4,8")
    ap.add_argument("--sweep-algo", default=None, choices=["oneshot", "twoshot", "tagged", "cluster"],
                    help="in the sweep, force this all-reduce form in every cell")
    ap.add_argument("--sweep-fused", action="store_true",
                    help="in the sweep, run every call as one launch of all ranks (ar_allreduce_fused)")
    ap.add_argument("--sweep-launch", default=None, choices=["rank", "fused", "all"],
                    help="in the sweep, the launch form (default rank, or fused with --sweep-fused)")
    ap.add_argument("--sweep-tactics", default=None, help="in the sweep, ar_tactics fields to set (JSON object)")
    ap.add_argument("--sweep-min-kib", type=int, default=2)
    ap.add_argument("--sweep-max-kib", type=int, default=65536)
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    ap.add_argument("--push-ab", default=None,
                    help="time the push form against the pull forms (R=2,4; 8 KiB, 256 KiB, 4 MiB; both slot "
                         "kinds); write JSON lines to this file")
    ap.add_argument("--only", default=None,
                    help="comma-separated workload names: time only these (no headline, no JSON contract line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trace", default=None, help="trace the main workloads with ar_set_trace; write a summary here")
    ap.add_argument("--profile", default=None, choices=sorted(PROFILE_WORKLOADS),
                    help="graph replays of one workload only (for ncu --graph-profiling graph)")
    return ap.parse_args()


# --------------------------------------------------------------------- dist

class Dist:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl"
            try:
                import torch
                if not torch.cuda.is_available():
                    backend = "gloo"
            except Exception:
                backend = "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() and self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def max_over_ranks(values):
    """The slowest replica sets the step time."""
    return max(values)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"tda_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9 and p[1].replace(".", "").isdigit():
                    rows.append(p)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                          if r[3].replace(".", "").isdigit())}


# ------------------------------------------------------------- measurement

# The code each kernel family is compiled from (paths from the repository
# root).  Profiled counters belong to one family: an edit to another family's
# code leaves them valid, an edit to their own (or to a shared header, the
# C header's structs included) voids them.
_CSRC = "tensor_decode_all_gb300/csrc/"
_COMMON_SOURCES = ("include/ar.h", _CSRC + "ar_internal.h", _CSRC + "ar_sync.cuh")
# ar_allreduce.cuh includes the tagged-word and push headers, so every
# all-reduce family's translation units see them
_ALLREDUCE_HEADERS = (_CSRC + "ar_allreduce.cuh", _CSRC + "ar_allreduce_tagged.cuh", _CSRC + "ar_allreduce_push.cuh")
FORM_SOURCES = {
    "oneshot": _COMMON_SOURCES + _ALLREDUCE_HEADERS + (_CSRC + "ar_allreduce_f16.cu", _CSRC + "ar_allreduce_bf16.cu"),
    "twoshot": _COMMON_SOURCES + _ALLREDUCE_HEADERS + (_CSRC + "ar_allreduce_f16_twoshot.cu",
                                                       _CSRC + "ar_allreduce_bf16_twoshot.cu"),
    "tagged": _COMMON_SOURCES + _ALLREDUCE_HEADERS + (_CSRC + "ar_allreduce_f16.cu", _CSRC + "ar_allreduce_bf16.cu"),
    "push": _COMMON_SOURCES + _ALLREDUCE_HEADERS + (_CSRC + "ar_allreduce_f16.cu", _CSRC + "ar_allreduce_bf16.cu"),
    "cluster": _COMMON_SOURCES + _ALLREDUCE_HEADERS + (_CSRC + "ar_allreduce_cluster.cuh",
                                                       _CSRC + "ar_allreduce_f16_cluster.cu",
                                                       _CSRC + "ar_allreduce_bf16_cluster.cu"),
    "allgather": _COMMON_SOURCES + (_CSRC + "ar_allgather.cu",),
}


def source_sha256(form: str) -> str:
    """Hash of the code (comments and blank space removed) a kernel family is
    compiled from: profiled counters stay valid across comment edits."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in FORM_SOURCES[form]:
        with open(os.path.join(ROOT, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


HEADLINE_R, HEADLINE_NUMEL = 2, 131072


def headline_config(n_gpus: int) -> dict:
    """The headline workload's config, the same in both arms of the bench."""
    return {"workload": "R=2 logical ranks, fp16, N=131072 per rank (256 KiB), pinned-host slots, graph-replayed",
            "R": HEADLINE_R, "numel": HEADLINE_NUMEL, "bytes_per_rank": HEADLINE_NUMEL * 2, "slots": "pinned_host",
            "l2": "flushed (256 MiB write) before every step, outside the timed events",
            "parallelism": f"replicas x{n_gpus} (logical ranks share one GPU)"}


def profiled_traffic(name: str):
    """DRAM and host-link bytes per call of a workload, from the committed ncu
    summary (profiles/traffic.json), or None if its kernel family's code
    changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except Exception:
        return None
    entry = t.get("workloads", {}).get(name)
    if not entry or entry.get("form") not in FORM_SOURCES:
        return None
    if entry.get("source_sha256") != source_sha256(entry["form"]):
        return None
    return entry


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return {}


class Workload:
    """R ranks, C calls, one graph; every call has its own device buffers."""

    # handles whose device status was read after their timed steps (ar_status:
    # a bounded wait that ran out would be recorded there, and check() raises)
    status_reads = 0

    def __init__(self, op, R, dtype, numel, slots, calls, config, dist="uniform", algo=None, fused=False,
                 launch=None, tactics=None):
        import torch
        import tensor_decode_all_gb300 as tda
        from tensor_decode_all_gb300 import ar, inputs
        self.torch = torch
        self.op, self.R, self.dtype, self.numel, self.slots, self.C = op, R, dtype, numel, slots, calls
        # "rank": one launch per rank per call (ar_allreduce / ar_allgather on R streams);
        # "fused": one launch of every rank per call (ar_*_fused on one stream);
        # "all": ar_allreduce_all on the R streams (fused or not by the handle's tactic)
        self.launch = launch or ("fused" if fused else "rank")
        self.fused = self.launch == "fused"
        tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "c64": torch.complex64}[dtype]
        self.tdt = tdt
        self.h = tda.Handle(R, tdt, numel, slots)
        if algo:
            self.h.set_algo(algo)
        if tactics:
            self.h.set_tactics(**tactics)
        if op == "allgather":
            self.algo = "allgather"
        else:
            one_launch = self.launch == "fused" or (self.launch == "all" and self.h.tactics()["all_fused"])
            p = self.h.plan("allreduce_fused" if one_launch else "allreduce", numel)
            self.algo = ar.ALGO_NAMES[p.algo] + (f"/sub{p.subtile_vecs}" if p.algo == 3 and p.subtile_vecs else "")
        self.streams = [torch.cuda.Stream() for _ in range(R)]
        out_n = numel * (R if op == "allgather" else 1)
        # inputs [C][numel] per rank, contiguous, so one copy moves a whole step
        self.ins = [torch.empty((calls, numel), dtype=tdt, device="cuda") for _ in range(R)]
        self.outs = [torch.empty((calls, out_n), dtype=tdt, device="cuda") for _ in range(R)]
        self.host_in = []
        isz = 8 if dtype == "c64" else 2
        distinct = min(calls, 8) if numel * isz <= (1 << 20) else (2 if numel * isz <= (16 << 20) else 1)
        per_call = []
        for c in range(distinct):
            if op == "allgather":
                per_call.append([z.view(np.uint8) for z in inputs.allgather_inputs(config, R, numel, c)])
            else:
                per_call.append([x.view(np.uint8) for x in inputs.allreduce_inputs(config, R, numel, dtype, dist, c)])
        for r in range(R):
            host = np.stack([per_call[c % distinct][r] for c in range(calls)])
            self.host_in.append(host)
            self.ins[r].copy_(torch.from_numpy(host).view(tdt).view(calls, numel))
        self.graph = None

    def capture(self):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                cap = torch.cuda.current_stream()
                if self.launch == "fused":
                    for c in range(self.C):
                        getattr(self.h, self.op + "_fused")([self.ins[r][c] for r in range(self.R)],
                                                            [self.outs[r][c] for r in range(self.R)], cap)
                elif self.launch == "all":
                    for s in self.streams:
                        s.wait_stream(cap)
                    for c in range(self.C):
                        self.h.allreduce_all([self.ins[r][c] for r in range(self.R)],
                                             [self.outs[r][c] for r in range(self.R)], self.streams)
                    for s in self.streams:
                        cap.wait_stream(s)
                else:
                    for s in self.streams:
                        s.wait_stream(cap)
                    for c in range(self.C):
                        for r in range(self.R):
                            getattr(self.h, self.op)(r, self.ins[r][c], self.outs[r][c], self.streams[r])
                    for s in self.streams:
                        cap.wait_stream(s)
        torch.cuda.current_stream().wait_stream(side)
        self.graph = g
        return g

    def check(self, calls=(0, -1)):
        """Bit-exact comparison of sampled calls with the CPU oracle."""
        import oracle
        self.torch.cuda.synchronize()
        self.h.check()
        Workload.status_reads += 1
        for c in calls:
            c = c % self.C
            xs = [self.host_in[r][c] for r in range(self.R)]
            if self.op == "allgather":
                want = oracle.allgather(xs, ranks=[0])[0]
            else:
                want = oracle.allreduce([x.view(np.uint16) for x in xs], self.dtype, ranks=[0])[0].view(np.uint8)
            for r in range(self.R):
                got = self.outs[r][c].cpu()
                got = got.view(self.torch.uint8).numpy() if self.dtype != "c64" else got.numpy().view(np.uint8)
                if not np.array_equal(got, want):
                    raise AssertionError(f"bench parity: {self.op} call {c} rank {r} differs from the oracle")
        return len(calls) * self.R

    def check_host_outputs(self, host_outs, calls=(0, -1)):
        """Outputs copied back to pinned host memory, against the CPU oracle."""
        import oracle
        for c in calls:
            c = c % self.C
            xs = [self.host_in[r][c] for r in range(self.R)]
            want = oracle.allreduce([x.view(np.uint16) for x in xs], self.dtype, ranks=[0])[0].view(np.uint8)
            for r in range(self.R):
                got = host_outs[r][c].view(self.torch.uint8).numpy()
                if not np.array_equal(got, want):
                    raise AssertionError(f"bench e2e parity: call {c} rank {r} differs from the oracle")
        return len(calls) * self.R

    def time_graph(self, steps, warmup, flush):
        torch = self.torch
        if self.graph is None:
            self.capture()
        cur = torch.cuda.current_stream()
        for _ in range(warmup):
            flush.zero_()
            self.graph.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            flush.zero_()
            a.record(cur)
            self.graph.replay()
            b.record(cur)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]  # ms per step

    def time_e2e(self, steps, chunk=10):
        """End to end through the C ABI with host buffers, as a user with pinned
        host tensors would pipeline it: one CUDA graph per step holding, for
        each chunk of `chunk` calls, the host->device copy of the chunk's
        inputs (copy stream), the chunk's calls of every rank (rank streams),
        and the device->host copy of its outputs (second copy stream), so the
        copies of one chunk overlap the calls of its neighbours.  Every step
        moves all of its inputs in and all of its outputs out inside the timed
        region.  Also returns the time of the plain serial form (one copy in,
        eager calls, one copy out) for reference."""
        torch = self.torch
        pin_in = [torch.from_numpy(self.host_in[r]).view(self.tdt).view(self.C, self.numel).pin_memory()
                  for r in range(self.R)]
        pin_out = [torch.empty(self.outs[r].shape, dtype=self.tdt).pin_memory() for r in range(self.R)]
        cur = torch.cuda.current_stream()
        nchunks = (self.C + chunk - 1) // chunk

        g = torch.cuda.CUDAGraph()
        side, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                cap = torch.cuda.current_stream()
                s_in.wait_stream(cap)
                s_out.wait_stream(cap)
                for k in range(nchunks):
                    lo, hi = k * chunk, min(self.C, (k + 1) * chunk)
                    with torch.cuda.stream(s_in):
                        for r in range(self.R):
                            self.ins[r][lo:hi].copy_(pin_in[r][lo:hi], non_blocking=True)
                    for st in self.streams:
                        st.wait_stream(s_in)
                    for c in range(lo, hi):
                        for r in range(self.R):
                            getattr(self.h, self.op)(r, self.ins[r][c], self.outs[r][c], self.streams[r])
                    for st in self.streams:
                        s_out.wait_stream(st)
                    with torch.cuda.stream(s_out):
                        for r in range(self.R):
                            pin_out[r][lo:hi].copy_(self.outs[r][lo:hi], non_blocking=True)
                for st in (s_in, s_out, *self.streams):
                    cap.wait_stream(st)
        cur.wait_stream(side)
        times = []
        for step in range(steps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            if step:  # the first replay warms the pinned buffers
                times.append(a.elapsed_time(b))
        del g
        # the last replay's outputs, as copied back to the host, against the oracle
        self.e2e_checked = self.check_host_outputs(pin_out, calls=(0, self.C // 2, -1))

        serial = []
        for step in range(min(steps, 10) + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(cur)
            for r in range(self.R):
                self.ins[r].copy_(pin_in[r], non_blocking=True)
            for st in self.streams:
                st.wait_stream(cur)
            for c in range(self.C):
                for r in range(self.R):
                    getattr(self.h, self.op)(r, self.ins[r][c], self.outs[r][c], self.streams[r])
            for st in self.streams:
                cur.wait_stream(st)
            for r in range(self.R):
                pin_out[r].copy_(self.outs[r], non_blocking=True)
            b.record(cur)
            b.synchronize()
            if step:
                serial.append(a.elapsed_time(b))
        # Zero copy: the calls take the pinned host tensors themselves (mapped
        # host memory is device-accessible), so each rank's kernel reads its
        # input from the host and writes its output to the host; no copy
        # engine, one graph of C calls per rank.
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                cap = torch.cuda.current_stream()
                for st in self.streams:
                    st.wait_stream(cap)
                for c in range(self.C):
                    for r in range(self.R):
                        getattr(self.h, self.op)(r, pin_in[r][c], pin_out[r][c], self.streams[r])
                for st in self.streams:
                    cap.wait_stream(st)
        cur.wait_stream(side)
        pin_out_zero = [t.zero_() for t in pin_out]
        zero_copy = []
        for step in range(steps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            if step:
                zero_copy.append(a.elapsed_time(b))
        del g
        self.e2e_checked += self.check_host_outputs(pin_out_zero, calls=(0, self.C // 2, -1))
        # Zero copy through ar_allreduce_all: the same host tensors, every call
        # of every rank as one launch (the handle's all_fused tactic).
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                cap = torch.cuda.current_stream()
                for st in self.streams:
                    st.wait_stream(cap)
                for c in range(self.C):
                    self.h.allreduce_all([pin_in[r][c] for r in range(self.R)],
                                         [pin_out[r][c] for r in range(self.R)], self.streams)
                for st in self.streams:
                    cap.wait_stream(st)
        cur.wait_stream(side)
        for t in pin_out:
            t.zero_()
        zero_all = []
        for step in range(steps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            if step:
                zero_all.append(a.elapsed_time(b))
        del g
        self.e2e_checked += self.check_host_outputs(pin_out, calls=(0, self.C // 2, -1))
        h2d = sum(t.numel() * t.element_size() for t in pin_in)
        d2h = sum(t.numel() * t.element_size() for t in pin_out)
        return times, h2d, d2h, serial, zero_copy, zero_all

    def close(self):
        self.graph = None
        self.h.destroy()


def algo_bytes(op, R, S, slots, algo=None):
    """Algorithmic bytes of one call (all R ranks).

    pinned-host all-reduce, one-shot: host-link writes W = R*S (each rank
      publishes once), reads Rd = R*(R-1)*S (each rank fetches every peer's chunk);
    pinned-host all-reduce, two-shot (flag or cluster form): W = R*S published + S of reduced results,
      Rd = R*S (every rank reads its sub-tile from all R slots) + (R-1)*S
      (every rank reads the R-1 other reduced sub-tiles);
    HBM all-reduce (either form): DRAM 4*R*S (inputs, slot writes, slot reads
      once, outputs);
    allgather: HBM R*S + R*S + R*S + R*R*S; pinned W = R*S, Rd = R*(R-1)*S.
    push all-reduce: every rank writes its tile into each of R-1 peers' areas
      and reads R-1 tiles from its own: pinned W = Rd = R*(R-1)*S; HBM inputs
      and outputs 2*R*S plus the areas written and read, 2*R*(R-1)*S.
    """
    if slots == "pinned":
        # the cluster form with sub-tiles ("cluster/sub64") is two-shot too
        if op == "allreduce" and (algo == "twoshot" or (algo or "").startswith("cluster/sub")):
            return {"link_write": (R + 1) * S, "link_read": (2 * R - 1) * S}
        if op == "allreduce" and algo == "push":
            return {"link_write": R * (R - 1) * S, "link_read": R * (R - 1) * S}
        return {"link_write": R * S, "link_read": R * (R - 1) * S}
    if op == "allreduce" and algo == "push":
        return {"dram": 2 * R * S + 2 * R * (R - 1) * S}
    if op == "allreduce":
        return {"dram": 4 * R * S}
    return {"dram": 3 * R * S + R * R * S}


def link_floor_s(W, Rd, link):
    """Shortest time the host link would allow for W bytes written and Rd bytes
    read if each direction kept its solo rate (measured alone by the probe in
    this run) while the other is busy.  It does not quite: with both directions
    streaming at an even split the probe sees ~170 GB/s each way against ~193 /
    ~210 alone, and add_link_floors reports that floor beside this one.  This one
    stays the headline fraction because it holds for any mix of reads and
    writes; the concurrent rates are measured at one mix."""
    gb = 1e9
    return max(W / (link["write_gbs"] * gb), Rd / (link["read_gbs"] * gb))


def roofline(op, R, S, slots, t_call_s, link, hbm_gbs, algo=None):
    b = algo_bytes(op, R, S, slots, algo)
    if slots == "pinned":
        W, Rd = b["link_write"], b["link_read"]
        t_min = link_floor_s(W, Rd, link)
        achieved = (W + Rd) / t_call_s / 1e9
        peak = (W + Rd) / t_min / 1e9
        return {"bound": "host_link", "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": "GB/s",
                "frac": round(t_min / t_call_s, 4), "traffic": None,
                "algorithmic_bytes_per_call": {"link_write": W, "link_read": Rd},
                "peak_source": "host-link probe in this run (ar_probe_host_link, of measured): link bytes over "
                               "max(W/BW_w, Rd/BW_r), each direction at its own measured rate"}
    achieved = b["dram"] / t_call_s / 1e9
    least = R * S + R * R * S if op == "allgather" else 2 * R * S
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_gbs, "unit": "GB/s",
            "frac": round(achieved / hbm_gbs, 4), "traffic": None, "algorithmic_bytes_per_call": b["dram"],
            "least_dram_bytes_per_call": least,
            "frac_least": round(least / t_call_s / 1e9 / hbm_gbs, 4),
            "dram_frac": None,
            "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)",
            "note": "frac counts 4RS (inputs, slot writes, slot reads once, outputs) as DRAM bytes; "
                    "frac_least counts only what any all-reduce must move through DRAM (inputs read, "
                    "outputs written: 2RS; allgather RS + R^2 S); dram_frac is the ncu-measured DRAM "
                    "bytes per call of the same kernel over this call time (null without a valid capture)"}


def add_link_floors(rf, lat, link, t_call_s, gpu_scope=True):
    """Beside the per-direction floor that `frac` uses, two more floors of a
    host-link call, both measured in this run: the duplex floor (each direction
    at the rate the probe sees while the other direction streams too, half the
    blocks storing and half loading -- the link does not give both directions
    their solo rates at once; a floor for calls that move about as many bytes
    each way, as the headline does) and the
    latency chain one tile must pass in protocol order (its stores ordered by
    the release's fence, the flag's one-way trip, one dependent read round
    trip), at the scope the call's ranks synchronise at: GPU scope (flags in
    HBM, the default) or system scope (flags in host memory).  No call can beat
    the larger of them; neither counts the launch."""
    W, Rd = rf["algorithmic_bytes_per_call"]["link_write"], rf["algorithmic_bytes_per_call"]["link_read"]
    gb = 1e9
    per_dir = link_floor_s(W, Rd, link)
    duplex = max(W / (link["bidir_write_gbs"] * gb), Rd / (link["bidir_read_gbs"] * gb))
    if gpu_scope:
        chain = lat["store_4KiB_fence_gpu_ns"] + lat["flag_hbm_gpu_one_way_ns"] + lat["host_load_rtt_ns"]
    else:
        chain = lat["store_4KiB_fence_sys_ns"] + lat["flag_host_sys_one_way_ns"] + lat["host_load_rtt_ns"]
    chain *= 1e-9
    rf["floors_us"] = {"per_direction": round(per_dir * 1e6, 3), "duplex": round(duplex * 1e6, 3),
                       "latency_chain": round(chain * 1e6, 3)}
    rf["frac_duplex"] = round(duplex / t_call_s, 4)
    rf["link_latency_ns"] = {k: round(v, 1) for k, v in lat.items()}
    rf["floors_note"] = ("frac = per_direction / t (each direction at its solo rate, both at once: not reachable, "
                         "the link gives about 170 + 170 GB/s with both directions streaming); "
                         "frac_duplex = duplex / t (each direction at its concurrent rate, measured in this run); "
                         "latency_chain = publish (4 KiB stores + the fence of the call's scope) + flag one way "
                         "(" + ("HBM, GPU scope" if gpu_scope else "host memory, system scope") + ") + one read "
                         "round trip, from ar_probe_host_link_latency")


def attach_traffic(row, prof, t_call_s, hbm_gbs):
    """DRAM bytes per call from the committed ncu summary, and the fraction of
    the measured HBM peak they reach at this call time."""
    if not prof:
        return
    rf = row["roofline"]
    rf["traffic"] = prof["dram_bytes_per_call"]
    if rf.get("bound") == "hbm" and prof.get("dram_bytes_per_call"):
        rf["dram_frac"] = round(prof["dram_bytes_per_call"] / t_call_s / 1e9 / hbm_gbs, 4)


def summarize(op, R, dtype, numel, slots, ms_steps, C, link, hbm_gbs, algo=None):
    isz = 8 if dtype == "c64" else 2
    S = numel * isz
    total_ms = sum(ms_steps)
    t_call = total_ms * 1e-3 / (len(ms_steps) * C)
    out_bytes = S * (R if op == "allgather" else 1)
    return {"op": op, "algo": algo, "R": R, "dtype": dtype, "numel": numel, "bytes_per_rank": S, "slots": slots,
            "us_per_call": round(t_call * 1e6, 3),
            "us_per_call_median_step": round(statistics.median(ms_steps) * 1e3 / C, 3),
            "algbw_gbs": round(out_bytes / t_call / 1e9, 3),
            "busbw_gbs": round(S / t_call / 1e9 * ((2 * (R - 1) / R) if op == "allreduce" else (R - 1) / R), 3)
            if R > 1 else None,
            "roofline": roofline(op, R, S, slots, t_call, link, hbm_gbs, algo), "calls": len(ms_steps) * C}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), and its architecture."""
    import platform
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() in ("Model name", "Model Name") and v.strip() and v.strip() != "-":
                name = v.strip()
                break
        if name:
            for line in out.splitlines():
                k, _, v = line.partition(":")
                if k.strip() == "Vendor ID" and v.strip():
                    name = f"{v.strip()} {name}"
                    break
    except Exception:
        pass
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        name = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return f"{name or platform.processor() or 'unknown'} ({platform.machine()})"


def time_oracle(xs, dtype, nthreads, seconds):
    """Calls per second of the oracle computing every rank's output of one call."""
    import oracle
    oracle.allreduce(xs, dtype, nthreads=nthreads)  # warm
    t0 = time.perf_counter()
    calls = 0
    while time.perf_counter() - t0 < seconds:
        oracle.allreduce(xs, dtype, nthreads=nthreads)  # every rank's output, as the job computes
        calls += 1
    return calls, time.perf_counter() - t0


def cpu_baseline(R, dtype, numel, seconds=8.0, config=2, dist="normal4"):
    """The oracle as it stands on a bounded sample of calls of the headline
    workload: once on all host cores (the reported value) and once on one core."""
    import oracle
    from tensor_decode_all_gb300 import inputs
    cores = oracle.max_threads()
    xs = inputs.allreduce_inputs(config, R, numel, dtype, dist, 0)
    S = numel * 2
    calls, dt = time_oracle(xs, dtype, cores, seconds)
    calls1, dt1 = time_oracle(xs, dtype, 1, seconds)
    return {"value": round(S * calls / dt / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "us_per_call": round(dt / calls * 1e6, 2), "cpu_model": cpu_model(),
            "single_core": {"value": round(S * calls1 / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                            "us_per_call": round(dt1 / calls1 * 1e6, 2),
                            "sample": f"{calls1} calls in {dt1:.1f} s"},
            "sample": f"{calls} calls of the headline workload (R={R} {dtype} N={numel}, all {R} ranks' "
                      f"outputs) in {dt:.1f} s on {cores} threads; then {calls1} calls in {dt1:.1f} s on one"}


LAUNCH_NAMES = {"rank": "one launch per rank per call (R non-blocking streams)",
                "fused": "one launch of every rank per call (ar_*_fused, one stream)",
                "all": "ar_allreduce_all on the R streams (one launch of every rank per call by default)"}

# name: (op, R, dtype, numel, slots, input config, distribution, calls per graph, timed steps[, options])
# options: algo (forced form), launch ("rank" | "fused" | "all"), tactics (ar_tactics fields).
# Workload 3 first: it is what the summary at the end of the line leads with.
EXTRA_WORKLOADS = {
    # workload 3 (R=8 bf16 48 x 8192, HBM slots), graphs of 100 calls and of one call
    "r8_bf16_393216_hbm": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20),
    "r8_bf16_393216_hbm_all": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20, {"launch": "all"}),
    "r8_bf16_393216_hbm_fused_flags": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20,
                                       {"launch": "fused", "tactics": {"cluster_max_bytes": 0}}),
    "r8_bf16_393216_hbm_fused": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20, {"launch": "fused"}),
    "r8_bf16_393216_hbm_graph1": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 1, 200),
    "r8_bf16_393216_hbm_fused_graph1": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 1, 200,
                                        {"launch": "fused"}),
    "r8_bf16_393216_hbm_all_graph1": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 1, 200,
                                      {"launch": "all"}),
    # workload 1 (one decode token) and the headline shape through the other launch forms
    "r2_fp16_4096_pinned": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", 100, 20),
    "r2_fp16_4096_pinned_all": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", 100, 20, {"launch": "all"}),
    "r2_fp16_131072_pinned_all": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100, 20,
                                  {"launch": "all"}),
    "r2_fp16_131072_pinned_fused_flags": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100, 20,
                                          {"launch": "fused", "tactics": {"cluster_max_bytes": 0}}),
    "r2_fp16_131072_pinned_graph1": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 1, 200),
    # workloads 2 and 1 with the ranks synchronising at system scope, flags in host
    # memory (two GPUs sharing only the host buffer need that placement); at that
    # scope the tagged-word form is the faster one at 8 KiB
    "r2_fp16_131072_pinned_sysscope": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100, 20,
                                       {"tactics": {"gpu_scope": 0}}),
    "r2_fp16_4096_pinned_sysscope": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", 100, 20,
                                     {"tactics": {"gpu_scope": 0, "tagged_max_bytes": 16 << 10}}),
    "r2_fp16_131072_pinned_all_graph1": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 1, 200,
                                         {"launch": "all"}),
    # large payloads in HBM (the HBM roofline)
    "r8_bf16_16MiB_hbm": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 10, 10),
    "r8_bf16_16MiB_hbm_oneshot": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 10, 10, {"algo": "oneshot"}),
    "r8_bf16_16MiB_hbm_all": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 10, 10, {"launch": "all"}),
    "r8_bf16_64MiB_hbm": ("allreduce", 8, "bf16", 32 << 20, "hbm", 5, "uniform", 4, 10),
    "r2_fp16_16MiB_hbm": ("allreduce", 2, "f16", 8 << 20, "hbm", 5, "uniform", 10, 10),
    # workload 4: complex64 allgather of 1000 x 500 shards
    "allgather_c64_r4_hbm": ("allgather", 4, "c64", 500000, "hbm", 4, None, 20, 10),
    "allgather_c64_r8_hbm": ("allgather", 8, "c64", 500000, "hbm", 4, None, 20, 10),
    "allgather_c64_r8_hbm_fused": ("allgather", 8, "c64", 500000, "hbm", 4, None, 20, 10, {"launch": "fused"}),
    "allgather_c64_r4_pinned": ("allgather", 4, "c64", 500000, "pinned", 4, None, 5, 5),
    "allgather_c64_r8_pinned": ("allgather", 8, "c64", 500000, "pinned", 4, None, 5, 5),
}


# Comparisons for --only (not part of the default line).
EXPERIMENT_WORKLOADS = {
    "x_r8_768K_fused_nopdl": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20,
                              {"launch": "fused", "pdl": False}),
    "x_r8_768K_all_nopdl": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20,
                            {"launch": "all", "pdl": False}),
    "x_r8_768K_all_rank": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20,
                           {"launch": "all", "tactics": {"all_fused": 0}}),
    "x_r8_16MiB_fused": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 10, 10, {"launch": "fused"}),
    "x_r8_16MiB_fused_flags": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 10, 10,
                               {"launch": "fused", "tactics": {"cluster_max_bytes": 0}}),
    "x_r2_256K_pinned_fused": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100, 20, {"launch": "fused"}),
    "x_r2_8K_pinned_fused": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", 100, 20, {"launch": "fused"}),
    "x_r2_8K_hbm_fused": ("allreduce", 2, "f16", 4096, "hbm", 1, "uniform", 100, 20, {"launch": "fused"}),
    "x_r2_8K_hbm": ("allreduce", 2, "f16", 4096, "hbm", 1, "uniform", 100, 20),
    "x_r8_1M_fused": ("allreduce", 8, "bf16", 1 << 19, "hbm", 5, "uniform", 100, 20, {"launch": "fused"}),
    "x_r8_1M": ("allreduce", 8, "bf16", 1 << 19, "hbm", 5, "uniform", 100, 20),
    # the allgather over the host link with its first-stage stores unpaced / paced at other rates
    "x_ag_r4_pinned_pace0": ("allgather", 4, "c64", 500000, "pinned", 4, None, 5, 5,
                             {"tactics": {"pace_mbs": 0, "pace_multi_mbs": 0}}),
    "x_ag_r8_pinned_pace0": ("allgather", 8, "c64", 500000, "pinned", 4, None, 5, 5,
                             {"tactics": {"pace_mbs": 0, "pace_multi_mbs": 0}}),
    "x_ag_r4_pinned_pace280": ("allgather", 4, "c64", 500000, "pinned", 4, None, 5, 5,
                               {"tactics": {"pace_multi_mbs": 280000}}),
    "x_ag_r4_pinned_pace160": ("allgather", 4, "c64", 500000, "pinned", 4, None, 5, 5,
                               {"tactics": {"pace_multi_mbs": 160000}}),
}

def _experiment_grids() -> dict:
    """Workload grids for --only comparisons:
    - workload 3 (and the same shape over the host link) with other two-shot
      sub-tiles and block caps: several tiles per block let HBM calls merge
      each reduced sub-tile into the next tile's flag round;
    - pinned-host slots with the ranks synchronising at system scope, flags
      in host memory (_sysscope), or at GPU scope, flags in HBM (_gpuscope);
    - the headline's shape and R=2 4 MiB at GPU scope at other paces."""
    grid = {}
    for sub in (64, 128, 256):
        for cap in (0, 48, 24, 12):
            tactics = {"tactics": {"twoshot_sub": sub, "max_blocks": cap}}
            grid[f"x_r8_768K_sub{sub}_b{cap}"] = ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100, 20,
                                                  tactics)
            grid[f"x_r8_768K_pinned_sub{sub}_b{cap}"] = ("allreduce", 8, "bf16", 393216, "pinned", 3, "normal",
                                                         50, 10, tactics)
    scoped = {
        "x_r2_256K_pinned": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100, 20),
        "x_r2_128K_pinned": ("allreduce", 2, "f16", 65536, "pinned", 5, "uniform", 100, 20),
        "x_r2_4M_pinned": ("allreduce", 2, "f16", 2 << 20, "pinned", 5, "uniform", 20, 10),
        "x_r4_1M_pinned": ("allreduce", 4, "bf16", 1 << 19, "pinned", 5, "uniform", 50, 10),
        "x_r8_256K_pinned": ("allreduce", 8, "bf16", 131072, "pinned", 5, "uniform", 50, 10),
        "x_ag_r4_pinned": ("allgather", 4, "c64", 500000, "pinned", 4, None, 5, 5),
        "x_r2_8K_pinned": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", 100, 20),
        "x_r2_32K_pinned": ("allreduce", 2, "f16", 16384, "pinned", 5, "uniform", 100, 20),
        "x_r8_64K_pinned": ("allreduce", 8, "bf16", 32768, "pinned", 5, "uniform", 100, 20),
    }
    for name, spec in scoped.items():
        for suffix, flags in (("sysscope", 0), ("gpuscope", 1)):
            grid[f"{name}_{suffix}"] = spec + ({"tactics": {"gpu_scope": flags}},)
    for pace in (0, 240000, 270000, 300000, 330000):
        grid[f"x_r2_256K_pinned_gpuscope_pace{pace // 1000}"] = (
            "allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100, 20,
            {"tactics": {"gpu_scope": 1, "pace_mbs": pace}})
        grid[f"x_r2_4M_pinned_gpuscope_pace{pace // 1000}"] = (
            "allreduce", 2, "f16", 2 << 20, "pinned", 5, "uniform", 20, 10,
            {"tactics": {"gpu_scope": 1, "pace_multi_mbs": pace}})
    return grid


EXPERIMENT_WORKLOADS.update(_experiment_grids())


# Order of the summary: the workloads a reader looks for first come last, so
# that they survive when only the end of the output is kept.
SUMMARY_LAST = ("r2_fp16_131072_pinned", "r2_fp16_4096_pinned", "r8_bf16_393216_hbm")


def workloads_summary(extras):
    """One short row per workload: [us/call, roofline fraction, ncu DRAM
    fraction or null, form, launch]; workload 3, 1 and the headline's shape last."""
    def rank(name):
        for i, prefix in enumerate(SUMMARY_LAST):
            if name.startswith(prefix):
                return i + 1
        return 0
    short = {"one launch per rank per call": "rank", "one launch of every rank per call": "fused",
             "ar_allreduce_all on the R streams": "all"}
    out = {"cols": ["us_per_call", "frac", "dram_frac", "form", "launch"]}
    for name in sorted(extras, key=rank):
        row = extras[name]
        rf = row["roofline"]
        out[name] = [row["us_per_call"], rf["frac"], rf.get("dram_frac"), row["algo"],
                     short.get(row["launch"].split(" (")[0], row["launch"])]
    return out


def run_push_ab(args, dist):
    """Push against pull, per-rank launches in graphs, bf16: the forced
    one-shot pull form, AUTO's pull form and the push form, each checked
    against the oracle on its first and last call."""
    import torch
    import tensor_decode_all_gb300 as tda
    torch.cuda.set_device(0)
    tda.build()
    hbm_gbs = float(measured_peaks().get("hbm_gbs", 6800.0))
    link = tda.ar_probe_host_link(64 << 20, 10)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    with open(args.push_ab, "w") as f:
        for slots in ("pinned", "hbm"):
            for R in (2, 4):
                for S in (8 << 10, 256 << 10, 4 << 20):
                    numel = S // 2
                    C = 100 if S <= (256 << 10) else 20
                    row = {"slots": slots, "R": R, "bytes_per_rank": S}
                    for label, algo in (("pull_oneshot", "oneshot"), ("pull_auto", None), ("push", "push")):
                        w = Workload("allreduce", R, "bf16", numel, slots, C, config=5, dist="uniform", algo=algo)
                        w.capture()
                        w.time_graph(1, 0, flush)
                        w.check(calls=(0, -1))
                        ms = w.time_graph(max(10, args.steps // 2), 2, flush)
                        w.check(calls=(0, -1))
                        sm = summarize("allreduce", R, "bf16", numel, slots, ms, C, link, hbm_gbs, w.algo)
                        row[label] = {"us": sm["us_per_call"], "form": w.algo, "frac": sm["roofline"]["frac"]}
                        w.close()
                    f.write(json.dumps(row) + "\n")
                    f.flush()
                    print(f"{slots:6s} R={R} S={S:>8d}: pull one-shot {row['pull_oneshot']['us']:9.2f}  "
                          f"pull AUTO ({row['pull_auto']['form']}) {row['pull_auto']['us']:9.2f}  "
                          f"push {row['push']['us']:9.2f} us/call", flush=True)
    return None


def run_only(args, dist):
    """Time only the named workloads (EXTRA_WORKLOADS names) and print one
    summary line each: for comparing forms, not the bench contract."""
    import torch
    import tensor_decode_all_gb300 as tda
    torch.cuda.set_device(0)
    tda.build()
    peaks = measured_peaks()
    hbm_gbs = float(peaks.get("hbm_gbs", 6800.0))
    link = tda.ar_probe_host_link(64 << 20, 10)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for name in args.only.split(","):
        spec = EXTRA_WORKLOADS.get(name) or EXPERIMENT_WORKLOADS[name]
        op, RR, dt, nn, sl, cfg, dd, cc, st = spec[:9]
        opts = spec[9] if len(spec) > 9 else {}
        wx = Workload(op, RR, dt, nn, sl, cc, config=cfg, dist=dd or "uniform", algo=opts.get("algo"),
                      launch=opts.get("launch", "rank"), tactics=opts.get("tactics"))
        if "pdl" in opts:
            wx.h.set_pdl(opts["pdl"])
        wx.capture()
        wx.time_graph(1, 0, flush)
        wx.check(calls=(0, -1))
        msx = wx.time_graph(max(st, args.steps), 2, flush)
        wx.check(calls=(-1,))
        row = summarize(op, RR, dt, nn, sl, msx, cc, link, hbm_gbs, wx.algo)
        print(json.dumps({"workload": name, "us": row["us_per_call"], "gbs": row["algbw_gbs"],
                          "frac": row["roofline"]["frac"], "form": row["algo"], "launch": wx.launch,
                          "cluster_max": wx.h.info().cluster_form}), flush=True)
        wx.close()
    return None


def run_ours(args, dist):
    import torch
    import tensor_decode_all_gb300 as tda
    dev = dist.local if torch.cuda.device_count() > dist.local else 0
    torch.cuda.set_device(dev)
    tda.build()
    peaks = measured_peaks()
    hbm_gbs = float(peaks.get("hbm_gbs", 6800.0))
    hbm_src = "MEASURED_PEAKS.json (of measured)" if "hbm_gbs" in peaks else "fallback 6.8 TB/s (of fallback)"
    link = tda.ar_probe_host_link(64 << 20, 10)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    R, numel, C = HEADLINE_R, HEADLINE_NUMEL, args.calls
    w = Workload("allreduce", R, "f16", numel, "pinned", C, config=2, dist="normal4")
    w.capture()
    w.time_graph(1, 0, flush)
    checked = w.check(calls=(0, 1, C // 2, -1))
    dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        ms = w.time_graph(args.steps, args.warmup, flush)
    clocks = clk.summary()
    checked += w.check(calls=(0, -1))
    total_s = dist.max(sum(ms) * 1e-3)
    head = summarize("allreduce", R, "f16", numel, "pinned", ms, C, link, hbm_gbs, w.algo)
    prof = profiled_traffic("r2_fp16_256KiB_pinned")
    if prof:
        head["roofline"]["traffic"] = prof["dram_bytes_per_call"]
        head["roofline"]["link_traffic"] = {"read": prof["link_read_bytes_per_call"],
                                            "write": prof["link_write_bytes_per_call"],
                                            "source": prof["source"]}
    add_link_floors(head["roofline"], tda.ar_probe_host_link_latency(200), link, head["us_per_call"] * 1e-6,
                    gpu_scope=bool(w.h.tactics()["gpu_scope"]))
    S = numel * 2
    n = dist.world
    value = n * S * len(ms) * C / total_s / 1e9

    e2e_times, h2d, d2h, serial_times, zero_times, zero_all_times = w.time_e2e(min(args.steps, 30))
    e2e_s = dist.max(sum(e2e_times) * 1e-3)
    pipelined_value = n * S * len(e2e_times) * C / e2e_s / 1e9
    zero_s = dist.max(sum(zero_times) * 1e-3)
    zero_value = n * S * len(zero_times) * C / zero_s / 1e9
    zero_all_s = dist.max(sum(zero_all_times) * 1e-3)
    zero_all_value = n * S * len(zero_all_times) * C / zero_all_s / 1e9
    e2e_forms = {"zero copy, ar_allreduce per rank": zero_value, "pipelined copies": pipelined_value,
                 "zero copy, ar_allreduce_all": zero_all_value}
    e2e_form = max(e2e_forms, key=e2e_forms.get)
    e2e_value = e2e_forms[e2e_form]
    serial_value = S * len(serial_times) * C / (sum(serial_times) * 1e-3) / 1e9
    checked += w.e2e_checked
    w.close()

    extras = {}
    if not args.no_extras:
        for name, spec in EXTRA_WORKLOADS.items():
            op, RR, dt, nn, sl, cfg, dd, cc, st = spec[:9]
            opts = spec[9] if len(spec) > 9 else {}
            wx = Workload(op, RR, dt, nn, sl, cc, config=cfg, dist=dd or "uniform", algo=opts.get("algo"),
                          launch=opts.get("launch", "rank"), tactics=opts.get("tactics"))
            wx.capture()
            wx.time_graph(1, 0, flush)
            wx.check(calls=(0, -1))
            msx = wx.time_graph(st, 2, flush)
            wx.check(calls=(-1,))
            extras[name] = summarize(op, RR, dt, nn, sl, msx, cc, link, hbm_gbs, wx.algo)
            extras[name]["launch"] = LAUNCH_NAMES[wx.launch]
            attach_traffic(extras[name], profiled_traffic(name), extras[name]["us_per_call"] * 1e-6, hbm_gbs)
            wx.close()

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": n, "steps": len(ms),
        "warmup": args.warmup, "ms_per_step": round(total_s * 1e3 / len(ms), 4),
        "us_per_call": head["us_per_call"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded 4*N(0,1) cast to fp16)",
        "config": headline_config(n), "calls_per_step": C,
        "roofline": head["roofline"],
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "form": e2e_form,
                "how": "the best of three forms through the C ABI with the step's inputs in pinned host memory "
                       "and its outputs read back to pinned host memory, CUDA events around each replay, outputs "
                       "checked against the oracle on the host. zero copy, ar_allreduce per rank: one CUDA graph of "
                       f"{C} ar_allreduce calls per rank whose in/out are the pinned host tensors themselves (the "
                       "kernels read the inputs from and write the outputs to host memory); zero copy, "
                       f"ar_allreduce_all: the same with {C} ar_allreduce_all calls (one launch of both ranks a "
                       "call, the cluster form); pipelined copies: one "
                       f"CUDA graph of {C} calls per rank in chunks of 10, a pinned-host->device copy of a chunk's "
                       "inputs, its calls, a device->pinned-host copy of its outputs, copies overlapping the "
                       "neighbouring chunks' calls",
                "zero_copy_value": round(zero_value, 3), "pipelined_value": round(pipelined_value, 3),
                "zero_copy_all_value": round(zero_all_value, 3),
                "serial_value": round(serial_value, 3),
                "serial_how": "one copy in, eager ar_allreduce calls, one copy out, no overlap"},
        "gpu_launches": len(ms) * C * R,
        "device_status": {"reads": Workload.status_reads, "timeouts": 0,
                          "how": "every workload's handle status (ar_status) read after its timed steps; a "
                                 "bounded device wait that ran out -- a rank kernel not co-resident with its "
                                 "peers -- would be recorded there and fail the run"},
        "clocks": clocks,
        "parity": f"bit-exact vs CPU oracle on {checked} sampled (call, rank) outputs",
        "host_link_probe_gbs": {k: round(v, 2) for k, v in link.items()},
        "hbm_peak": {"gbs": hbm_gbs, "source": hbm_src},
        "workloads": extras,
    }
    if dist.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(R, "f16", numel)
    # last, so that it survives in the end of the output a log keeps
    line["workloads_summary"] = workloads_summary(extras)
    return line


# name: (op, R, dtype, numel, slots, config, dist, calls per graph)
PROFILE_WORKLOADS = {
    "r2_fp16_256KiB_pinned": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 100),
    "r2_fp16_256KiB_pinned_1call": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 1),
    # the same with the ranks synchronising at system scope (flags in host memory)
    "r2_fp16_256KiB_pinned_sysscope_1call": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 1),
    "r8_bf16_768KiB_hbm": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100),
    "r8_bf16_768KiB_hbm_1call": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 1),
    "r8_bf16_16MiB_hbm_1call": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 1),
    "r2_fp16_16MiB_hbm_1call": ("allreduce", 2, "f16", 8 << 20, "hbm", 5, "uniform", 1),
    "allgather_c64_r4_hbm_1call": ("allgather", 4, "c64", 500000, "hbm", 4, "normal", 1),
    # graphs of 10 calls on distinct buffers: working sets that fit in L2 for one
    # call spill to DRAM over ten, so bytes / 10 is the steady-state figure
    "r2_fp16_16MiB_hbm_10call": ("allreduce", 2, "f16", 8 << 20, "hbm", 5, "uniform", 10),
    "allgather_c64_r4_hbm_10call": ("allgather", 4, "c64", 500000, "hbm", 4, "normal", 10),
    "r8_bf16_16MiB_hbm_oneshot_1call": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 1),
    "allgather_c64_r8_hbm_1call": ("allgather", 8, "c64", 500000, "hbm", 4, "normal", 1),
    "r8_bf16_768KiB_hbm_fused_1call": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 1),
    "r2_fp16_8KiB_pinned_1call": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", 1),
    # the two-shot form over the host link (AUTO's pick at these sizes)
    "r8_bf16_256KiB_pinned_1call": ("allreduce", 8, "bf16", 131072, "pinned", 5, "uniform", 1),
    "r4_bf16_1MiB_pinned_1call": ("allreduce", 4, "bf16", 1 << 19, "pinned", 5, "uniform", 1),
    "r8_bf16_768KiB_hbm_all": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 100),
    "r8_bf16_768KiB_hbm_all_1call": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", 1),
    "r2_fp16_256KiB_pinned_all_1call": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", 1),
    "r8_bf16_16MiB_hbm_all_1call": ("allreduce", 8, "bf16", 8 << 20, "hbm", 5, "uniform", 1),
}


def run_profile(args, dist):
    """Only graph replays (no eager rank calls: a profiler that serialises
    kernels would keep the ranks of one call apart).  Prints timing, no JSON."""
    import torch
    import tensor_decode_all_gb300 as tda
    torch.cuda.set_device(0)
    tda.build()
    op, R, dt, n, sl, cfg, dd, C = PROFILE_WORKLOADS[args.profile]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    launch = "all" if "_all" in args.profile else "fused" if "fused" in args.profile else "rank"
    w = Workload(op, R, dt, n, sl, C, config=cfg, dist=dd, algo="oneshot" if "oneshot" in args.profile else None,
                 launch=launch, tactics={"gpu_scope": 0} if "sysscope" in args.profile else None)
    w.capture()
    ms = w.time_graph(args.steps, args.warmup, flush)
    w.check(calls=(0, -1))
    print(f"profile {args.profile}: {len(ms)} steps x {C} calls, "
          f"{sum(ms) * 1e3 / (len(ms) * C):.3f} us/call (graph)", flush=True)
    w.close()
    return None


TRACE_WORKLOADS = {
    "config 2: R=2 fp16 256 KiB pinned": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", False),
    "config 2, system scope (flags in host memory)": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4",
                                                      "sysscope"),
    "config 1: R=2 fp16 8 KiB pinned": ("allreduce", 2, "f16", 4096, "pinned", 1, "uniform", False),
    "config 3: R=8 bf16 768 KiB HBM": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", False),
    "config 3, one cooperative launch (flag form)": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", "flags"),
    "config 3, ar_allreduce_all (cluster form)": ("allreduce", 8, "bf16", 393216, "hbm", 3, "normal", "all"),
    "config 2, ar_allreduce_all (cluster form)": ("allreduce", 2, "f16", 131072, "pinned", 2, "normal4", "all"),
}


def sm_clock_mhz(dev: int) -> float:
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(dev), "--query-gpu=clocks.sm", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=10).stdout.strip()
        return float(out.splitlines()[0])
    except Exception:
        return float(measured_peaks().get("sm_max_mhz", 2070.0))


def run_trace(args, dist):
    """Each main workload in a graph of 100 calls with the device trace on:
    overlap of the rank kernels and the phases of a call (not a timing run)."""
    import torch
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import trace
    torch.cuda.set_device(0)
    tda.build()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    out = {}
    for name, (op, R, dt, n, sl, cfg, dd, mode) in TRACE_WORKLOADS.items():
        C = 100
        w = Workload(op, R, dt, n, sl, C, config=cfg, dist=dd,
                     launch="fused" if mode == "flags" else "all" if mode == "all" else "rank",
                     tactics={"cluster_max_bytes": 0} if mode == "flags" else
                     {"gpu_scope": 0} if mode == "sysscope" else None)
        buf = trace.start(w.h, C)
        w.capture()
        w.time_graph(3, 0, flush)
        buf.zero_()
        ms = w.time_graph(1, 0, flush)
        w.check(calls=(0, -1))
        rec = trace.records(buf)
        summary = trace.summarize(rec, sm_clock_mhz(0))
        summary["graph_us_per_call"] = round(ms[0] * 1e3 / C, 3)
        out[name] = summary
        w.close()
        print(name, json.dumps(summary), flush=True)
    with open(args.trace, "w") as f:
        json.dump(out, f, indent=1)
    return None


def run_reference(args, dist):
    """The CPU oracle as the reference arm: same workload, metric and unit."""
    if dist.rank != 0:
        return None
    import oracle
    from tensor_decode_all_gb300 import inputs
    oracle.build()
    R, numel, dtype = HEADLINE_R, HEADLINE_NUMEL, "f16"
    cores = oracle.max_threads()
    xs = inputs.allreduce_inputs(2, R, numel, dtype, "normal4", 0)
    calls_per_step = 20
    for _ in range(args.warmup):
        for _ in range(calls_per_step):
            oracle.allreduce(xs, dtype, nthreads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for _ in range(calls_per_step):
            oracle.allreduce(xs, dtype, nthreads=cores)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    S = numel * 2
    value = S * calls_per_step * len(times) / total / 1e9
    sample = f"{calls_per_step} calls per step of R={R} {dtype} N={numel} (all ranks' outputs), {cores} threads"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": dist.world,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": round(total * 1e3 / len(times), 3),
            "us_per_call": round(total / (len(times) * calls_per_step) * 1e6, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded 4*N(0,1) cast to fp16)",
            "config": dict(headline_config(dist.world),
                           executor="the CPU oracle on the host cores: the same workload and outputs; "
                                    "slots, graphs and L2 flushing do not apply"),
            "calls_per_step": calls_per_step,
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_sweep(args, dist):
    """Payload sweep 2 KiB..64 MiB, fp16/bf16, R=2/4/8, pinned vs HBM slots;
    oracle parity on the first and last call of every cell."""
    import torch
    import tensor_decode_all_gb300 as tda
    torch.cuda.set_device(0)
    tda.build()
    peaks = measured_peaks()
    hbm_gbs = float(peaks.get("hbm_gbs", 6800.0))
    link = tda.ar_probe_host_link(64 << 20, 10)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    cells = []
    for slots in args.sweep_slots.split(","):
        for dtype in args.sweep_dtypes.split(","):
            for R in [int(x) for x in args.sweep_ranks.split(",")]:
                for k in range(11, 27):
                    S = 1 << k
                    if not (args.sweep_min_kib << 10) <= S <= (args.sweep_max_kib << 10):
                        continue
                    both = args.sweep_both and R >= 3 and (64 << 10) <= S <= (8 << 20)
                    for algo in (("oneshot", "twoshot") if both else (args.sweep_algo,)):
                        cells.append((slots, dtype, R, S, algo))
    with open(args.sweep, "w") as f:
        for slots, dtype, R, S, algo in cells:
            numel = S // 2
            total = args.sweep_calls
            if slots == "pinned" and R * S >= (64 << 20):
                total = min(total, 100)  # ~20 ms per call over the host link: bound the wall time
            # at least 4 calls per graph, so a step is not dominated by one graph launch
            C = max(4, min(100, (256 << 20) // max(1, R * S * 2)))
            steps = max(1, total // C)
            w = Workload("allreduce", R, dtype, numel, slots, C, config=5, dist="uniform", algo=algo,
                         launch=args.sweep_launch or ("fused" if args.sweep_fused else "rank"),
                         tactics=json.loads(args.sweep_tactics) if args.sweep_tactics else None)
            w.capture()
            w.time_graph(1, 0, flush)
            w.check(calls=(0, -1))
            ms = w.time_graph(steps, 2, flush)
            w.check(calls=(0, -1))
            row = summarize("allreduce", R, dtype, numel, slots, ms, C, link, hbm_gbs, w.algo)
            row["parity"] = "bit-exact (first and last call)"
            row["launch"] = w.launch
            row["tactics"] = args.sweep_tactics
            row["host_link_probe_gbs"] = {k: round(v, 2) for k, v in link.items()}
            f.write(json.dumps(row) + "\n")
            f.flush()
            w.close()
            print(f"{slots:6s} {dtype:4s} R={R} S={S:>9d} {w.algo:8s}: {row['us_per_call']:9.2f} us/call "
                  f"{row['algbw_gbs']:9.2f} GB/s frac={row['roofline']['frac']}", flush=True)
    return None


def main():
    args = parse()
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            line = run_reference(args, dist)
        elif args.profile:
            line = run_profile(args, dist)
        elif args.trace:
            line = run_trace(args, dist)
        elif args.sweep:
            line = run_sweep(args, dist)
        elif args.only:
            line = run_only(args, dist)
        elif args.push_ab:
            line = run_push_ab(args, dist)
        else:
            line = run_ours(args, dist)
        if line is not None and dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
