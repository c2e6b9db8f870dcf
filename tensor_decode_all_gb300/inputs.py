"""Seeded synthetic inputs for the five workloads (shared by tests, bench, smoke).

This module holds none of the method's arithmetic: it only draws numbers.
Generator: numpy PCG64 (``np.random.default_rng``) with
``seed = 20261202 + 1000 * config + 10 * rank + call``.  Values are drawn in
float32 and cast to the element type with round-to-nearest-even (numpy's cast
for fp16, torch's for bf16); the cast is part of the input recipe, not of the
operation under test.

Workloads (the decode-time all-reduce shapes the pages describe; there is no
dataset):
  1  R=2, fp16, N=4096 (one decode token, hidden 4096), U[-1,1], pinned-host slots
  2  R=2, fp16, N=131072 (256 KiB, the host all-reduce's payload cap), 4*N(0,1), pinned-host
  3  R=8, bf16, N=393216 (48 rows x hidden 8192, the decode-sized max_numel), N(0,1), HBM
  4  allgather, complex64 shards of 1000x500, re/im N(0,1), R=4 and 8, HBM and pinned-host
     (long runs: each rank's call-0 shard rotated by call + 1 elements per call)
  5  sweep: 2 KiB..64 MiB per rank, fp16/bf16, R=2/4/8, U[-1,1], both slot kinds
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202

CONFIGS = {
    1: dict(name="r2_fp16_4096_pinned", R=2, dtype="f16", numel=4096, dist="uniform", slots="pinned", calls=100),
    2: dict(name="r2_fp16_131072_pinned", R=2, dtype="f16", numel=131072, dist="normal4", slots="pinned", calls=1000),
    3: dict(name="r8_bf16_393216_hbm", R=8, dtype="bf16", numel=393216, dist="normal", slots="hbm", calls=1000),
    4: dict(name="allgather_c64_1000x500", R=(4, 8), dtype="c64", shape=(1000, 500), dist="normal",
            slots=("hbm", "pinned"), calls=1000),
    5: dict(name="sweep", R=(2, 4, 8), dtype=("f16", "bf16"), bytes=[2 ** k for k in range(11, 27)],
            dist="uniform", slots=("pinned", "hbm"), calls=1000),
}


def seed_for(config: int, rank: int, call: int) -> int:
    return BASE_SEED + 1000 * int(config) + 10 * int(rank) + int(call)


def draw(dist: str, n: int, rng: np.random.Generator) -> np.ndarray:
    """n float32 values from the named distribution."""
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, n).astype(np.float32)
    if dist == "normal":
        return rng.standard_normal(n, dtype=np.float32)
    if dist == "normal4":
        return (4.0 * rng.standard_normal(n, dtype=np.float32)).astype(np.float32)
    raise ValueError(dist)


def to_bits(values: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> 16-bit patterns (uint16) of fp16 or bf16, round to nearest even."""
    values = np.ascontiguousarray(values, np.float32)
    if dtype in ("f16", "fp16"):
        with np.errstate(over="ignore"):
            return values.astype(np.float16).view(np.uint16)
    if dtype in ("bf16",):
        import torch
        return torch.from_numpy(values).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def allreduce_inputs(config: int, R: int, numel: int, dtype: str, dist: str, call: int = 0):
    """R uint16 arrays of numel elements: rank r's input of the given call."""
    out = []
    for r in range(R):
        rng = np.random.default_rng(seed_for(config, r, call))
        out.append(to_bits(draw(dist, numel, rng), dtype))
    return out


def allgather_inputs(config: int, R: int, numel: int, call: int = 0):
    """R complex64 arrays of numel elements (real and imaginary parts N(0,1))."""
    out = []
    for r in range(R):
        rng = np.random.default_rng(seed_for(config, r, call))
        re = rng.standard_normal(numel, dtype=np.float32)
        im = rng.standard_normal(numel, dtype=np.float32)
        z = np.empty(numel, np.complex64)
        z.real = re
        z.imag = im
        out.append(z)
    return out


_BASE_SHARDS = {}


def allgather_inputs_rotated(config: int, R: int, numel: int, call: int):
    """R complex64 shards for call `call` of a long run, cheaply: rank r's base
    shard (allgather_inputs of call 0, re/im N(0,1)) rotated by call + 1
    elements.  Every call and every rank gets its own contents, so a shard
    read from the wrong call or rank cannot pass for the right one; the values
    are still N(0,1) draws.  (Drawing 1000 calls of fresh 4 MB shards takes
    minutes; a rotation is a copy.)"""
    key = (config, R, numel)
    if key not in _BASE_SHARDS:
        _BASE_SHARDS.clear()
        _BASE_SHARDS[key] = allgather_inputs(config, R, numel, 0)
    return [np.roll(b, (call + 1) % max(numel, 1)) for b in _BASE_SHARDS[key]]


def numel_for_bytes(nbytes: int, dtype: str) -> int:
    return nbytes // (8 if dtype == "c64" else 2)
