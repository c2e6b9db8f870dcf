"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test checks the oracle (oracle/oracle.c) against a fact fixed by the pages
or by mathematics, never against a retyping of its own formula:

* hand-derived cases (tests/golden/allreduce_cases.txt), each with its
  derivation;
* closed form for R = 2: rounding a binary16/bfloat16 sum first to binary32
  and then to the 16-bit format is innocuous, because binary32 has
  24 >= 2*11 + 2 bits (S. Figueroa, "When is double rounding innocuous?",
  SIGNUM Newsletter 30(3), 1995).  So the two-rank result must equal the
  correctly rounded sum RNE16(a + b), which "[Kernel] Two-rank FP16 all-reduce
  through pinned host memory for GPUs without P2P" (section "Purpose") also
  states: a single FP16 rounding, independent of operand order, matching a
  two-rank NCCL sum bit for bit;
* library routines for the special cases that reduce to them: numpy's
  float64 -> float16 and float32 -> float16 casts and torch's
  float32 -> bfloat16 cast (all round to nearest even);
* an independent arithmetic rounding (frexp / rint / ldexp) for bfloat16;
* invariants: R = 1 is the identity, the two-rank sum commutes, the allgather
  is a concatenation.
"""
import math
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "allreduce_cases.txt")


def _is_nan16(bits, fmt):
    bits = np.asarray(bits, np.uint16)
    if fmt == "f16":
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def _assert_same(got, want, fmt, what=""):
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    gn, wn = _is_nan16(got, fmt), _is_nan16(want, fmt)
    assert np.array_equal(gn, wn), f"{what}: NaN-ness differs at {np.flatnonzero(gn != wn)[:8]}"
    ok = gn | (got == want)
    if not ok.all():
        i = np.flatnonzero(~ok)[:8]
        raise AssertionError(f"{what}: {ok.size - ok.sum()} mismatches, first at {i}: "
                             f"got {[hex(x) for x in got[i]]} want {[hex(x) for x in want[i]]}")


# ---------------------------------------------------------------- golden cases

def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for ln, line in enumerate(f, 1):
            body = line.split("#", 1)[0].split()
            if not body:
                continue
            fmt, expected, xs = body[0], body[1], body[2:]
            cases.append(pytest.param(fmt, expected, [int(x, 16) for x in xs], id=f"L{ln}"))
    return cases


@pytest.mark.parametrize("fmt,expected,xs", _golden_cases())
def test_golden_case(fmt, expected, xs):
    ins = [np.array([x], np.uint16) for x in xs]
    outs = oracle.allreduce(ins, fmt)
    for out in outs:  # every rank gets the same bits
        if expected == "nan":
            assert _is_nan16(out, fmt)[0], hex(out[0])
        else:
            assert out[0] == int(expected, 16), (hex(out[0]), expected)


# ------------------------------------------------------------ conversions alone

def test_widen_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen("f16", bits)
    want = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_widen_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen("bf16", bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _f32_samples(n, seed):
    """Random binary32 bit patterns over every exponent, plus the edges."""
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    edges = []
    for e in list(range(0, 8)) + list(range(100, 160)) + list(range(248, 256)):
        for m in (0, 1, 0x1FFF, 0x2000, 0x2001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xFFFF,
                  0x10000, 0x7FFFFF, 0x400000, 0x3FFFFF):
            for s in (0, 1):
                edges.append((s << 31) | (e << 23) | m)
    return np.concatenate([u, np.array(edges, np.uint32)]).view(np.float32)


def test_narrow_f16_matches_numpy_cast():
    x = _f32_samples(1 << 21, 11)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    _assert_same(oracle.narrow("f16", x), want, "f16", "f32->f16")


def test_narrow_bf16_matches_torch_cast():
    x = _f32_samples(1 << 21, 12)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    _assert_same(oracle.narrow("bf16", x), want, "bf16", "f32->bf16")


# ------------------------------------------------ R = 2: the closed form, fp16

def _f16_pair_chunk(args):
    """Worker: oracle vs RNE16(a + b) for a block of a-values.

    The exact sum of two binary16 values needs at most 40 significant bits, so
    the binary64 sum is exact, and numpy's float64 -> float16 cast rounds it
    once, to nearest even: that is the correctly rounded sum.
    """
    a_lo, a_hi, stride = args
    import numpy as np
    import oracle as orc
    bad = 0
    first = None
    for a0 in range(a_lo, a_hi, 64):
        a = np.arange(a0, min(a0 + 64, a_hi), dtype=np.uint32)
        if stride == 1:
            b = np.arange(65536, dtype=np.uint32)
            A = np.repeat(a, b.size).astype(np.uint16)
            B = np.tile(b, a.size).astype(np.uint16)
        else:
            # every a, and for each a the b-values with one low-bit pattern that
            # rotates with a, so all (a, b mod stride) combinations occur
            j = np.arange(65536 // stride, dtype=np.uint32)
            A = np.repeat(a, j.size)
            B = (np.tile(j, a.size) * stride + (A * 5 + 3) % stride)
            A = A.astype(np.uint16)
            B = B.astype(np.uint16)
        got = orc.allreduce([A, B], "f16", ranks=[0])[0]
        with np.errstate(over="ignore", invalid="ignore"):
            want = (A.view(np.float16).astype(np.float64)
                    + B.view(np.float16).astype(np.float64)).astype(np.float16).view(np.uint16)
        gn = ((got & 0x7C00) == 0x7C00) & ((got & 0x3FF) != 0)
        wn = ((want & 0x7C00) == 0x7C00) & ((want & 0x3FF) != 0)
        mism = (gn != wn) | (~gn & (got != want))
        if mism.any():
            bad += int(mism.sum())
            if first is None:
                i = int(np.flatnonzero(mism)[0])
                first = (int(A[i]), int(B[i]), int(got[i]), int(want[i]))
    return bad, first


def test_f16_two_rank_sum_is_correctly_rounded():
    """Every one of the 2^32 ordered pairs (about 40 s on 8 cores).  With
    TDA_ORACLE_QUICK=1: every a and a rotating 1/8 of the b-values."""
    stride = 8 if os.environ.get("TDA_ORACLE_QUICK") == "1" else 1
    oracle.build()
    nproc = max(1, min(8, os.cpu_count() or 1))
    step = 65536 // (nproc * 8)
    jobs = [(lo, min(lo + step, 65536), stride) for lo in range(0, 65536, step)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(nproc) as pool:
        res = pool.map(_f16_pair_chunk, jobs)
    bad = sum(r[0] for r in res)
    firsts = [r[1] for r in res if r[1] is not None]
    assert bad == 0, f"{bad} pairs differ from RNE16(a+b); first (a, b, got, want) = {firsts[0]}"


# ------------------------------------------------ R = 2: the closed form, bf16

def _bf16_round_independent(s):
    """Round float64 values to bfloat16 bit patterns, by arithmetic.

    frexp gives s = f * 2^e with 0.5 <= |f| < 1, so the leading bit has exponent
    e-1; bfloat16 keeps 8 significant bits for exponents >= -126 and a fixed
    quantum 2^-133 below.  rint rounds half to even.  Overflow past the largest
    finite bfloat16 gives inf.
    """
    s = np.asarray(s, np.float64)
    out = np.empty(s.shape, np.uint16)
    fin = np.isfinite(s)
    f, e = np.frexp(s[fin])
    q = np.maximum(e - 1, -126) - 7
    k = np.rint(np.ldexp(s[fin], -q))
    r = np.ldexp(k, q)
    big = np.abs(r) >= 2.0**128
    r32 = r.astype(np.float32)  # exact: r is a bfloat16 value (or overflowed)
    bits = (r32.view(np.uint32) >> 16).astype(np.uint16)
    bits[big] = np.where(r[big] > 0, 0x7F80, 0xFF80)
    # signed zero: the binary64 sum already carries IEEE's sign of zero
    out[fin] = bits
    nf = ~fin
    out[nf] = np.where(np.isnan(s[nf]), 0x7FC0, np.where(s[nf] > 0, 0x7F80, 0xFF80))
    return out


def _bf16_specials():
    v = set()
    for e in list(range(0, 4)) + list(range(118, 136)) + list(range(250, 256)):
        for m in (0, 1, 2, 0x3F, 0x40, 0x41, 0x7E, 0x7F):
            for s in (0, 1):
                v.add((s << 15) | (e << 7) | m)
    return np.array(sorted(v), np.uint16)


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_two_rank_sum_is_correctly_rounded():
    sp = _bf16_specials()
    A1 = np.repeat(sp, sp.size)
    B1 = np.tile(sp, sp.size)
    rng = np.random.default_rng(7)
    n = 1 << 22
    A2 = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    # partners within a few binades of A2, where rounding decisions happen
    shift = rng.integers(-10, 11, n).astype(np.int32)
    e2 = np.clip(((A2.astype(np.int32) >> 7) & 0xFF) + shift, 0, 254)
    B2 = ((rng.integers(0, 2, n) << 15) | (e2 << 7) | rng.integers(0, 128, n)).astype(np.uint16)
    A = np.concatenate([A1, A2])
    B = np.concatenate([B1, B2])
    got = oracle.allreduce([A, B], "bf16", ranks=[0])[0]
    with np.errstate(over="ignore", invalid="ignore"):
        s = _bf16_to_f64(A) + _bf16_to_f64(B)  # RNE53 of the exact sum: innocuous (53 >= 2*8+2)
    want = _bf16_round_independent(s)
    _assert_same(got, want, "bf16", "bf16 a+b")


# --------------------------------------------------------------- invariants

@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_single_rank_is_identity(fmt):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.allreduce([bits], fmt)[0]
    nan = _is_nan16(bits, fmt)
    assert np.array_equal(got[~nan], bits[~nan])
    assert _is_nan16(got[nan], fmt).all()


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_two_rank_sum_commutes_and_ranks_agree(fmt):
    rng = np.random.default_rng(3)
    a = rng.integers(0, 65536, 1 << 20, dtype=np.uint32).astype(np.uint16)
    b = rng.integers(0, 65536, 1 << 20, dtype=np.uint32).astype(np.uint16)
    ab = oracle.allreduce([a, b], fmt)
    ba = oracle.allreduce([b, a], fmt)
    _assert_same(ab[0], ab[1], fmt, "rank 0 vs rank 1")
    _assert_same(ab[0], ba[0], fmt, "a+b vs b+a")


# ------------------------------------------ R > 2: library routines in rank order

def _library_rank_order(ins, fmt):
    """numpy float32 adds, left to right, then the library's RNE cast."""
    acc = None
    for x in ins:
        if fmt == "f16":
            v = x.view(np.float16).astype(np.float32)
        else:
            v = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()
        acc = v.copy() if acc is None else (acc + v).astype(np.float32)
    if fmt == "f16":
        with np.errstate(over="ignore"):
            return acc.astype(np.float16).view(np.uint16)
    return torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("R", [3, 4, 5, 8])
def test_rank_order_sum_matches_library(fmt, R):
    rng = np.random.default_rng(100 + R)
    n = 1 << 18
    ins = []
    for p in range(R):
        # a mix: uniform [-1, 1], 4*N(0,1), wide exponent spread, random patterns
        vals = np.concatenate([rng.uniform(-1, 1, n // 4), 4 * rng.standard_normal(n // 4),
                               rng.standard_normal(n // 4) * np.exp2(rng.integers(-30, 16, n // 4))])
        vals = vals.astype(np.float32)
        if fmt == "f16":
            with np.errstate(over="ignore"):
                bits = vals.astype(np.float16).view(np.uint16)
        else:
            bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        rnd = rng.integers(0, 65536, n - bits.size, dtype=np.uint32).astype(np.uint16)
        ins.append(np.concatenate([bits, rnd]))
    got = oracle.allreduce(ins, fmt)
    want = _library_rank_order(ins, fmt)
    for r in range(R):
        _assert_same(got[r], want, fmt, f"R={R} rank {r}")


def test_three_rank_brute_force_small_set():
    """All 64^3 ordered triples of a set holding zeros, subnormals, normals of
    every scale, the largest finite values and infinities."""
    vals = [0x0000, 0x8000, 0x0001, 0x8001, 0x0002, 0x03FF, 0x0400, 0x8400, 0x1000, 0x1400,
            0x2000, 0x3400, 0x3800, 0xB800, 0x3BFF, 0x3C00, 0xBC00, 0x3C01, 0xBC01, 0x3E00,
            0x4000, 0xC000, 0x4200, 0x4400, 0x4B80, 0x4C00, 0x5000, 0x5800, 0x6000, 0x6400,
            0xE400, 0x6401, 0x6800, 0xE800, 0x6801, 0x7000, 0x7800, 0xF800, 0x7BFE, 0x7BFF,
            0xFBFF, 0x7C00, 0xFC00, 0x0010, 0x0200, 0x1C00, 0x2E66, 0x3555, 0x3A00, 0xBA00,
            0x4155, 0x4800, 0xC800, 0x5555, 0x5A00, 0x6C00, 0x7400, 0xF400, 0x7A00, 0x3FFF,
            0x43FF, 0x47FF, 0x0401, 0x7E00]
    v = np.array(vals, np.uint16)
    assert v.size == 64
    a = np.repeat(v, 64 * 64)
    b = np.tile(np.repeat(v, 64), 64)
    c = np.tile(v, 64 * 64)
    got = oracle.allreduce([a, b, c], "f16", ranks=[0])[0]
    _assert_same(got, _library_rank_order([a, b, c], "f16"), "f16", "R=3 brute force")


# ------------------------------------------------------------------- allgather

@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_allgather_is_concatenation(R):
    rng = np.random.default_rng(R)
    shards = [(rng.standard_normal(1000) + 1j * rng.standard_normal(1000)).astype(np.complex64)
              for _ in range(R)]
    outs = oracle.allgather(shards)
    want = np.concatenate(shards).view(np.uint8)
    for r in range(R):
        assert np.array_equal(outs[r], want)
        # rank p's shard sits at bytes [p*S, (p+1)*S)
        S = shards[0].nbytes
        for p in range(R):
            assert np.array_equal(outs[r][p * S:(p + 1) * S], shards[p].view(np.uint8))


def test_allgather_odd_byte_sizes():
    rng = np.random.default_rng(5)
    shards = [rng.integers(0, 256, 13, dtype=np.uint16).astype(np.uint8) for _ in range(3)]
    assert np.array_equal(oracle.allgather(shards)[2], np.concatenate(shards))
