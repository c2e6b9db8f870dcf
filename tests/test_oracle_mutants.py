"""The pins must catch plausible mistakes in the oracle.

Each case copies oracle/oracle.c to a temporary directory, plants one mistake
by a text substitution, builds the copy with gcc and checks that the
hand-derived cases in tests/golden/allreduce_cases.txt (plus a few library
cross-checks) reject it.  The committed oracle is never modified.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "allreduce_cases.txt")

MUTANTS = {
    "ties_away_from_zero": ("(rem > half || (rem == half && (k & 1ull)))", "(rem >= half)"),
    "truncate": ("if (rem > half || (rem == half && (k & 1ull))) k++;", ";"),
    "accumulate_from_plus_zero": ("float acc = widen(fmt, ins[0][i]);\n            for (int p = 1; p < R; p++) {",
                                  "float acc = 0.0f;\n            for (int p = 0; p < R; p++) {"),
    "accumulate_in_double": ("float acc = widen(fmt, ins[0][i]);", "double acc = widen(fmt, ins[0][i]);"),
    "reverse_rank_order": ("acc = acc + widen(fmt, ins[p][i]);", "acc = acc + widen(fmt, ins[R - p][i]) + 0.0f * widen(fmt, ins[0][i]);"),
    "round_after_each_add": ("acc = acc + widen(fmt, ins[p][i]);", "acc = widen(fmt, narrow(fmt, acc + widen(fmt, ins[p][i])));"),
    "flush_subnormal_results": ("if (k < (1ull << frac)) return (uint16_t)(sign | (uint16_t)k);",
                                "if (k < (1ull << frac)) return sign;"),
    "widen_subnormal_exponent_off_by_one": ("uint32_t e32 = (uint32_t)(127 - 14 - k);", "uint32_t e32 = (uint32_t)(127 - 15 - k);"),
    "overflow_test_one_binade_late": ("if (E > emax) return", "if (E > emax + 1) return"),
    "bf16_bias_wrong": ("narrow_f32(x, 7, -126, 127, 127)", "narrow_f32(x, 7, -126, 127, 126)"),
}


def _golden():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            body = line.split("#", 1)[0].split()
            if body:
                out.append((body[0], body[1], [int(x, 16) for x in body[2:]]))
    return out


def _build(tmp_path, text):
    src = tmp_path / "m.c"
    so = tmp_path / "m.so"
    src.write_text(text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-w",
                    "-o", str(so), str(src)], check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    vp = ctypes.c_void_p
    lib.oracle_allreduce.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp),
                                     ctypes.POINTER(vp), ctypes.c_size_t, ctypes.c_int]
    return lib


def _run(lib, fmt, xs):
    ins = [np.array([x], np.uint16) for x in xs]
    out = np.zeros(1, np.uint16)
    ip = (ctypes.c_void_p * len(ins))(*[a.ctypes.data for a in ins])
    op = (ctypes.c_void_p * len(ins))(*([out.ctypes.data] + [None] * (len(ins) - 1)))
    assert lib.oracle_allreduce(len(ins), 1 if fmt == "f16" else 2, ip, op, 1, 1) == 0
    return int(out[0])


def _golden_failures(lib):
    fails = 0
    for fmt, expected, xs in _golden():
        got = _run(lib, fmt, xs)
        if expected == "nan":
            mask_e, mask_m = (0x7C00, 0x3FF) if fmt == "f16" else (0x7F80, 0x7F)
            fails += not ((got & mask_e) == mask_e and (got & mask_m) != 0)
        else:
            fails += got != int(expected, 16)
    return fails


def test_unmutated_copy_passes(tmp_path):
    lib = _build(tmp_path, open(SRC).read())
    assert _golden_failures(lib) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert old in text, f"mutation site for {name} not found"
    lib = _build(tmp_path, text.replace(old, new, 1))
    assert _golden_failures(lib) > 0, f"the golden cases do not catch mutant {name}"


def _segments(fmt, R, seed):
    """Inputs by segment: near 1 (ties and carries), random patterns, tiny
    values (subnormal results), values near the largest finite (overflow),
    specials, and cancellation -- rank 0 a large b, rank 1 a small s that a
    binary32 sum with b drops, rank 2 exactly -b -- where the result depends
    on the precision of the running sum and on the order of the ranks."""
    rng = np.random.default_rng(seed)
    one, top, tiny = (0x3C00, 0x7BFF, 0x0800) if fmt == "f16" else (0x3F80, 0x7F7F, 0x0100)
    big_lo, big_hi, small_lo, small_hi = ((0x6000, 0x7800, 0x0400, 0x1C00) if fmt == "f16"
                                          else (0x6000, 0x7000, 0x2000, 0x3000))
    big = rng.integers(big_lo, big_hi, 200).astype(np.uint16)
    xs = []
    for r in range(R):
        sign = rng.integers(0, 2, 200).astype(np.uint16) << 15
        small = sign | rng.integers(small_lo, small_hi, 200).astype(np.uint16)
        cancel = big if r == 0 else (big ^ np.uint16(0x8000)) if r == 2 else small
        segs = [one + rng.integers(-300, 300, 200),
                rng.integers(0, 65536, 200),
                sign | rng.integers(0, tiny, 200).astype(np.uint16),
                top - rng.integers(0, 40, 200),
                np.resize(np.array([0x0000, 0x8000, 0x0001, 0x8001, top, top | 0x8000, one, one | 0x8000],
                                   np.uint16), 200),
                cancel]
        xs.append(np.concatenate([np.asarray(s).astype(np.uint16) for s in segs]))
    return xs


def _exact_failures(lib):
    from tests.test_oracle_exact import _is_nan, exact_rank_order
    fails = 0
    for fmt in ("f16", "bf16"):
        for R in (3, 5):
            xs = _segments(fmt, R, 10 * R + (fmt == "bf16"))
            n = xs[0].size
            out = np.zeros(n, np.uint16)
            ip = (ctypes.c_void_p * R)(*[a.ctypes.data for a in xs])
            op = (ctypes.c_void_p * R)(*([out.ctypes.data] + [None] * (R - 1)))
            assert lib.oracle_allreduce(R, 1 if fmt == "f16" else 2, ip, op, n, 1) == 0
            want = exact_rank_order(xs, fmt)
            gn, wn = _is_nan(out, fmt), _is_nan(want, fmt)
            fails += int((gn != wn).sum() + (~gn & ~wn & (out != want)).sum())
    return fails


def test_unmutated_copy_passes_the_exact_pin(tmp_path):
    lib = _build(tmp_path, open(SRC).read())
    assert _exact_failures(lib) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_exact_pin_catches_mutant(tmp_path, name):
    """The exact-arithmetic pin (tests/test_oracle_exact.py) rejects every
    planted mistake too, at R = 3 and 5."""
    old, new = MUTANTS[name]
    lib = _build(tmp_path, open(SRC).read().replace(old, new, 1))
    assert _exact_failures(lib) > 0, f"the exact pin does not catch mutant {name}"
