"""A pin for the oracle at any R from exact rational arithmetic.

The oracle's result has a plain definition: binary32 additions in rank order,
each rounded to nearest with ties to even, then one rounding to binary16 or
bfloat16 ("[Kernel] Two-rank FP16 all-reduce through pinned host memory for
GPUs without P2P", section "Purpose": one final rounding; "[SM120] Add
optional FlashInfer PCIe-IPC all-reduce for switch-free hosts", section
"Accuracy": a fixed accumulation order).  This test evaluates that definition
with Python fractions: every input is decoded from its bit layout into an
exact rational, every addition is exact, and every rounding is done from the
IEEE 754 definition of round-to-nearest-even for a format of p significand
bits and exponent range [emin, emax] (overflow to infinity when the rounded
magnitude reaches 2^(emax+1)).  Nothing here uses numpy's or torch's float
arithmetic or casts, so it checks the oracle independently of the library
pins, at R = 3 .. 8 where no closed form exists.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

# (significand bits incl. the hidden one, emin, emax, exponent bits, fraction bits, bias)
FORMATS = {"f16": (11, -14, 15, 5, 10, 15), "bf16": (8, -126, 127, 8, 7, 127)}
BINARY32 = (24, -126, 127)
NAN = "nan"


def _pow2(k: int) -> Fraction:
    return Fraction(1 << k) if k >= 0 else Fraction(1, 1 << -k)


def decode(bits: int, fmt: str):
    """16-bit pattern -> NAN, ('inf', sign) or (exact value, sign)."""
    _, _, _, eb, fb, bias = FORMATS[fmt]
    s = bits >> 15
    e = (bits >> fb) & ((1 << eb) - 1)
    m = bits & ((1 << fb) - 1)
    if e == (1 << eb) - 1:
        return NAN if m else ("inf", s)
    if e == 0:
        mag = Fraction(m, 1 << fb) * _pow2(1 - bias)
    else:
        mag = (1 + Fraction(m, 1 << fb)) * _pow2(e - bias)
    return (-mag if s else mag), s


def round_rne(q: Fraction, p: int, emin: int, emax: int):
    """q rounded to nearest-even in a format of p bits, exponents emin..emax:
    a Fraction, or ('inf', sign) on overflow.  q != 0."""
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if _pow2(e) > a:
        e -= 1
    if _pow2(e + 1) <= a:
        e += 1
    ulp = _pow2(max(e, emin) - p + 1)
    k = a / ulp
    n = k.numerator // k.denominator
    r = k - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * ulp
    if v >= _pow2(emax + 1):
        return ("inf", 1 if q < 0 else 0)
    return -v if q < 0 else v


def add32(x, y):
    """IEEE binary32 addition, round to nearest even, of two decoded values."""
    if x == NAN or y == NAN:
        return NAN
    if isinstance(x[0], str) or isinstance(y[0], str):
        infs = [v[1] for v in (x, y) if isinstance(v[0], str)]
        return NAN if len(set(infs)) > 1 else ("inf", infs[0])
    exact = x[0] + y[0]
    if exact == 0:
        return Fraction(0), 1 if (x[1] == 1 and y[1] == 1) else 0
    r = round_rne(exact, *BINARY32)
    if isinstance(r, tuple):
        return r
    return r, 1 if r < 0 else 0


def encode(v, fmt: str) -> int:
    """A decoded value rounded to the 16-bit format -> its bit pattern."""
    p, emin, emax, eb, fb, bias = FORMATS[fmt]
    if v == NAN:
        return ((1 << eb) - 1) << fb | (1 << (fb - 1))
    if isinstance(v[0], str):
        return v[1] << 15 | ((1 << eb) - 1) << fb
    q, s = v
    if q != 0:
        q = round_rne(q, p, emin, emax)
        if isinstance(q, tuple):
            return q[1] << 15 | ((1 << eb) - 1) << fb
        s = 1 if q < 0 else s if q == 0 else 0
    if q == 0:
        return s << 15
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if _pow2(e) > a:
        e -= 1
    if e < emin:        # subnormal: a multiple of 2^(emin - p + 1)
        m = a / _pow2(emin - p + 1)
        assert m.denominator == 1
        return s << 15 | int(m)
    m = (a / _pow2(e) - 1) * (1 << fb)
    assert m.denominator == 1
    return s << 15 | (e + bias) << fb | int(m)


def exact_rank_order(xs, fmt: str):
    """The definition, element by element: binary32 adds in rank order from
    f32(x_0), one rounding to the format."""
    n = len(xs[0])
    out = np.empty(n, np.uint16)
    for i in range(n):
        acc = decode(int(xs[0][i]), fmt)
        for p in range(1, len(xs)):
            acc = add32(acc, decode(int(xs[p][i]), fmt))
        out[i] = encode(acc, fmt)
    return out


def _is_nan(bits, fmt):
    if fmt == "f16":
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def test_the_rounding_is_the_definition_on_known_values():
    """round_rne and encode against values fixed by the formats themselves."""
    assert encode((Fraction(1), 0), "f16") == 0x3C00
    assert encode((Fraction(65504), 0), "f16") == 0x7BFF
    assert encode((Fraction(65520), 0), "f16") == 0x7C00          # max + half ulp ties to even: inf
    assert encode((Fraction(65519), 0), "f16") == 0x7BFF
    assert encode((_pow2(-24), 0), "f16") == 0x0001               # smallest subnormal
    assert encode((_pow2(-25), 0), "f16") == 0x0000               # half of it ties to even zero
    assert encode((_pow2(-25) * 3 / 2, 0), "f16") == 0x0001
    assert encode((-_pow2(-26), 1), "f16") == 0x8000              # underflow keeps the sign
    assert encode((1 + _pow2(-11), 0), "f16") == 0x3C00           # tie to even (down)
    assert encode((1 + 3 * _pow2(-11), 0), "f16") == 0x3C02       # tie to even (up)
    assert encode((Fraction(1), 0), "bf16") == 0x3F80
    assert encode((1 + _pow2(-8), 0), "bf16") == 0x3F80
    assert encode((1 + 3 * _pow2(-8), 0), "bf16") == 0x3F82
    assert encode((_pow2(-133), 0), "bf16") == 0x0001
    assert round_rne(Fraction(1) + _pow2(-24), *BINARY32) == 1
    assert round_rne(Fraction(1) + 3 * _pow2(-24), *BINARY32) == 1 + _pow2(-22)
    assert round_rne(_pow2(128), *BINARY32) == ("inf", 0)
    for bits in (0x0000, 0x8000, 0x3555, 0xBC01, 0x03FF, 0x7BFF, 0xFC00):
        assert encode(decode(bits, "f16"), "f16") == bits
    for bits in (0x0000, 0x8000, 0x3F81, 0x0001, 0x7F7F, 0xFF80):
        assert encode(decode(bits, "bf16"), "bf16") == bits


def _inputs(rng, R, n, fmt):
    special = {"f16": [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00,
                       0x3C00, 0xBC00, 0x3C01, 0x7E00],
               "bf16": [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80,
                        0x3F80, 0xBF80, 0x3F81, 0x7FC0]}[fmt]
    # a cancellation block: rank 0 a large b, rank 1 a small s that the
    # binary32 sum b + s drops, rank 2 exactly -b (the order and the
    # precision of the running sum decide the result)
    big = rng.integers(0x6000, 0x7800 if fmt == "f16" else 0x7000, n // 4).astype(np.uint16)
    xs = []
    for r in range(R):
        kind = rng.integers(0, 4, n)
        near = (0x3C00 if fmt == "f16" else 0x3F80) + rng.integers(-600, 600, n)
        rnd = rng.integers(0, 65536, n)
        sp = np.array(special)[rng.integers(0, len(special), n)]
        # mostly values near 1 (rounding ties and carries), some random
        # patterns (every scale), a few specials
        x = np.where(kind < 2, near, np.where(kind == 2, rnd, np.where(rng.random(n) < 0.3, sp, near)))
        x = x.astype(np.uint16)
        small = (rng.integers(0, 2, n // 4).astype(np.uint16) << 15) | rng.integers(
            0x0400 if fmt == "f16" else 0x2000, 0x1C00 if fmt == "f16" else 0x3000, n // 4).astype(np.uint16)
        x[: n // 4] = big if r == 0 else (big ^ np.uint16(0x8000)) if r == 2 else small
        xs.append(x)
    return xs


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("R", [3, 5, 8])
def test_oracle_equals_the_exact_definition(fmt, R):
    rng = np.random.default_rng(1000 * R + (fmt == "bf16"))
    xs = _inputs(rng, R, 1500, fmt)
    want = exact_rank_order(xs, fmt)
    got = oracle.allreduce(xs, fmt)
    for r in range(R):
        g = np.asarray(got[r], np.uint16)
        gn, wn = _is_nan(g, fmt), _is_nan(want, fmt)
        assert np.array_equal(gn, wn), f"R={R} rank {r}: NaN-ness differs at {np.flatnonzero(gn != wn)[:5]}"
        bad = ~gn & (g != want)
        assert not bad.any(), (f"R={R} rank {r}: {int(bad.sum())} differ, first at {np.flatnonzero(bad)[:5]}: "
                               f"got {[hex(v) for v in g[bad][:5]]} want {[hex(v) for v in want[bad][:5]]}")
