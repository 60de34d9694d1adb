"""The fused epilogue's quotient method, checked on the CPU in exact
arithmetic.

The re-quantised output divides each bf16 value v by its group's scale s.
Instead of an IEEE division per value the kernel takes y = RN(1/s) once per
group and per value q = RN(v*y), then two remainder corrections
q <- RN(q + RN(v - s*q)*y) (each step one rounded fused multiply-add).  The
second correction is Markstein's (P. Markstein, IBM J. Res. Dev. 34(1), 1990;
J.-M. Muller et al., Handbook of Floating-Point Arithmetic, division with a
fused multiply-add): from a quotient within one ulp and a correctly rounded
reciprocal it yields the correctly rounded quotient.  This test restates the
five steps with exact rational arithmetic and a round-to-nearest-even fp32
rounding, and checks them against the exactly rounded quotient on random
values, on quotients next to fp32 rounding midpoints and on quotients next
to E4M3 rounding midpoints, for scales of the quantiser's form
max(amax, 1e-4)/448.  (The GPU tests check the kernel itself: its codes
equal those of the quantiser, which divides.)"""
import math
import random
import struct
from fractions import Fraction

F = Fraction


def rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest fp32 value, ties to even (normal and
    subnormal range; no overflow in this test)."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while F(2) ** e > x:
        e -= 1
    while F(2) ** (e + 1) <= x:
        e += 1
    ulp = F(2) ** (max(e, -126) - 23)
    m = x / ulp
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def bf16(x: float) -> Fraction:
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return F(struct.unpack("<f", struct.pack("<I", u))[0])


def corrected_quotient(v: Fraction, s: Fraction) -> Fraction:
    y = rn32(1 / s)
    q = rn32(v * y)
    for _ in range(2):
        r = rn32(v - s * q)
        q = rn32(q + r * y)
    return q


def scale_of(amax: Fraction) -> Fraction:
    return rn32(max(amax, rn32(F(1, 10000))) / 448)


def cases(n, seed):
    rng = random.Random(seed)
    e4m3_mids = [1 + (2 * k + 1) / 16 for k in range(8)]
    for i in range(n):
        amax = bf16(abs(rng.gauss(0, 1)) * 10 ** rng.uniform(-5, 4))
        s = scale_of(amax)
        kind = i % 3
        if kind == 0:
            v = bf16(rng.uniform(-1, 1) * float(amax))
        elif kind == 1:
            # v*1/s lands next to the midpoint between two fp32 values
            t = rn32(F(rng.uniform(-448, 448)))
            if t == 0:
                continue
            e = math.floor(math.log2(abs(t)))
            v = rn32((t + F(2) ** (e - 24) * (1 if t > 0 else -1)) * s)
        else:
            # next to a rounding midpoint of E4M3
            m = rng.choice(e4m3_mids) * 2.0 ** rng.randint(-6, 8)
            v = bf16(float(rn32(F(m) * s)) * (1 + rng.uniform(-1e-6, 1e-6)))
        yield v, s


def test_corrected_reciprocal_quotient_is_correctly_rounded():
    bad = [(v, s) for v, s in cases(6000, seed=3) if corrected_quotient(v, s) != rn32(v / s)]
    assert not bad, f"{len(bad)} quotients differ, first {bad[:3]}"


def test_one_correction_is_not_relied_on():
    """The first correction alone is only guaranteed within one ulp; the
    method keeps the second.  Sanity of the restatement: the uncorrected
    product is sometimes off, so the cases do exercise the corrections."""
    off = 0
    for v, s in cases(3000, seed=4):
        if rn32(v * rn32(1 / s)) != rn32(v / s):
            off += 1
    assert off > 0
