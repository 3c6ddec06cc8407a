"""The quantize pass of DynamicQuantizeLinear divides by the scale with one
reciprocal and a residual correction instead of an IEEE division per element:

    r = RN(1/b),  q = RN(x*r),  e = RN(x - q*b) (one FMA),  q' = RN(q + e*r) (one FMA)

(P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
processor", IBM J. Res. Dev. 34(1), 1990). The quantised byte is only correct
if q' is the correctly rounded quotient, because rint(q') decides it. This test
emulates the sequence in float64 (both FMAs are exact there up to their final
rounding, which is redone in float32) and compares it with numpy's IEEE
float32 division on random pairs and on pairs whose quotient sits next to a
float32 midpoint. It pins the method, not the kernel; the GPU tests compare the
kernel's bytes with the oracle, which divides with IEEE float32 division."""
from fractions import Fraction

import numpy as np

f32 = np.float32


def _round_f32_exact(value):
    """Round an exact rational to float32, ties to even."""
    c = f32(float(value))
    cands = [np.nextafter(c, f32(-np.inf)), c, np.nextafter(c, f32(np.inf))]
    return min(cands, key=lambda v: (abs(Fraction(float(v)) - value), int(np.array(v).view(np.int32)) & 1))


def corrected_quotient(x, b):
    r = (f32(1) / b).astype(f32)
    q = (x * r).astype(f32)
    # x - q*b: q*b has at most 48 significant bits, so the float64 difference is
    # exact whenever the residual is small, which is the case here
    e = (x.astype(np.float64) - q.astype(np.float64) * b.astype(np.float64)).astype(f32)
    s = e.astype(np.float64) * r.astype(np.float64) + q.astype(np.float64)
    out = s.astype(f32)
    # float64 -> float32 can double-round only when s lies on a float32 midpoint
    lo = out.astype(np.float64)
    nxt = np.nextafter(out, np.where(s > lo, f32(np.inf), f32(-np.inf))).astype(np.float64)
    mid = (lo + nxt) / 2
    for i in np.nonzero(np.abs(s - mid) <= np.abs(mid) * 2.0 ** -50)[0]:
        out[i] = _round_f32_exact(Fraction(float(e[i])) * Fraction(float(r[i])) + Fraction(float(q[i])))
    return out


def _assert_same(x, b, what):
    got = corrected_quotient(x, b)
    ref = (x / b).astype(f32)
    bad = np.nonzero(got.view(np.int32) != ref.view(np.int32))[0]
    assert bad.size == 0, f"{what}: {bad.size} quotients differ, first x={x[bad[0]]!r} b={b[bad[0]]!r}"


def test_random_pairs_match_ieee_division():
    rng = np.random.default_rng(11)
    n = 3_000_000
    b = rng.integers(0x3F800000, 0x40000000, n).astype(np.int32).view(f32)   # [1, 2)
    x = rng.integers(0x3F800000, 0x40800000, n).astype(np.int32).view(f32)   # [1, 4)
    _assert_same(x, b, "random")


def test_quotients_next_to_midpoints_match_ieee_division():
    rng = np.random.default_rng(12)
    n = 3_000_000
    b = rng.integers(0x3F800000, 0x40000000, n).astype(np.int32).view(f32)
    qv = rng.integers(0x3F000000, 0x40800000, n).astype(np.int32).view(f32)
    half_ulp = (np.nextafter(qv, f32(np.inf)).astype(np.float64) - qv.astype(np.float64)) / 2
    x = ((qv.astype(np.float64) + half_ulp) * b.astype(np.float64)).astype(f32)
    x = (x.view(np.int32) + rng.integers(-2, 3, n).astype(np.int32)).view(f32)
    _assert_same(x, b, "near midpoints")


def test_dql_shaped_scales_and_inputs():
    """Scales of the form (hi - lo)/255 and inputs across the whole range."""
    rng = np.random.default_rng(13)
    for _ in range(20):
        lo = -f32(rng.uniform(1e-3, 100))
        hi = f32(rng.uniform(1e-3, 100))
        scale = f32(f32(hi - lo) / f32(255))
        x = rng.uniform(lo, hi, 200_000).astype(f32)
        _assert_same(x, np.full_like(x, scale), "dql-shaped")
