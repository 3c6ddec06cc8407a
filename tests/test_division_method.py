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


R_MAX = f32(2.0 ** 100)        # the kernel's bound on r = RN(1/b) for the fast path
R_MIN = f32(2.0 ** -126)


def corrected_quotient(x, b, guard=True):
    """The kernel's quotient: Markstein's sequence where r is a normal float no
    larger than 2^100 (guard=False: wherever r is finite and normal), IEEE
    division elsewhere. float32 roundings, subnormals included, are numpy's."""
    with np.errstate(over="ignore", divide="ignore", invalid="ignore", under="ignore"):
        r = (f32(1) / b).astype(f32)
        fast = np.isfinite(r) & (np.abs(r) >= R_MIN)
        if guard:
            fast &= np.abs(r) <= R_MAX
        out = _markstein(x, b, np.where(fast, r, f32(1)))
        return np.where(fast, out, (x / b).astype(f32))


def _markstein(x, b, r):
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


def _mismatches(x, b, guard=True):
    got = corrected_quotient(x, b, guard)
    ref = (x / b).astype(f32)
    return np.count_nonzero(got.view(np.int32) != ref.view(np.int32))


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


def _near_midpoints(rng, n, b):
    """Inputs whose quotient by b lies within two ulps of a float32 midpoint in [1/4, 256)."""
    qv = rng.integers(0x3E800000, 0x43800000, n).astype(np.int32).view(f32)
    half_ulp = (np.nextafter(qv, f32(np.inf)).astype(np.float64) - qv.astype(np.float64)) / 2
    x = ((qv.astype(np.float64) + half_ulp) * b.astype(np.float64)).astype(f32)
    return (x.view(np.int32) + rng.integers(-2, 3, n).astype(np.int32)).view(f32)


def test_tiny_scales_need_the_bound_on_the_reciprocal():
    """Below scale = 2^-100 the residual x - q*b falls into float32's subnormal
    range and loses bits: without the bound some quotients next to midpoints
    come out one ulp off, with it (IEEE division there) none do."""
    rng = np.random.default_rng(14)
    n = 400_000
    e = rng.integers(-126, -104, n)
    b = np.ldexp(rng.uniform(1, 2, n), e).astype(f32)
    x = _near_midpoints(rng, n, b)
    assert _mismatches(x, b, guard=False) > 0
    assert _mismatches(x, b, guard=True) == 0


def test_scales_across_the_float_range_match_ieee_division():
    """Scales from subnormal (2^-149) up to 2^120, quotients next to midpoints."""
    rng = np.random.default_rng(15)
    n = 600_000
    e = rng.integers(-149, 121, n)
    b = np.ldexp(rng.uniform(1, 2, n), e).astype(f32)
    b = np.where(b == 0, f32(2.0 ** -149), b).astype(f32)
    x = _near_midpoints(rng, n, b)
    ok = np.isfinite(x) & (x != 0)
    assert _mismatches(x[ok], b[ok]) == 0
