"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each test compares the oracle with one of: a value the pages print (fixtures in
tests/golden/, each carrying its citation), a closed form, an algebraic identity
the pages state, or brute force in exact Python integers / rationals with float32
rounding done by ``struct`` (independent of numpy's float32 arithmetic). They are
chosen so that a dropped term, a wrong sign or index, or a transposed operand in
the oracle fails at least one of them.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import qmm_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --- independent float helpers (no numpy float32 arithmetic) ---------------

def f32(x: float) -> float:
    """Round a Python float (double) to the nearest float32, ties to even."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f32_from_bits(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def bf16_round_value(v: float) -> float:
    """Nearest bf16 value (8 significant bits), ties to even, via frexp + round()."""
    if v == 0.0:
        return 0.0
    m, e = math.frexp(v)          # v = m * 2**e with 0.5 <= |m| < 1
    r = round(m * 256)            # Python's round() breaks ties to even
    return math.ldexp(r, e - 8)


def bf16_bits_value(bits: int) -> float:
    return f32_from_bits(int(bits) << 16)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_wrap_int32_closed_form():
    vals = np.array([0, 2**31 - 1, 2**31, -2**31, -2**31 - 1, 2**32 + 5, 65025 * 34816], np.int64)
    got = O.wrap_int32(vals)
    want = [0, 2**31 - 1, -2**31, -2**31, 2**31 - 1, 5, 65025 * 34816 - 2**32]
    assert got.tolist() == want


def test_bf16_rounding_specials():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2**-8: 0x3F80,               # tie, kept part even -> stays
        one + 3 * 2**-8: 0x3F82,           # tie, kept part odd -> rounds up
        one + 2**-8 + 2**-20: 0x3F81,      # just above the tie
        -(one + 2**-8): 0xBF80,
        255.0: 0x437F,
        257.0: 0x4380,                     # 256 + 1: tie at ulp 2 -> even (256)
        259.0: 0x4382,                     # tie -> even (260)
    }
    x = np.array(list(cases.keys()), np.float32)
    got = O.f32_to_bf16_bits(x)
    assert [int(g) for g in got] == list(cases.values())


def test_bf16_rounding_bruteforce():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    got = O.f32_to_bf16_bits(x)
    for xi, gi in zip(x.tolist(), got.tolist()):
        assert bf16_bits_value(gi) == bf16_round_value(xi)


# ---------------------------------------------------------------------------
# form (a): factored int8-weight dequant matmul
# ---------------------------------------------------------------------------

def _w8_case(seed, M, K, N, per_column):
    rng = np.random.default_rng(seed)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.integers(-128, 128, (K, N), dtype=np.int8)
    if per_column:
        scale = rng.uniform(0.001, 0.05, N).astype(np.float32)
        zp = rng.integers(-20, 20, N).astype(np.int32)
    else:
        scale = np.array([0.02], np.float32)
        zp = np.array([3], np.int32)
    return A, B, scale, zp


@pytest.mark.parametrize("per_column", [False, True])
def test_w8_bruteforce_unfactored_rationals(per_column):
    """Exact rational sum of a_k * (b_k - zp) * scale, the unfactored dequantisation."""
    A, B, scale, zp = _w8_case(2, 3, 9, 4, per_column)
    got = O.w8_dequant(A, B, scale, zp)
    M, K = A.shape
    N = B.shape[1]
    for m in range(M):
        for n in range(N):
            s = Fraction(float(scale[n if per_column else 0]))
            z = int(zp[n if per_column else 0])
            exact = sum(Fraction(float(A[m, k])) * (int(B[k, n]) - z) * s for k in range(K))
            assert abs(got[m, n] - float(exact)) <= 1e-12 * (1 + abs(float(exact)))


@pytest.mark.parametrize("per_column", [False, True])
def test_w8_factoring_identity_vs_explicit_dequant(per_column):
    """The factored form equals dequantise-then-matmul (the identity the kernel rests on)."""
    A, B, scale, zp = _w8_case(3, 17, 130, 23, per_column)
    fused = O.w8_dequant(A, B, scale, zp)
    explicit = O.w8_dequant_explicit(A, B, scale, zp)
    mag = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64) + 1.0
    assert np.all(np.abs(fused - explicit) <= 1e-12 * mag)


def test_w8_zero_point_zero_is_plain_matmul():
    A, B, _, _ = _w8_case(4, 5, 33, 6, False)
    got = O.w8_dequant(A, B, [0.5], [0])
    M, K = A.shape
    for m in range(M):
        for n in range(B.shape[1]):
            exact = sum(Fraction(float(A[m, k])) * int(B[k, n]) for k in range(K)) * Fraction(1, 2)
            assert abs(got[m, n] - float(exact)) <= 1e-12 * (1 + abs(float(exact)))


def test_w8_error_bound_shape_and_value():
    A = np.array([[1.0, -2.0]], np.float32)
    B = np.array([[3], [-4]], np.int8)
    bound = O.w8_dequant_error_bound(A, B, [0.5], [1])
    # |1|*|0.5*(3-1)| + |-2|*|0.5*(-4-1)| = 1 + 5 = 6
    assert bound.shape == (1, 1)
    assert abs(bound[0, 0] - (1e-3 * 6 + 1e-6)) < 1e-15


# ---------------------------------------------------------------------------
# form (b): A8W8
# ---------------------------------------------------------------------------

def test_a8w8_bruteforce_python_ints_and_struct_f32():
    rng = np.random.default_rng(5)
    M, K, N = 4, 37, 5
    A = rng.integers(-127, 128, (M, K), dtype=np.int8)
    B = rng.integers(-127, 128, (K, N), dtype=np.int8)
    a_s = rng.uniform(0.005, 0.02, M).astype(np.float32)
    w_s = rng.uniform(0.001, 0.01, N).astype(np.float32)
    got32 = O.a8w8(A, B, a_s, w_s, "f32")
    got16 = O.a8w8(A, B, a_s, w_s, "bf16")
    for m in range(M):
        for n in range(N):
            acc = sum(int(A[m, k]) * int(B[k, n]) for k in range(K))
            f = f32(float(acc))
            f = f32(f * float(a_s[m]))
            f = f32(f * float(w_s[n]))
            assert float(got32[m, n]) == f
            assert bf16_bits_value(got16[m, n]) == bf16_round_value(f)


def test_a8w8_scale_orientation_golden():
    g = golden("a8w8_scale_orientation.json")
    M, N = g["M"], g["N"]
    A = np.eye(M, dtype=np.int8)
    B = np.ones((M, N), np.int8)
    got = O.a8w8(A, B, np.array(g["act_scale"], np.float32), np.array(g["weight_scale"], np.float32))
    assert got.tolist() == g["expected_f32"]


def test_a8w8_scalar_scales_broadcast():
    A = np.array([[1, 2], [3, 4]], np.int8)
    B = np.array([[1, 0], [0, 1]], np.int8)
    got = O.a8w8(A, B, [0.5], [2.0])
    assert got.tolist() == [[1.0, 2.0], [3.0, 4.0]]


def test_a8w8_acc_wraps():
    K = 131073                      # 16384 * K > 2^31
    A = np.full((1, K), -128, np.int8)
    B = np.full((K, 1), -128, np.int8)
    assert int(O.a8w8_acc(A, B)[0, 0]) == 16384 * K - 2**32


def _exact_scaled(acc: int, a: float, w: float) -> Fraction:
    return Fraction(acc) * Fraction(a) * Fraction(w)


@pytest.mark.parametrize("shape", [(3, 29, 5), (4, 16, 4)])
def test_a8w8_exact_against_rationals(shape):
    """a8w8_exact is the real value acc * act_scale[m] * weight_scale[n]: each
    element within 2 ulps (two float64 roundings) of the exact rational, with
    row-only and column-only scales so that swapping the two orientations, even
    when M == N, moves every element by far more."""
    M, K, N = shape
    rng = np.random.default_rng(21)
    A = rng.integers(-127, 128, (M, K), dtype=np.int8)
    B = rng.integers(-127, 128, (K, N), dtype=np.int8)
    a_s = (np.arange(1, M + 1) * 0.25).astype(np.float32)            # rows: 0.25, 0.5, ...
    w_s = (np.arange(1, N + 1) * 0.001 + 0.003).astype(np.float32)    # columns, a different law
    got = O.a8w8_exact(A, B, a_s, w_s)
    assert got.dtype == np.float64 and got.shape == (M, N)
    for m in range(M):
        for n in range(N):
            acc = sum(int(A[m, k]) * int(B[k, n]) for k in range(K))
            want = _exact_scaled(acc, float(a_s[m]), float(w_s[n]))
            err = abs(Fraction(float(got[m, n])) - want)
            assert err <= 2 * Fraction(math.ulp(float(want))), (m, n)
    if M == N:   # the square case: a last-dimension broadcast would give this instead
        assert not np.allclose(O.a8w8_exact(A, B, w_s, a_s), got)


def test_a8w8_exact_scalar_scales_and_wrapped_accumulator():
    """Scalar scales broadcast; the accumulator is the wrapped int32 one (the
    value the float32 chain starts from), here past 2^31."""
    K = 133200                       # 127 * 127 * K > 2^31
    A = np.full((1, K), 127, np.int8)
    B = np.full((K, 2), 127, np.int8)
    got = O.a8w8_exact(A, B, [0.5], [0.25])
    wrapped = 16129 * K - 2**32
    assert wrapped < 0
    assert got.tolist() == [[wrapped * 0.125, wrapped * 0.125]]


def test_a8w8_error_bound_value():
    A = np.array([[2, -3]], np.int8)
    B = np.array([[5], [7]], np.int8)
    b = O.a8w8_error_bound(A, B, [0.5], [0.25])
    assert abs(b[0, 0] - (1e-3 * (10 + 21) * 0.125 + 1e-6)) < 1e-15


# ---------------------------------------------------------------------------
# form (c): MatMulInteger
# ---------------------------------------------------------------------------

def test_matmul_integer_page_value_len259():
    g = golden("matmul_integer_u8_len259.json")
    K = g["K"]
    A = np.full((1, K), g["a_value"], np.uint8)
    B = np.full((K, 1), g["b_value"], np.uint8)
    got = O.matmul_integer(A, B, g["a_zero_point"], g["b_zero_point"])
    assert int(got[0, 0]) == g["expected"]


def test_f32_accumulation_threshold_of_the_page():
    """65025*K fits the 24-bit significand only up to K=258, so float32 cannot hold the 259 sum."""
    assert 65025 * 258 < 2**24 <= 65025 * 259
    acc = np.float32(0)
    for _ in range(259):
        acc = np.float32(acc + np.float32(65025))
    assert int(acc) != 16841475


def test_matmul_integer_max_magnitude_product():
    K = 3
    A = np.full((1, K), 255, np.uint8)
    B = np.full((K, 1), -128, np.int8)
    assert int(O.matmul_integer(A, B, 0, 127)[0, 0]) == -65025 * K


def test_matmul_integer_wrap_k34816():
    K = 34816
    A = np.full((1, K), 255, np.uint8)
    B = np.full((K, 2), 255, np.uint8)
    got = O.matmul_integer(A, B)
    assert got.tolist() == [[65025 * K - 2**32] * 2]


@pytest.mark.parametrize("adt,bdt", [(np.uint8, np.int8), (np.int8, np.int8), (np.uint8, np.uint8), (np.int8, np.uint8)])
def test_matmul_integer_bruteforce(adt, bdt):
    rng = np.random.default_rng(6)
    M, K, N = 3, 11, 4
    info_a, info_b = np.iinfo(adt), np.iinfo(bdt)
    A = rng.integers(info_a.min, info_a.max + 1, (M, K)).astype(adt)
    B = rng.integers(info_b.min, info_b.max + 1, (K, N)).astype(bdt)
    a_zp = rng.integers(info_a.min, info_a.max + 1, M).astype(adt)      # per row
    b_zp = rng.integers(info_b.min, info_b.max + 1, N).astype(bdt)      # per column
    got = O.matmul_integer(A, B, a_zp, b_zp)
    for m in range(M):
        for n in range(N):
            s = sum((int(A[m, k]) - int(a_zp[m])) * (int(B[k, n]) - int(b_zp[n])) for k in range(K))
            assert int(got[m, n]) == s


def test_matmul_integer_direct_equals_expanded_mod_2_32():
    """sum (a-za)(b-zb) == sum ab - za*colsum(B) - zb*rowsum(A) + K*za*zb (mod 2^32)."""
    rng = np.random.default_rng(7)
    M, K, N = 6, 300, 9
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    za = 131
    zb = rng.integers(-128, 128, N).astype(np.int8)
    got = O.matmul_integer(A, B, za, zb)
    for m in range(M):
        for n in range(N):
            ab = sum(int(A[m, k]) * int(B[k, n]) for k in range(K))
            rs = sum(int(A[m, k]) for k in range(K))
            cs = sum(int(B[k, n]) for k in range(K))
            e = ab - za * cs - int(zb[n]) * rs + K * za * int(zb[n])
            e = (e + 2**31) % 2**32 - 2**31
            assert int(got[m, n]) == e


def test_matmul_integer_shared_b_equals_per_batch_copies():
    rng = np.random.default_rng(8)
    A = rng.integers(-128, 128, (2, 3, 4, 40)).astype(np.int8)
    B = rng.integers(-128, 128, (40, 5)).astype(np.int8)
    shared = O.matmul_integer(A, B, -5, 7)
    copied = O.matmul_integer(A, np.broadcast_to(B, (2, 3, 40, 5)).copy(), -5, 7)
    assert shared.shape == (2, 3, 4, 5)
    assert np.array_equal(shared, copied)
    # and each batch equals its own rank-2 product
    for i in range(2):
        for j in range(3):
            assert np.array_equal(shared[i, j], O.matmul_integer(A[i, j], B, -5, 7))


def test_matmul_integer_zero_points_zero_is_a8w8_acc():
    rng = np.random.default_rng(9)
    A = rng.integers(-127, 128, (5, 70)).astype(np.int8)
    B = rng.integers(-127, 128, (70, 6)).astype(np.int8)
    assert np.array_equal(O.matmul_integer(A, B, 0, 0), O.a8w8_acc(A, B))
    for m in range(5):
        for n in range(6):
            assert int(O.a8w8_acc(A, B)[m, n]) == sum(int(A[m, k]) * int(B[k, n]) for k in range(70))


# ---------------------------------------------------------------------------
# form (d): DynamicQuantizeLinear
# ---------------------------------------------------------------------------

def test_dql_all_zero_golden():
    g = golden("dql_all_zero.json")
    y, s, zp = O.dynamic_quantize_linear(np.array(g["x"], np.float32))
    assert float(s) == g["scale"] and int(zp) == g["zero_point"]
    assert y.tolist() == g["y"]


def test_dql_empty_input():
    y, s, zp = O.dynamic_quantize_linear(np.zeros(0, np.float32))
    assert float(s) == 1.0 and int(zp) == 0 and y.size == 0


def test_dql_hand_worked_golden():
    g = golden("dql_hand_worked.json")
    y, s, zp = O.dynamic_quantize_linear(np.array(g["x"], np.float32))
    assert int(np.float32(s).view(np.uint32)) == g["scale_f32_bits"]
    assert int(zp) == g["zero_point"]
    assert y.tolist() == g["y"]


def test_dql_ties_to_even_golden():
    g = golden("dql_ties.json")
    y, s, zp = O.dynamic_quantize_linear(np.array(g["x"], np.float32))
    assert float(s) == g["scale"] and int(zp) == g["zero_point"]
    assert y.tolist() == g["y"]


def test_dql_one_sided_golden():
    for c in golden("dql_one_sided.json")["cases"]:
        y, _, zp = O.dynamic_quantize_linear(np.array(c["x"], np.float32))
        assert int(zp) == c["zero_point"]
        assert y.tolist() == c["y"]


def test_quantize_linear_saturates():
    y = O.quantize_linear(np.array([1000.0, -1000.0, 3.0, 10.0], np.float32), np.float32(1.0), 0)
    assert y.tolist() == [255, 0, 3, 10]
    y = O.quantize_linear(np.array([10.0, -300.0], np.float32), np.float32(1.0), 250)
    assert y.tolist() == [255, 0]


def test_dql_bruteforce_struct_f32():
    rng = np.random.default_rng(10)
    for trial in range(20):
        n = int(rng.integers(1, 300))
        x = rng.standard_normal(n).astype(np.float32)
        x[rng.random(n) < 0.05] *= np.float32(20)
        if trial % 5 == 1:
            x = np.abs(x)
        if trial % 5 == 2:
            x = -np.abs(x)
        y, s, zp = O.dynamic_quantize_linear(x)
        xs = [float(v) for v in x]
        lo = min(0.0, min(xs))
        hi = max(0.0, max(xs))
        r = f32(hi - lo)
        scale = 1.0 if r == 0.0 else f32(r / 255.0)
        z = min(255, max(0, round(f32(-lo / scale))))
        assert float(s) == scale and int(zp) == z
        want = [min(255, max(0, round(f32(v / scale)) + z)) for v in xs]
        assert y.tolist() == want


def test_row_and_col_sums_bruteforce():
    rng = np.random.default_rng(11)
    y = rng.integers(0, 256, 4 * 13).astype(np.uint8)
    rs = O.row_sums(y, 13)
    assert rs.tolist() == [sum(int(v) for v in y[i * 13:(i + 1) * 13]) for i in range(4)]
    B = rng.integers(-128, 128, (9, 5)).astype(np.int8)
    cs = O.col_sums(B)
    assert cs.tolist() == [sum(int(B[k, n]) for k in range(9)) for n in range(5)]


# ---------------------------------------------------------------------------
# The accumulating A8W8 variant
# ---------------------------------------------------------------------------

def test_a8w8_dequant_acc_with_zero_accumulator_is_a8w8():
    rng = np.random.default_rng(41)
    A = rng.integers(-128, 128, (7, 33)).astype(np.int8)
    B = rng.integers(-128, 128, (33, 5)).astype(np.int8)
    a_s = rng.uniform(0.01, 0.02, 7).astype(np.float32)
    w_s = rng.uniform(0.001, 0.01, 5).astype(np.float32)
    for out in ("f32", "bf16"):
        assert np.array_equal(O.a8w8_dequant_acc(np.zeros((7, 5), np.int32), A, B, a_s, w_s, out),
                              O.a8w8(A, B, a_s, w_s, out))


def test_a8w8_dequant_acc_chains_a_split_of_k():
    """Linearity of the sum over K: the product of the first K columns/rows,
    handed over as the accumulator of the second, gives the whole product."""
    rng = np.random.default_rng(42)
    A = rng.integers(-128, 128, (6, 40)).astype(np.int8)
    B = rng.integers(-128, 128, (40, 9)).astype(np.int8)
    a_s = rng.uniform(0.01, 0.02, 6).astype(np.float32)
    w_s = rng.uniform(0.001, 0.01, 9).astype(np.float32)
    for k1 in (1, 16, 39):
        first = O.a8w8_acc(A[:, :k1], B[:k1])
        got = O.a8w8_dequant_acc(first, A[:, k1:], B[k1:], a_s, w_s, "f32")
        assert np.array_equal(got, O.a8w8(A, B, a_s, w_s, "f32")), k1


def test_a8w8_dequant_acc_brute_force_with_wrap():
    """Python-int brute force, struct-rounded float32 steps; accumulators near
    the int32 limits so the sum wraps."""
    rng = np.random.default_rng(43)
    M, K, N = 3, 4, 2
    A = rng.integers(-128, 128, (M, K)).astype(np.int8)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    acc = np.array([[2**31 - 5, -2**31 + 3], [7, -9], [2**31 - 1, -2**31]], np.int32)
    a_s = np.array([0.5, 0.25, 3.0], np.float32)
    w_s = np.array([0.125, 2.0], np.float32)
    got = O.a8w8_dequant_acc(acc, A, B, a_s, w_s, "f32")

    def f32(x):
        return struct.unpack("f", struct.pack("f", x))[0]

    for m in range(M):
        for n in range(N):
            s = int(acc[m, n]) + sum(int(A[m, k]) * int(B[k, n]) for k in range(K))
            s = (s + 2**31) % 2**32 - 2**31
            v = f32(f32(f32(float(s)) * float(a_s[m])) * float(w_s[n]))
            assert got[m, n] == np.float32(v), (m, n)


# ---------------------------------------------------------------------------
# ConvInteger
# ---------------------------------------------------------------------------

def _conv_brute(x, w, xzp, wzp, pads, strides, dils, group):
    """Exact Python integers, one output at a time, straight from the definition."""
    N, C, H, Wd = x.shape
    M, Cg, kH, kW = w.shape
    pt, pl, pb, pr = pads
    oH = (H + pt + pb - dils[0] * (kH - 1) - 1) // strides[0] + 1
    oW = (Wd + pl + pr - dils[1] * (kW - 1) - 1) // strides[1] + 1
    Mg = M // group
    wz = list(wzp) if len(wzp) == M else [wzp[0]] * M
    out = np.zeros((N, M, oH, oW), dtype=np.int64)
    for n in range(N):
        for m in range(M):
            g = m // Mg
            for oh in range(oH):
                for ow in range(oW):
                    s = 0
                    for c in range(Cg):
                        for kh in range(kH):
                            for kw in range(kW):
                                ih = oh * strides[0] + kh * dils[0] - pt
                                iw = ow * strides[1] + kw * dils[1] - pl
                                if 0 <= ih < H and 0 <= iw < Wd:
                                    xv = int(x[n, g * Cg + c, ih, iw]) - int(xzp)
                                else:
                                    xv = 0
                                s += xv * (int(w[m, c, kh, kw]) - int(wz[m]))
                    out[n, m, oh, ow] = (s + 2**31) % 2**32 - 2**31
    return out


@pytest.mark.parametrize("xdt,wdt", [(np.uint8, np.int8), (np.int8, np.int8), (np.uint8, np.uint8)])
def test_conv_integer_brute_force(xdt, wdt):
    rng = np.random.default_rng(51)
    info = {np.uint8: (0, 256), np.int8: (-128, 128)}
    x = rng.integers(*info[xdt], size=(2, 4, 6, 7)).astype(xdt)
    w = rng.integers(*info[wdt], size=(6, 2, 3, 2)).astype(wdt)
    xzp = np.array([rng.integers(*info[xdt])], xdt)
    wzp = rng.integers(*info[wdt], size=6).astype(wdt)
    for pads, strides, dils, group in [([1, 0, 2, 1], [2, 1], [1, 2], 2), ([0, 0, 0, 0], [1, 1], [1, 1], 1)]:
        wg = w if group == 2 else rng.integers(*info[wdt], size=(6, 4, 3, 2)).astype(wdt)
        got = O.conv_integer(x, wg, xzp, wzp, pads, strides, dils, group)
        assert np.array_equal(got, _conv_brute(x, wg, xzp[0], wzp, pads, strides, dils, group)), (pads, group)


def test_conv_integer_single_channel_is_scipy_correlate():
    """One input and one output channel: the zero-point-shifted input, zero
    padded, correlated with the shifted kernel (scipy), then subsampled by
    the stride; a dilation spreads the kernel taps apart with zeros."""
    scipy_signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(52)
    x = rng.integers(0, 256, size=(1, 1, 11, 9)).astype(np.uint8)
    w = rng.integers(-128, 128, size=(1, 1, 3, 4)).astype(np.int8)
    xzp, wzp = 131, -7
    for pads, strides, dils in [([0, 0, 0, 0], [1, 1], [1, 1]), ([2, 1, 1, 3], [2, 3], [1, 1]),
                                ([1, 2, 2, 1], [1, 2], [2, 3])]:
        xs = np.pad(x[0, 0].astype(np.int64) - xzp, ((pads[0], pads[2]), (pads[1], pads[3])))
        ks = w[0, 0].astype(np.int64) - wzp
        kd = np.zeros(((ks.shape[0] - 1) * dils[0] + 1, (ks.shape[1] - 1) * dils[1] + 1), np.int64)
        kd[::dils[0], ::dils[1]] = ks
        full = scipy_signal.correlate2d(xs, kd, mode="valid")
        want = full[::strides[0], ::strides[1]]
        got = O.conv_integer(x, w, xzp, wzp, pads, strides, dils)
        assert np.array_equal(got[0, 0], want), (pads, strides, dils)


def test_conv_integer_rank3_is_a_sum_of_1d_correlations():
    scipy_signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(53)
    x = rng.integers(-128, 128, size=(2, 3, 20)).astype(np.int8)
    w = rng.integers(-128, 128, size=(4, 3, 5)).astype(np.int8)
    wzp = rng.integers(-128, 128, size=4).astype(np.int8)
    got = O.conv_integer(x, w, -3, wzp, pads=[2, 1], strides=[2], dilations=[1])
    for n in range(2):
        for m in range(4):
            acc = sum(scipy_signal.correlate(np.pad(x[n, c].astype(np.int64) + 3, (2, 1)),
                                             w[m, c].astype(np.int64) - int(wzp[m]), mode="valid")
                      for c in range(3))
            assert np.array_equal(got[n, m], acc[::2]), (n, m)


def test_conv_integer_1x1_is_a_matmul_per_image():
    rng = np.random.default_rng(54)
    x = rng.integers(0, 256, size=(3, 17, 5, 6)).astype(np.uint8)
    w = rng.integers(-128, 128, size=(9, 17, 1, 1)).astype(np.int8)
    wzp = rng.integers(-128, 128, size=9).astype(np.int8)
    got = O.conv_integer(x, w, 100, wzp)
    Wm = w[:, :, 0, 0].astype(np.int64) - wzp[:, None].astype(np.int64)
    for n in range(3):
        want = Wm @ (x[n].reshape(17, 30).astype(np.int64) - 100)
        assert np.array_equal(got[n].reshape(9, 30), want)


def test_conv_integer_output_extent_and_wrap():
    """Closed form: every tap 255 * 127 over C*kH*kW taps, past the int32 range."""
    C = 8000
    x = np.full((1, C, 3, 3), 255, np.uint8)
    w = np.full((2, C, 3, 3), 127, np.int8)
    got = O.conv_integer(x, w)
    assert got.shape == (1, 2, 1, 1)
    total = 255 * 127 * C * 9
    assert total > 2**31
    assert (got == (total + 2**31) % 2**32 - 2**31).all()
    assert O.conv_output_size(56, 3, 1, 1, 1, 1) == 56 and O.conv_output_size(56, 3, 1, 1, 2, 1) == 28
    assert O.conv_output_size(10, 3, 0, 0, 1, 4) == 2


# ---------------------------------------------------------------------------
# DynamicQuantizeLinear -> MatMulInteger -> dequantise
# ---------------------------------------------------------------------------

def test_dynamic_quantize_matmul_within_the_quantisation_bound():
    """Against float64 x @ ((W - w_zp) * w_scale): quantising x moves each
    element by at most y_scale / 2 (the range covers all of x, so nothing
    saturates), so |C - exact| <= y_scale/2 * sum_k |W_deq[k, n]| plus the
    fp32 rounding of the last steps."""
    rng = np.random.default_rng(61)
    M, K, N = 9, 70, 13
    x = (rng.standard_normal((M, K)) * 2.0).astype(np.float32)
    W = rng.integers(-128, 128, size=(K, N)).astype(np.int8)
    w_scale = rng.uniform(0.001, 0.01, N).astype(np.float32)
    w_zp = rng.integers(-20, 20, size=N).astype(np.int8)
    bias = rng.standard_normal(N).astype(np.float32)
    C, ys, _ = O.dynamic_quantize_matmul(x, W, w_scale, w_zp, bias)
    Wd = (W.astype(np.float64) - w_zp.astype(np.float64)) * w_scale.astype(np.float64)
    exact = x.astype(np.float64) @ Wd + bias.astype(np.float64)
    bound = float(ys) / 2 * np.abs(Wd).sum(axis=0)[None, :] + 4 * 2.0**-23 * (np.abs(exact) + 1)
    assert (np.abs(C.astype(np.float64) - exact) <= bound).all()
    # the bound is tight enough to catch an activation zero point off by one:
    # on a column whose dequantised weights are all positive that error is
    # y_scale * sum_k W_deq[k, n], twice the bound's main term
    y, _, yzp = O.dynamic_quantize_linear(x)
    Wp = np.abs(Wd[:, :1]) + 1e-3
    off = (float(ys) * (y.astype(np.float64) - (float(yzp) + 1))) @ Wp
    bound_p = float(ys) / 2 * Wp.sum() + 4 * 2.0**-23 * (np.abs(x.astype(np.float64) @ Wp) + 1)
    assert (np.abs(off - x.astype(np.float64) @ Wp) > bound_p).all()


def test_dynamic_quantize_matmul_uint8_weight_and_no_bias():
    rng = np.random.default_rng(62)
    x = rng.uniform(-3, 5, (6, 40)).astype(np.float32)
    W = rng.integers(0, 256, size=(40, 7)).astype(np.uint8)
    C, ys, yzp = O.dynamic_quantize_matmul(x, W, np.float32(0.004), np.uint8(128))
    Wd = (W.astype(np.float64) - 128) * 0.004
    err = np.abs(C.astype(np.float64) - x.astype(np.float64) @ Wd)
    assert (err <= float(ys) / 2 * np.abs(Wd).sum(axis=0)[None, :] + 1e-5).all()
    # integer core: brute force in Python integers from the pinned quantiser's outputs
    y, _, _ = O.dynamic_quantize_linear(x)
    for m in range(6):
        for n in range(7):
            acc = sum((int(y[m, k]) - int(yzp)) * (int(W[k, n]) - 128) for k in range(40))
            s = np.float32(np.float32(ys) * np.float32(0.004))
            assert C[m, n] == np.float32(np.float32(acc) * s)
