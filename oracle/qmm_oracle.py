"""CPU oracle for the integer-quantised matmul with fused dequantisation.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``, and by nothing else. The product path (the CUDA library
and its Python binding) never imports or calls it, and the two share no code:
the only module both sides use is ``qmm_workloads``, which draws seeded random
inputs and does none of the method's arithmetic.

It is deliberately plain and slow: integer sums are taken in int64 with numpy's
integer matmul (exact), real-valued references in float64, and the steps that
the pages fix in single precision (the A8W8 epilogue chain, DynamicQuantizeLinear)
in numpy float32 scalar/array arithmetic, which rounds every operation to
nearest-even. No step is blocked, fused or reordered beyond what its definition
states.

Sources (the five pages the method is taken from):
  [P1] TrainDeeploy PR #53, "feat(PULPOpen): matmul that dequantises an int8
       weight in-kernel" -- sections "The kernel" and the author's follow-up.
  [P2] PyPTO PR #1920, "Feature/a8w8 matmul dequant fusion" -- the walkthrough's
       sequence diagram, and the two review comments on 1-D scale shapes.
  [P5] ROCm hip-ep PR #1248, "feat(onnx-to-hip): lower quantized integer conv
       and matmul" -- sections "What" (DynamicQuantizeLinear, MatMulInteger),
       "Test plan", and the review comments.

Parity pins: every public function below is pinned in
``tests/test_oracle_pins.py`` against facts that do not come from this file
(the pages' worked values under ``tests/golden/``, closed forms, algebraic
identities, and brute force in exact Python integers/rationals).
"""
from __future__ import annotations

import numpy as np

INT32_MOD = 1 << 32


# ---------------------------------------------------------------------------
# Number-format helpers
# ---------------------------------------------------------------------------

def wrap_int32(x: np.ndarray) -> np.ndarray:
    """Two's-complement wrap of an int64 array to int32.

    [P5] "What", MatMulInteger paragraph: a long reduction accumulates in int64
    and then stores a wrapping int32."""
    x = np.asarray(x, dtype=np.int64)
    return (((x + (1 << 31)) % INT32_MOD) - (1 << 31)).astype(np.int32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16, nearest with ties to even, returning uint16 bits.

    bf16 keeps the top 16 bits of a float32. Adding 0x7FFF plus the lowest kept
    bit before truncating rounds to nearest and breaks ties toward an even kept
    part. NaN/Inf inputs are outside the method's domain."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def _as_vector(v, length: int, name: str) -> np.ndarray:
    v = np.asarray(v).reshape(-1)
    if v.size == 1:
        return np.repeat(v, length)
    if v.size != length:
        raise ValueError(f"{name}: expected 1 or {length} values, got {v.size}")
    return v


# ---------------------------------------------------------------------------
# Form (a): int8-weight matmul with the affine dequantisation factored out
# ---------------------------------------------------------------------------

def w8_dequant(A: np.ndarray, B: np.ndarray, scale, zero_point) -> np.ndarray:
    """C[m,n] = scale_n * (sum_k A[m,k]*B[k,n] - zp_n * sum_k A[m,k]), in float64.

    [P1] "The kernel": the affine dequantisation of the weight,
    a_k*(b_k - zp)*scale summed over k, factors into scale times the plain dot
    product minus zp times the sum of the activations, so the correction is one
    multiply per output. The page has one per-tensor scale and zero point; a
    per-column scale/zero point (one value per output column n) is the same
    identity applied column by column and is what the decode workload uses.

    A: float activations [M, K] (fp32, or bf16 widened exactly to fp32).
    B: int8 weight [K, N]. scale: 1 or N values. zero_point: 1 or N integers.
    Returns the exact-arithmetic reference in float64 (no output rounding)."""
    A64 = np.asarray(A, dtype=np.float64)
    B64 = np.asarray(B, dtype=np.int64).astype(np.float64)
    M, K = A64.shape
    N = B64.shape[1]
    s = _as_vector(scale, N, "scale").astype(np.float64)
    zp = _as_vector(zero_point, N, "zero_point").astype(np.float64)
    dot = A64 @ B64                       # sum_k a*b
    rowsum = A64.sum(axis=1)              # sum_k a
    return s[None, :] * (dot - zp[None, :] * rowsum[:, None])


def w8_dequant_explicit(A: np.ndarray, B: np.ndarray, scale, zero_point) -> np.ndarray:
    """The unfused form: materialise the dequantised weight, then matmul (float64).

    [P1] first paragraph: a separate Dequant node materialises the whole float
    weight scale*(B - zp) before the matmul reads it. This is the form the
    fused kernel avoids; the oracle keeps it only as a cross-check of
    ``w8_dequant`` (the factoring identity of [P1] "The kernel")."""
    A64 = np.asarray(A, dtype=np.float64)
    N = B.shape[1]
    s = _as_vector(scale, N, "scale").astype(np.float64)
    zp = _as_vector(zero_point, N, "zero_point").astype(np.float64)
    Bf = s[None, :] * (np.asarray(B, dtype=np.float64) - zp[None, :])
    return A64 @ Bf


def w8_dequant_error_bound(A: np.ndarray, B: np.ndarray, scale, zero_point) -> np.ndarray:
    """Per-element tolerance: 1e-3 * sum_k |a_k * scale_n*(b_k - zp_n)| + 1e-6.

    The stated bound is 1e-3 * scale * sum_k |a_k b_k| + 1e-6; with a nonzero
    zero point the summand actually dequantised is scale*(b_k - zp), so that is
    the term whose magnitude is summed."""
    A64 = np.abs(np.asarray(A, dtype=np.float64))
    N = B.shape[1]
    s = _as_vector(scale, N, "scale").astype(np.float64)
    zp = _as_vector(zero_point, N, "zero_point").astype(np.float64)
    Bd = np.abs(s[None, :] * (np.asarray(B, dtype=np.float64) - zp[None, :]))
    return 1e-3 * (A64 @ Bd) + 1e-6


# ---------------------------------------------------------------------------
# Form (b): A8W8 -- exact int32 product, then row and column scales
# ---------------------------------------------------------------------------

def a8w8_acc(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """acc[m,n] = sum_k A[m,k]*B[k,n], int8 x int8 summed exactly, wrapped to int32.

    [P2] sequence diagram, first step: the int8 matmul lowers into an INT32
    accumulator."""
    acc = np.matmul(np.asarray(A, dtype=np.int64), np.asarray(B, dtype=np.int64))
    return wrap_int32(acc)


def a8w8(A: np.ndarray, B: np.ndarray, act_scale, weight_scale, out: str = "f32"):
    """A8W8 matmul-dequant in the pages' order, every step in float32.

    [P2] sequence diagram: INT32 accumulator -> cast to FP32 -> multiply by
    act_scale on rows -> multiply by weight_scale on columns -> cast to
    out_dtype. [P2] review comments on 1-D scales: an [M] activation scale
    scales rows (it is [M,1]) and an [N] weight scale scales columns ([1,N]),
    never a last-dimension broadcast, even when M == N. A single value is a
    scalar scale.

    Returns float32 [M,N] for out="f32", or bf16 bits (uint16) for out="bf16"."""
    acc = a8w8_acc(A, B)
    M, N = acc.shape
    a_s = _as_vector(act_scale, M, "act_scale").astype(np.float32)
    w_s = _as_vector(weight_scale, N, "weight_scale").astype(np.float32)
    f = acc.astype(np.float32)                 # int32 -> fp32, nearest even
    f = (f * a_s[:, None]).astype(np.float32)  # rows first
    f = (f * w_s[None, :]).astype(np.float32)  # then columns
    if out == "f32":
        return f
    if out == "bf16":
        return f32_to_bf16_bits(f)
    raise ValueError(out)


def a8w8_dequant_acc(acc_in, A: np.ndarray, B: np.ndarray, act_scale, weight_scale, out: str = "f32"):
    """The accumulating A8W8 variant: the int32 accumulator is acc_in plus the
    exact int32 product, wrapping, then the same float32 steps as a8w8.

    [P2] names tensor.a8w8_matmul_dequant_acc (an INT32 accumulator input
    beside the INT8 operands, lowered through tile.matmul_acc / tile.gemv_acc
    then the cast and the two scale multiplies) without spelling out its
    arithmetic; this is the plainest reading: matmul_acc adds the product to
    the accumulator it is given. acc_in is an int32 [M,N] array (or 0).
    Returns what a8w8 returns for the combined accumulator."""
    prod = a8w8_acc(A, B)
    acc = wrap_int32(np.asarray(acc_in, dtype=np.int64) + prod.astype(np.int64))
    return _a8w8_epilogue(acc, act_scale, weight_scale, out)


def _a8w8_epilogue(acc: np.ndarray, act_scale, weight_scale, out: str):
    M, N = acc.shape
    a_s = _as_vector(act_scale, M, "act_scale").astype(np.float32)
    w_s = _as_vector(weight_scale, N, "weight_scale").astype(np.float32)
    f = acc.astype(np.float32)                 # int32 -> fp32, nearest even
    f = (f * a_s[:, None]).astype(np.float32)  # rows first
    f = (f * w_s[None, :]).astype(np.float32)  # then columns
    if out == "f32":
        return f
    if out == "bf16":
        return f32_to_bf16_bits(f)
    raise ValueError(out)


def a8w8_exact(A: np.ndarray, B: np.ndarray, act_scale, weight_scale) -> np.ndarray:
    """float64 value of act_scale[m] * weight_scale[n] * acc[m,n] (no float32 steps).

    The real-valued result the float32 chain of a8w8 approximates; acc is the
    int32 accumulator of a8w8_acc and the scales keep the [M] rows / [N]
    columns orientation of [P2]'s review comments."""
    acc = a8w8_acc(A, B).astype(np.float64)
    M, N = acc.shape
    a_s = _as_vector(act_scale, M, "act_scale").astype(np.float64)
    w_s = _as_vector(weight_scale, N, "weight_scale").astype(np.float64)
    return acc * a_s[:, None] * w_s[None, :]


def a8w8_error_bound(A: np.ndarray, B: np.ndarray, act_scale, weight_scale) -> np.ndarray:
    """1e-3 * act_scale[m]*weight_scale[n] * sum_k |a_k b_k| + 1e-6 per element."""
    absdot = np.matmul(np.abs(np.asarray(A, dtype=np.int64)),
                       np.abs(np.asarray(B, dtype=np.int64))).astype(np.float64)
    M, N = absdot.shape
    a_s = _as_vector(act_scale, M, "act_scale").astype(np.float64)
    w_s = _as_vector(weight_scale, N, "weight_scale").astype(np.float64)
    return 1e-3 * absdot * a_s[:, None] * w_s[None, :] + 1e-6


# ---------------------------------------------------------------------------
# Form (c): MatMulInteger with zero points
# ---------------------------------------------------------------------------

def matmul_integer(A: np.ndarray, B: np.ndarray, a_zero_point=0, b_zero_point=0) -> np.ndarray:
    """C = sum_k (A[...,m,k] - a_zp) * (B[...,k,n] - b_zp), int64 exact, wrapped to int32.

    [P5] "What", MatMulInteger paragraph: ranks 2 to 4; an 8-bit value minus an
    8-bit zero point is at most 255 in magnitude; the sum is taken in int64 and
    stored as a wrapping int32. A rank-2 B is one matrix shared by every batch
    of A (numpy broadcasting gives exactly that). The activation zero point is
    a scalar or one value per row m ([M]); the weight zero point is a scalar or
    one value per column n ([N], placed as [..., 1, N]).

    This is the direct definition; it does not use the expanded
    sum ab - a_zp*colsum(B) - b_zp*rowsum(A) + K*a_zp*b_zp form."""
    A64 = np.asarray(A, dtype=np.int64)
    B64 = np.asarray(B, dtype=np.int64)
    M = A64.shape[-2]
    N = B64.shape[-1]
    azp = np.asarray(a_zero_point, dtype=np.int64).reshape(-1)
    bzp = np.asarray(b_zero_point, dtype=np.int64).reshape(-1)
    if azp.size == 1:
        Ac = A64 - azp[0]
    elif azp.size == M:
        Ac = A64 - azp[:, None]                   # one value per row
    else:
        raise ValueError("a_zero_point must have 1 or M values")
    if bzp.size == 1:
        Bc = B64 - bzp[0]
    elif bzp.size == N:
        Bc = B64 - bzp[None, :]                   # one value per column
    else:
        raise ValueError("b_zero_point must have 1 or N values")
    return wrap_int32(np.matmul(Ac, Bc))


# ---------------------------------------------------------------------------
# ConvInteger
# ---------------------------------------------------------------------------

def conv_output_size(size: int, k: int, pad_begin: int, pad_end: int, stride: int, dilation: int) -> int:
    """Output extent of one spatial axis: floor((size + pads - dilation*(k-1) - 1) / stride) + 1."""
    return (size + pad_begin + pad_end - dilation * (k - 1) - 1) // stride + 1


def conv_integer(x: np.ndarray, w: np.ndarray, x_zero_point=0, w_zero_point=0, pads=None, strides=None,
                 dilations=None, group: int = 1) -> np.ndarray:
    """y[n,m,oh,ow] = sum over the group's channels c and the kernel taps (kh,kw) of
    (xs[n,c,oh*sh+kh*dh-pt, ow*sw+kw*dw-pl]) * (w[m,c,kh,kw] - w_zp[m]),
    xs = x - x_zp and 0 outside the input (the padding); int64, wrapped to int32.

    [P5] "What", ConvInteger paragraph: rank-4 NCHW, and rank-3 NCL widened to
    the rank-4 path with a unit spatial row (NC1L) whose result is collapsed;
    the activation zero point is a scalar; the weight zero point is a scalar or
    one value per output channel. The page does not state the value taken at
    padded positions; this reads the operator as the convolution of the
    zero-point-shifted tensors, so a padded position contributes nothing
    (equivalently, the input is padded with x_zp). pads follow ONNX order
    [top, left, bottom, right] ([begin, end] for rank 3); strides and
    dilations are (h, w) (one value for rank 3). w is [M, C/group, kH, kW]."""
    x = np.asarray(x)
    w = np.asarray(w)
    rank3 = x.ndim == 3
    if rank3:                                   # NCL -> NC1L
        x = x[:, :, None, :]
        w = w[:, :, None, :]
        pads = [0, 0, 0, 0] if pads is None else [0, pads[0], 0, pads[1]]
        strides = [1, 1] if strides is None else [1, strides[0]]
        dilations = [1, 1] if dilations is None else [1, dilations[0]]
    pads = [0, 0, 0, 0] if pads is None else list(pads)
    strides = [1, 1] if strides is None else list(strides)
    dilations = [1, 1] if dilations is None else list(dilations)
    Nb, C, H, W_ = x.shape
    M, Cg, kH, kW = w.shape
    if C != Cg * group or M % group != 0:
        raise ValueError("channels do not divide into the groups")
    Mg = M // group
    pt, pl, pb, pr = pads
    sh, sw = strides
    dh, dw = dilations
    oH = conv_output_size(H, kH, pt, pb, sh, dh)
    oW = conv_output_size(W_, kW, pl, pr, sw, dw)
    xzp = np.asarray(x_zero_point, dtype=np.int64).reshape(-1)
    wzp = np.asarray(w_zero_point, dtype=np.int64).reshape(-1)
    if xzp.size != 1:
        raise ValueError("x_zero_point must be a scalar")
    if wzp.size not in (1, M):
        raise ValueError("w_zero_point must have 1 or M values")
    xs = x.astype(np.int64) - xzp[0]
    ws = w.astype(np.int64) - (wzp[0] if wzp.size == 1 else wzp[:, None, None, None])
    xp = np.zeros((Nb, C, H + pt + pb, W_ + pl + pr), dtype=np.int64)
    xp[:, :, pt:pt + H, pl:pl + W_] = xs
    y = np.zeros((Nb, M, oH, oW), dtype=np.int64)
    for g in range(group):
        xg = xp[:, g * Cg:(g + 1) * Cg]
        for kh in range(kH):
            for kw in range(kW):
                h0, w0 = kh * dh, kw * dw
                patch = xg[:, :, h0:h0 + sh * (oH - 1) + 1:sh, w0:w0 + sw * (oW - 1) + 1:sw]   # [N, Cg, oH, oW]
                tap = ws[g * Mg:(g + 1) * Mg, :, kh, kw]                                        # [Mg, Cg]
                y[:, g * Mg:(g + 1) * Mg] += np.einsum("nchw,mc->nmhw", patch, tap)
    y = wrap_int32(y)
    return y[:, :, 0, :] if rank3 else y


# ---------------------------------------------------------------------------
# Form (d): DynamicQuantizeLinear (uint8)
# ---------------------------------------------------------------------------

def dql_range(x: np.ndarray):
    """(lo, hi) = (min(0, min x), max(0, max x)) in float32.

    [P5] "What", DynamicQuantizeLinear: single-axis ReduceMin / ReduceMax down
    to a scalar. The range is widened to include 0 so that zero is exactly
    representable and the zero point lands in [0, 255]. Empty input gives (0, 0)."""
    x = np.asarray(x, dtype=np.float32).reshape(-1)
    if x.size == 0:
        return np.float32(0.0), np.float32(0.0)
    lo = np.minimum(np.float32(0.0), x.min())
    hi = np.maximum(np.float32(0.0), x.max())
    return np.float32(lo), np.float32(hi)


def dql_scale_zero_point(lo: np.float32, hi: np.float32):
    """scale = (hi - lo) / 255, or 1 when the range is zero; zp = sat_u8(rne(-lo/scale)).

    [P5] "What": scale (max - min) / 255 with a zero range selecting scale 1,
    and a ties-to-even zero point. Each step is one float32 operation rounded
    to nearest even; the division is a true division."""
    lo = np.float32(lo)
    hi = np.float32(hi)
    r = np.float32(hi - lo)
    scale = np.float32(1.0) if r == np.float32(0.0) else np.float32(r / np.float32(255.0))
    q = np.float32(np.float32(-lo) / scale)
    zp = int(np.clip(np.rint(q), 0, 255))        # rint: nearest, ties to even
    return scale, np.uint8(zp)


def quantize_linear(x: np.ndarray, scale: np.float32, zero_point) -> np.ndarray:
    """y = sat_u8(rne(x / scale) + zero_point), elementwise, float32 division.

    [P5] "What": hip.quantize_linear at axis 0 with the scalar scale and zero
    point. Rounding is to nearest even (the plainest reading, the same rule the
    page gives for the zero point); the rounded quotient and the zero point are
    added as integers, then saturated to [0, 255]."""
    x = np.asarray(x, dtype=np.float32)
    q = (x / np.float32(scale)).astype(np.float32)
    r = np.rint(q).astype(np.int64) + int(zero_point)
    return np.clip(r, 0, 255).astype(np.uint8)


def dynamic_quantize_linear(x: np.ndarray):
    """(y uint8, y_scale float32, y_zero_point uint8) for a float32 tensor x."""
    lo, hi = dql_range(x)
    scale, zp = dql_scale_zero_point(lo, hi)
    y = quantize_linear(x, scale, zp)
    return y, scale, zp


def row_sums(y: np.ndarray, row_len: int) -> np.ndarray:
    """sum over each run of row_len consecutive elements, int32 (exact for u8 rows < 2^23)."""
    y = np.asarray(y).reshape(-1, row_len).astype(np.int64)
    return wrap_int32(y.sum(axis=1))


def col_sums(B: np.ndarray) -> np.ndarray:
    """sum_k B[k, n] as int32 (wrapped)."""
    return wrap_int32(np.asarray(B, dtype=np.int64).sum(axis=0))


# ---------------------------------------------------------------------------
# The chain DynamicQuantizeLinear -> MatMulInteger -> dequantise
# ---------------------------------------------------------------------------

def dynamic_quantize_matmul(x: np.ndarray, W: np.ndarray, w_scale, w_zero_point=0, bias=None, rows=None):
    """C = f32(f32(acc) * s[n]) (+ bias[n]), s[n] = f32(y_scale * w_scale[n]),
    acc = MatMulInteger(y, W, y_zp, w_zp), (y, y_scale, y_zp) = DynamicQuantizeLinear(x).

    [P5] "Why" and "What": a graph using MatMulInteger casts, scales and adds
    the bias after it (the fused qlinear ops would scale twice). This is the
    plainest reading of those graph steps, each an fp32 operation rounded to
    nearest even: Cast(int32 -> fp32), Mul(y_scale, w_scale) into one fp32
    multiplier per column, Mul(cast, multiplier), then Add(bias).
    x is float32 [M, K]; W is int8 or uint8 [K, N]; w_scale and w_zero_point
    have 1 or N values. Returns (C float32 [M, N], y_scale, y_zp); with rows
    given, C holds only those rows (the quantiser still sees all of x)."""
    x = np.asarray(x, dtype=np.float32)
    N = np.asarray(W).shape[1]
    y, ys, yzp = dynamic_quantize_linear(x)
    if rows is not None:
        y = y[rows]
    acc = matmul_integer(y, W, int(yzp), w_zero_point)
    ws = _as_vector(w_scale, N, "w_scale").astype(np.float32)
    s = (np.float32(ys) * ws).astype(np.float32)
    C = (acc.astype(np.float32) * s[None, :]).astype(np.float32)
    if bias is not None:
        C = (C + _as_vector(bias, N, "bias").astype(np.float32)[None, :]).astype(np.float32)
    return C, ys, yzp
