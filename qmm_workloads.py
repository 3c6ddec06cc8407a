"""Seeded synthetic inputs for the quantized-matmul hot path.

This module only draws random inputs. It holds none of the arithmetic of the
method: no matmul, no scaling, no rounding to an output type, no quantisation.
Both the CPU oracle (tests, bench baseline) and the CUDA path (tests, bench)
take their inputs from here, so the two sides see the same bytes.

Every generator uses ``numpy.random.default_rng(seed)`` (seed 0 for the five
named workloads) and draws its arrays in the order written below, so a
workload is reproducible from its name and seed alone.

bf16 activations are produced as float32 values whose low 16 bits are zero
(the draw is truncated, not rounded), so each value is exactly a bf16 number
and no rounding rule is needed here. They are returned both as the float32
array and as the uint16 bit pattern.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def rng_for(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def uniform_int(rng: np.random.Generator, lo: int, hi: int, shape, dtype) -> np.ndarray:
    """Integers uniform on the inclusive range [lo, hi]."""
    return rng.integers(lo, hi + 1, size=shape, dtype=dtype)


def uniform_f32(rng: np.random.Generator, lo: float, hi: float, shape) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def bf16_exact_normal(rng: np.random.Generator, shape):
    """N(0,1) draws truncated to bf16-representable float32 values.

    Returns (values_f32, bits_u16)."""
    v = normal_f32(rng, shape)
    bits32 = v.view(np.uint32) & np.uint32(0xFFFF0000)
    vals = bits32.view(np.float32)
    bits16 = (bits32 >> np.uint32(16)).astype(np.uint16)
    return vals, bits16


def with_outliers(rng: np.random.Generator, x: np.ndarray, prob: float, factor: float) -> np.ndarray:
    """Multiply each element, independently with probability ``prob``, by ``factor``."""
    mask = rng.random(size=x.shape) < prob
    out = x.copy()
    out[mask] *= np.float32(factor)
    return out


# ---------------------------------------------------------------------------
# The five named workloads. Shapes and distributions are those of the pages'
# hot path at its benchmark sizes; each is drawn from seed 0.
# ---------------------------------------------------------------------------

@dataclass
class W8DequantF32:
    """fp32 activations x int8 weight, one per-tensor scale and zero point."""
    A: np.ndarray          # f32 [M, K]
    B: np.ndarray          # i8  [K, N]
    scale: np.ndarray      # f32 [1]
    zero_point: np.ndarray  # i32 [1]


def w8_dequant_f32_64x256x192(seed: int = 0) -> W8DequantF32:
    rng = rng_for(seed)
    A = uniform_f32(rng, -1.0, 1.0, (64, 256))
    B = uniform_int(rng, -128, 127, (256, 192), np.int8)
    return W8DequantF32(A=A, B=B, scale=np.array([0.02], np.float32),
                        zero_point=np.array([3], np.int32))


@dataclass
class A8W8:
    A: np.ndarray            # i8 [M, K]
    B: np.ndarray            # i8 [K, N]
    act_scale: np.ndarray    # f32 [M]
    weight_scale: np.ndarray  # f32 [N]


def a8w8(M: int, K: int, N: int, seed: int = 0) -> A8W8:
    rng = rng_for(seed)
    A = uniform_int(rng, -127, 127, (M, K), np.int8)
    B = uniform_int(rng, -127, 127, (K, N), np.int8)
    act = uniform_f32(rng, 0.005, 0.02, (M,))
    ws = uniform_f32(rng, 0.001, 0.01, (N,))
    return A8W8(A=A, B=B, act_scale=act, weight_scale=ws)


def a8w8_4096(seed: int = 0) -> A8W8:
    return a8w8(4096, 4096, 4096, seed)


@dataclass
class A8W8Acc:
    A: np.ndarray             # i8, stored [M, K], or [K, M] when a_trans
    B: np.ndarray             # i8, stored [K, N], or [N, K] when b_trans
    acc_in: np.ndarray        # i32 [M, N]
    act_scale: np.ndarray     # f32 [M]
    weight_scale: np.ndarray  # f32 [N]
    a_trans: bool
    b_trans: bool


def a8w8_acc(M: int, K: int, N: int, seed: int = 0, a_trans: bool = False, b_trans: bool = False,
             acc_bound: int = 2**24) -> A8W8Acc:
    """The accumulating A8W8's inputs: the A8W8 operand recipe, stored in the
    given layouts, and an int32 accumulator uniform in [-acc_bound, acc_bound)
    (a partial sum carried in from an earlier part of K; 2**31 spans int32)."""
    w = a8w8(M, K, N, seed)
    rng = rng_for(seed + 1)
    acc = rng.integers(-acc_bound, acc_bound, size=(M, N), dtype=np.int64).astype(np.int32)
    A = np.ascontiguousarray(w.A.T) if a_trans else w.A
    B = np.ascontiguousarray(w.B.T) if b_trans else w.B
    return A8W8Acc(A=A, B=B, acc_in=acc, act_scale=w.act_scale, weight_scale=w.weight_scale, a_trans=a_trans,
                   b_trans=b_trans)


@dataclass
class ConvIntegerCase:
    x: np.ndarray        # u8 [N, C, H, W] or [N, C, L]
    w: np.ndarray        # s8 [M, C/group, kH, kW] or [M, C/group, k]
    x_zp: np.ndarray     # u8 [1]
    w_zp: np.ndarray     # s8 [M]
    pads: list
    strides: list
    dilations: list
    group: int


def conv_integer_case(x_shape, w_shape, pads=None, strides=None, dilations=None, group=1, seed=0,
                      x_dtype=np.uint8, w_dtype=np.int8) -> ConvIntegerCase:
    """Quantised-convolution inputs: activations and weights uniform over their
    8-bit range, a scalar activation zero point and one weight zero point per
    output channel, drawn from the same ranges."""
    rng = rng_for(seed)
    lo = {np.uint8: 0, np.int8: -128}
    x = uniform_int(rng, lo[x_dtype], lo[x_dtype] + 255, x_shape, x_dtype)
    w = uniform_int(rng, lo[w_dtype], lo[w_dtype] + 255, w_shape, w_dtype)
    xzp = uniform_int(rng, lo[x_dtype], lo[x_dtype] + 255, (1,), x_dtype)
    wzp = uniform_int(rng, lo[w_dtype], lo[w_dtype] + 255, (w_shape[0],), w_dtype)
    return ConvIntegerCase(x=x, w=w, x_zp=xzp, w_zp=wzp, pads=pads, strides=strides, dilations=dilations,
                           group=group)


def conv2d_3x3_8x256x56x56(seed: int = 0) -> ConvIntegerCase:
    """A 3x3 convolution layer, 256 -> 256 channels on 56 x 56 maps, batch 8, same padding."""
    return conv_integer_case((8, 256, 56, 56), (256, 256, 3, 3), pads=[1, 1, 1, 1], seed=seed)


def conv1d_k3_4x512x3000(seed: int = 0) -> ConvIntegerCase:
    """A rank-3 (NCL) encoder convolution, 512 -> 512 channels, kernel 3, length 3000, batch 4."""
    return conv_integer_case((4, 512, 3000), (512, 512, 3), pads=[1, 1], seed=seed)


@dataclass
class DqlMatMulInteger:
    x: np.ndarray      # f32 [M, K]
    B: np.ndarray      # i8 [K, N]
    b_zp: np.ndarray   # i8 [N]


def dql_matmul_integer(M: int, K: int, N: int, seed: int = 0) -> DqlMatMulInteger:
    rng = rng_for(seed)
    x = normal_f32(rng, (M, K))
    x = with_outliers(rng, x, 0.001, 20.0)
    B = uniform_int(rng, -128, 127, (K, N), np.int8)
    b_zp = uniform_int(rng, -128, 127, (N,), np.int8)
    return DqlMatMulInteger(x=x, B=B, b_zp=b_zp)


def dql_matmul_integer_8192x4096x11008(seed: int = 0) -> DqlMatMulInteger:
    return dql_matmul_integer(8192, 4096, 11008, seed)


@dataclass
class DecodeGemv:
    A: np.ndarray        # f32 [M, K], every value exactly bf16
    A_bits: np.ndarray   # u16 [M, K], the bf16 bit patterns of A
    W: np.ndarray        # i8 [K, N]
    scale: np.ndarray    # f32 [N]


def decode_gemv(M: int, K: int = 8192, N: int = 28672, seed: int = 0) -> DecodeGemv:
    rng = rng_for(seed)
    A, A_bits = bf16_exact_normal(rng, (M, K))
    W = uniform_int(rng, -127, 127, (K, N), np.int8)
    scale = uniform_f32(rng, 0.001, 0.01, (N,))
    return DecodeGemv(A=A, A_bits=A_bits, W=W, scale=scale)


@dataclass
class BatchedMatMulInteger:
    A: np.ndarray   # i8 [batch..., M, K]
    B: np.ndarray   # i8 [K, N], shared by every batch (batch stride 0)
    a_zp: int
    b_zp: int


def batched_matmul_integer(shape=(8, 16, 512, 1024), N: int = 1024, seed: int = 0,
                           a_zp: int = -5, b_zp: int = 7) -> BatchedMatMulInteger:
    rng = rng_for(seed)
    K = shape[-1]
    A = uniform_int(rng, -128, 127, shape, np.int8)
    B = uniform_int(rng, -128, 127, (K, N), np.int8)
    return BatchedMatMulInteger(A=A, B=B, a_zp=a_zp, b_zp=b_zp)


WORKLOADS = {
    "w8_dequant_f32_64x256x192": "A f32 [64,256] U(-1,1); B i8 [256,192] U{-128..127}; scale 0.02; zp 3",
    "a8w8_4096x4096x4096_bf16": "A,B i8 [4096,4096] U{-127..127}; act_scale [M] U(0.005,0.02); "
                                "weight_scale [N] U(0.001,0.01); bf16 out",
    "dql_matmul_integer_8192x4096x11008": "x f32 [8192,4096] N(0,1), 0.1% x20 outliers -> u8; "
                                          "B i8 [4096,11008] U{-128..127}; b_zp i8 [11008]; i32 out",
    "decode_gemv_Mx8192x28672": "A bf16 [M,8192] N(0,1), M in {1,4,16}; W i8 [8192,28672] U{-127..127}; "
                                "scale [N] U(0.001,0.01); zp 0; bf16 out",
    "batched_matmul_integer_8x16x512x1024x1024": "A i8 [8,16,512,1024] U{-128..127}; shared B i8 [1024,1024]; "
                                                 "a_zp -5; b_zp 7; i32 out",
}
