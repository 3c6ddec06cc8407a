"""ConvInteger against the oracle, bit for bit, on both routes -- the implicit
GEMM (fp16 NHWC input gathered by im2col tensor copies, for groups of whole
64-channel blocks) and the materialised im2col pre-pass + the SM-pair
MatMulInteger GEMM (the other shapes): every signedness pair, zero points absent / scalar /
per output channel, padding, strides, dilations, groups (depthwise
included), rank-3 NCL inputs, output extents that leave ragged pixel tiles,
long reductions at the exact-chunk edge, int32 wrap-around, empty outputs and
argument errors."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

KERNEL = "im2col_f16+gemm_tc05_pair_f16ops_matmul_integer"
DT = {"u8": np.uint8, "s8": np.int8}


def run(c, zp="both"):
    xzp = dev(c.x_zp) if zp in ("both", "x") else None
    wzp = {"both": dev(c.w_zp), "w": dev(c.w_zp), "w1": dev(c.w_zp[:1])}.get(zp)
    y = q.conv_integer(dev(c.x), dev(c.w), xzp, wzp, pads=c.pads, strides=c.strides, dilations=c.dilations,
                       group=c.group)
    q.check_device_error()
    return host(y)


def want(c, zp="both"):
    xzp = c.x_zp if zp in ("both", "x") else 0
    wzp = {"both": c.w_zp, "w": c.w_zp, "w1": c.w_zp[:1]}.get(zp, 0)
    return O.conv_integer(c.x, c.w, xzp, wzp, c.pads, c.strides, c.dilations, c.group)


GEOMETRIES = [
    # x shape, w shape, pads, strides, dilations, group
    ((2, 16, 13, 11), (24, 16, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 1),
    ((1, 8, 20, 17), (12, 8, 3, 2), [2, 0, 1, 3], [2, 3], [1, 2], 1),
    ((3, 12, 9, 9), (18, 6, 3, 3), [1, 2, 1, 0], [1, 1], [2, 1], 2),
    ((2, 32, 10, 10), (32, 1, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 32),     # depthwise
    ((2, 20, 7, 30), (300, 20, 1, 1), [0, 0, 0, 0], [1, 1], [1, 1], 1),    # 1x1, M > 256
    ((1, 3, 33, 35), (16, 3, 7, 7), [3, 3, 3, 3], [2, 2], [1, 1], 1),      # stem-like, K = 147
    ((2, 16, 16, 16), (32, 16, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 1),    # pixel rows of 16-byte multiples
    ((1, 32, 8, 8), (272, 32, 1, 1), [0, 0, 0, 0], [1, 1], [1, 1], 1),     # 1x1, 272 output channels
    ((3, 48, 12, 20), (300, 48, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 1),   # ragged pair row tile
]


@pytest.mark.parametrize("xdt,wdt", [("u8", "s8"), ("s8", "s8"), ("u8", "u8"), ("s8", "u8")])
@pytest.mark.parametrize("geom", range(len(GEOMETRIES)))
def test_conv_integer_matches_oracle(xdt, wdt, geom):
    xs, ws, pads, strides, dils, group = GEOMETRIES[geom]
    c = W.conv_integer_case(xs, ws, pads, strides, dils, group, seed=geom + 7 * len(xdt + wdt),
                            x_dtype=DT[xdt], w_dtype=DT[wdt])
    got = run(c)
    assert q.last_kernel() == KERNEL
    assert_equal(got, want(c), f"conv {xdt}x{wdt} geometry {geom}")


IM2COL = "conv_f16_nhwc+gemm_tc05_pair_f16ops_conv_im2col"
TMA_GEOMETRIES = [
    ((2, 64, 12, 12), (40, 64, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 1),
    ((1, 128, 18, 15), (72, 128, 3, 2), [2, 0, 1, 3], [2, 3], [1, 2], 1),     # asymmetric pads, strides, dilations
    ((2, 128, 10, 10), (96, 64, 3, 3), [1, 2, 1, 0], [1, 1], [2, 1], 2),      # two groups of 64 channels
    ((2, 64, 16, 30), (300, 64, 1, 1), [0, 0, 0, 0], [1, 1], [1, 1], 1),      # 1x1, M > 256: ragged pair row tile
    ((1, 64, 30, 31), (16, 64, 7, 7), [3, 3, 3, 3], [2, 2], [1, 1], 1),       # 7x7, stride 2
    ((2, 192, 14, 14), (64, 192, 5, 5), [2, 2, 2, 2], [1, 1], [1, 1], 1),     # K = 4800: many exact chunks
    ((1, 64, 36, 36), (8, 64, 3, 3), [0, 1, 2, 0], [3, 2], [2, 3], 1),        # stride 3, dilation 3
]


@pytest.mark.parametrize("xdt,wdt", [("u8", "s8"), ("s8", "s8"), ("u8", "u8"), ("s8", "u8")])
@pytest.mark.parametrize("geom", range(len(TMA_GEOMETRIES)))
def test_conv_integer_implicit_gemm_matches_oracle(xdt, wdt, geom):
    xs, ws, pads, strides, dils, group = TMA_GEOMETRIES[geom]
    c = W.conv_integer_case(xs, ws, pads, strides, dils, group, seed=geom + 11 * len(xdt + wdt),
                            x_dtype=DT[xdt], w_dtype=DT[wdt])
    got = run(c)
    assert q.last_kernel() == IM2COL
    assert_equal(got, want(c), f"implicit-GEMM conv {xdt}x{wdt} geometry {geom}")


@pytest.mark.parametrize("zp", ["none", "x", "w", "w1"])
def test_conv_integer_implicit_gemm_zero_point_forms(zp):
    c = W.conv_integer_case((2, 128, 10, 10), (96, 64, 3, 3), [1, 2, 1, 0], [1, 1], [2, 1], 2, seed=5)
    assert_equal(run(c, zp), want(c, zp), f"implicit GEMM, zero points {zp}")
    assert q.last_kernel() == IM2COL


@pytest.mark.parametrize("L,k,pads,stride,dil", [(52, 3, [1, 1], 1, 1), (301, 5, [2, 0], 2, 2)])
def test_conv_integer_implicit_gemm_rank3(L, k, pads, stride, dil):
    c = W.conv_integer_case((3, 64, L), (40, 64, k), pads, [stride], [dil], 1, seed=L + 1)
    got = run(c)
    assert q.last_kernel() == IM2COL
    assert_equal(got, want(c), f"implicit-GEMM rank-3 L={L} k={k}")


# Batches sized so that, on a 152-SM GB300 (76 SM pairs), the pair-tile width
# chosen for the convolution is 256 (25 images of 768 output pixels: 75 tiles
# of 256, one wave) and 224 (38 images of 448 pixels: 76 tiles of 224); the
# small geometries above all take 192.
WIDTH_GEOMETRIES = [
    ((25, 64, 24, 32), (16, 64, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 1),
    ((38, 64, 16, 28), (16, 64, 3, 3), [1, 1, 1, 1], [1, 1], [1, 1], 1),
]


@pytest.mark.parametrize("geom", range(len(WIDTH_GEOMETRIES)))
def test_conv_integer_implicit_gemm_tile_widths(geom):
    xs, ws, pads, strides, dils, group = WIDTH_GEOMETRIES[geom]
    c = W.conv_integer_case(xs, ws, pads, strides, dils, group, seed=geom + 77)
    got = run(c)
    assert q.last_kernel() == IM2COL
    assert_equal(got, want(c), f"implicit-GEMM conv, tile-width geometry {geom}")


def test_conv_integer_implicit_gemm_extremes_and_wrap():
    """Shifted operands at the extremes (255 - 0 and -128 - 127): each exact
    fp32 chunk of 256 taps sums to 256 * 65025 < 2^24; and a reduction long
    enough to wrap int32."""
    C = 1024
    x = np.full((1, C, 4, 4), 255, np.uint8)
    w = np.full((8, C, 3, 3), -128, np.int8)
    c = W.ConvIntegerCase(x=x, w=w, x_zp=np.array([0], np.uint8), w_zp=np.full(8, 127, np.int8), pads=[1, 1, 1, 1],
                          strides=None, dilations=None, group=1)
    got = run(c)
    assert q.last_kernel() == IM2COL
    assert_equal(got, want(c), "extreme values, 9216 taps")
    C = 4096
    x = np.full((1, C, 4, 4), 255, np.uint8)
    w = np.full((2, C, 3, 3), -128, np.int8)
    c = W.ConvIntegerCase(x=x, w=w, x_zp=np.array([0], np.uint8), w_zp=np.array([127, 127], np.int8), pads=None,
                          strides=None, dilations=None, group=1)
    got = run(c)
    assert q.last_kernel() == IM2COL
    total = 255 * (-255) * C * 9
    assert total < -2**31
    assert (got == (total + 2**31) % 2**32 - 2**31).all()


@pytest.mark.parametrize("zp", ["none", "x", "w", "w1"])
def test_conv_integer_zero_point_forms(zp):
    c = W.conv_integer_case((2, 24, 12, 9), (40, 12, 3, 3), [1, 0, 2, 1], [1, 2], [1, 1], 2, seed=3)
    assert_equal(run(c, zp), want(c, zp), f"zero points {zp}")


@pytest.mark.parametrize("L,k,pads,stride,dil", [(50, 3, [1, 1], 1, 1), (301, 5, [2, 0], 2, 2), (7, 1, [0, 0], 1, 1)])
def test_conv_integer_rank3(L, k, pads, stride, dil):
    c = W.conv_integer_case((3, 24, L), (40, 24, k), pads, [stride], [dil], 1, seed=L)
    got = run(c)
    assert got.shape == want(c).shape
    assert_equal(got, want(c), f"rank-3 L={L} k={k}")


def test_conv_integer_long_reduction_at_the_chunk_edge():
    """K = C*kH*kW = 9216 taps at the extreme values: every exact fp32 chunk of
    raw products (512 taps of -128 * 255) sums to within 2^16 of 2^24."""
    C = 1024
    x = np.full((1, C, 5, 5), 255, np.uint8)
    w = np.full((8, C, 3, 3), -128, np.int8)
    c = W.ConvIntegerCase(x=x, w=w, x_zp=np.array([0], np.uint8), w_zp=np.full(8, 127, np.int8), pads=[1, 1, 1, 1],
                          strides=None, dilations=None, group=1)
    got = run(c)
    ref = want(c)
    assert_equal(got, ref, "extreme values, 9216 taps")
    assert np.abs(ref.astype(np.int64)).max() > 2**28


def test_conv_integer_sums_wrap_modulo_2_32():
    C = 4096
    x = np.full((1, C, 3, 3), 255, np.uint8)
    w = np.full((2, C, 3, 3), -128, np.int8)
    c = W.ConvIntegerCase(x=x, w=w, x_zp=np.array([0], np.uint8), w_zp=np.array([127, 127], np.int8), pads=None,
                          strides=None, dilations=None, group=1)
    got = run(c)
    total = 255 * (-255) * C * 9
    assert total < -2**31
    assert (got == (total + 2**31) % 2**32 - 2**31).all()


def test_conv_integer_empty_and_errors():
    x = torch.zeros((2, 4, 3, 3), dtype=torch.uint8, device="cuda")
    w = torch.zeros((4, 4, 5, 5), dtype=torch.int8, device="cuda")
    y = q.conv_integer(x, w)                      # kernel wider than the input: empty output
    assert tuple(y.shape) == (2, 4, 0, 0)
    with pytest.raises(ValueError):
        q.conv_integer(x, torch.zeros((6, 3, 1, 1), dtype=torch.int8, device="cuda"), group=2)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        q.conv_integer(x, torch.zeros((4, 4, 1, 1), dtype=torch.int8, device="cuda"), workspace=ws)
    with pytest.raises(q.QmmError):
        q.conv_integer(x, torch.zeros((4, 4, 1, 1), dtype=torch.int8, device="cuda"), strides=[0, 1])
