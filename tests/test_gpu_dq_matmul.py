"""The fused DynamicQuantizeLinear -> MatMulInteger -> dequantise chain against
the oracle, bit for bit (the quantiser's scale and zero point, and every fp32
output): int8 and uint8 weights, weight zero points absent / scalar / per
column, scalar and per-column weight scales, with and without bias, rows whose
length is not a multiple of 4 (the scalar quantize path), ragged tiles, and
argument errors."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

KERNEL = "dql_f16+gemm_tc05_pair_f16ops_matmul_integer_dequant"


def case(M, K, N, seed, wdt=np.int8, zp="vector", scale="vector", bias=True):
    rng = np.random.default_rng(seed)
    x = W.with_outliers(rng, W.normal_f32(rng, (M, K)), 0.001, 20.0)
    lo = -128 if wdt == np.int8 else 0
    Wm = rng.integers(lo, lo + 256, size=(K, N)).astype(wdt)
    w_scale = rng.uniform(0.001, 0.01, N if scale == "vector" else 1).astype(np.float32)
    w_zp = {"none": None, "scalar": rng.integers(lo, lo + 256, size=1).astype(wdt),
            "vector": rng.integers(lo, lo + 256, size=N).astype(wdt)}[zp]
    b = rng.standard_normal(N).astype(np.float32) if bias else None
    return x, Wm, w_scale, w_zp, b


def run(x, Wm, w_scale, w_zp, b):
    C, ys, yz = q.dynamic_quantize_matmul(dev(x), dev(Wm), dev(w_scale), None if w_zp is None else dev(w_zp),
                                          None if b is None else dev(b))
    q.check_device_error()
    return host(C), float(ys.item()), int(yz.item())


def check(x, Wm, w_scale, w_zp, b, tag):
    C, ys, yz = run(x, Wm, w_scale, w_zp, b)
    assert q.last_kernel() == KERNEL
    want, wys, wyz = O.dynamic_quantize_matmul(x, Wm, w_scale, 0 if w_zp is None else w_zp, b)
    assert ys == float(wys) and yz == int(wyz), tag
    assert_equal(C, want, tag)


SHAPES = [(1, 64, 256), (7, 33, 5), (300, 1040, 272), (257, 100, 129), (130, 4104, 40), (512, 4096, 1008)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("wdt", [np.int8, np.uint8])
def test_chain_matches_oracle(M, K, N, wdt):
    check(*case(M, K, N, seed=M + K + N, wdt=wdt), f"{M}x{K}x{N} {np.dtype(wdt).name}")


@pytest.mark.parametrize("zp", ["none", "scalar", "vector"])
@pytest.mark.parametrize("scale", ["scalar", "vector"])
@pytest.mark.parametrize("bias", [False, True])
def test_chain_zero_point_scale_and_bias_forms(zp, scale, bias):
    check(*case(260, 520, 200, seed=5, zp=zp, scale=scale, bias=bias), f"zp={zp} scale={scale} bias={bias}")


def test_chain_constant_input():
    """A zero range: scale 1, zero point 0 (x all 0) and a one-sided range (x all positive)."""
    x = np.zeros((64, 96), np.float32)
    _, Wm, w_scale, w_zp, b = case(64, 96, 48, seed=3)
    check(x, Wm, w_scale, w_zp, b, "all zero")
    x = np.full((64, 96), 2.5, np.float32)
    check(x, Wm, w_scale, w_zp, b, "all positive")


def test_chain_argument_errors():
    x = torch.zeros((4, 8), device="cuda")
    Wm = torch.zeros((8, 3), dtype=torch.int8, device="cuda")
    with pytest.raises(ValueError):
        q.dynamic_quantize_matmul(x, Wm, torch.ones(2, device="cuda"))
    need = q.dynamic_quantize_matmul_workspace_bytes(4, 8, 3)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        q.dynamic_quantize_matmul(x, Wm, torch.ones(1, device="cuda"), workspace=small)


PACKED = "dql_f16+gemm_tc05_pair_f16ops_matmul_integer_dequant_packed"


def check_packed(x, Wm, w_scale, w_zp, b, tag, reuse=1):
    """The chain on a weight packed once, called `reuse` times on fresh
    activations: each call bit-exact against the oracle."""
    pw = q.dynamic_quantize_matmul_pack_weight(dev(Wm))
    assert q.last_kernel() == "dqm_weight_f16"
    rng = np.random.default_rng(len(tag))
    for i in range(reuse):
        xi = x if i == 0 else W.normal_f32(rng, x.shape) * np.float32(1 + i)
        C, ys, yz = q.dynamic_quantize_matmul_packed(dev(xi), pw, dev(w_scale), None if w_zp is None else dev(w_zp),
                                                     None if b is None else dev(b))
        q.check_device_error()
        assert q.last_kernel() == PACKED
        want, wys, wyz = O.dynamic_quantize_matmul(xi, Wm, w_scale, 0 if w_zp is None else w_zp, b)
        assert float(ys.item()) == float(wys) and int(yz.item()) == int(wyz), tag
        assert_equal(host(C), want, f"{tag} call {i}")


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("wdt", [np.int8, np.uint8])
def test_packed_chain_matches_oracle(M, K, N, wdt):
    check_packed(*case(M, K, N, seed=M + K + N + 1, wdt=wdt), f"{M}x{K}x{N} {np.dtype(wdt).name}")


@pytest.mark.parametrize("zp", ["none", "scalar", "vector"])
@pytest.mark.parametrize("scale", ["scalar", "vector"])
def test_packed_chain_forms_and_reuse(zp, scale):
    check_packed(*case(260, 520, 200, seed=7, zp=zp, scale=scale), f"zp={zp} scale={scale}", reuse=3)


def test_packed_chain_equals_the_unpacked_call():
    """The same bits as dynamic_quantize_matmul on the unpacked weight, on a
    larger shape with several pair tiles and K chunks."""
    x, Wm, w_scale, w_zp, b = case(1024, 4096, 1536, seed=11, wdt=np.uint8)
    C0, ys0, yz0 = q.dynamic_quantize_matmul(dev(x), dev(Wm), dev(w_scale), dev(w_zp), dev(b))
    pw = q.dynamic_quantize_matmul_pack_weight(dev(Wm))
    C1, ys1, yz1 = q.dynamic_quantize_matmul_packed(dev(x), pw, dev(w_scale), dev(w_zp), dev(b))
    q.check_device_error()
    assert torch.equal(C0, C1) and torch.equal(ys0, ys1) and torch.equal(yz0, yz1)


def test_packed_chain_argument_errors():
    x = torch.zeros((4, 8), device="cuda")
    Wm = torch.zeros((8, 3), dtype=torch.int8, device="cuda")
    pw = q.dynamic_quantize_matmul_pack_weight(Wm)
    short = q.DqmPackedWeight(pw.buf[:256], 8, 3, torch.int8)
    with pytest.raises(q.QmmError):   # packed buffer shorter than the layout
        q.dynamic_quantize_matmul_packed(x, short, torch.ones(1, device="cuda"))
    with pytest.raises(ValueError):   # K differs from the packed weight's
        q.dynamic_quantize_matmul_packed(torch.zeros((4, 16), device="cuda"), pw, torch.ones(1, device="cuda"))
    need = q.dynamic_quantize_matmul_packed_workspace_bytes(4, 8)
    with pytest.raises(q.QmmError):
        q.dynamic_quantize_matmul_packed(x, pw, torch.ones(1, device="cuda"),
                                         workspace=torch.empty(need - 256, dtype=torch.uint8, device="cuda"))
