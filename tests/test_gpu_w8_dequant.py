"""Form (a) through the C ABI: the factored int8-weight matmul against the
oracle's exact value, within 1e-3 * sum_k |a_k * scale*(b_k - zp)| + 1e-6 plus
half an ulp of the output type; and the small-M decode dispatch."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_within, bf16_bits_to_f64, bf16_dev, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")


def check(A_dev, A_vals, B, scale, zp, out, kernel, workspace=None):
    zp_dev = None if zp is None else dev(zp.astype(np.int32))
    C = q.qmm_w8_dequant(A_dev, dev(B), dev(scale), zp_dev, out_dtype=out, workspace=workspace)
    torch.cuda.synchronize()
    assert q.last_kernel() == kernel
    got = host(C)
    gotf = bf16_bits_to_f64(got) if out == torch.bfloat16 else got.astype(np.float64)
    zpv = np.zeros(1, np.int32) if zp is None else zp
    exact = O.w8_dequant(A_vals, B, scale, zpv)
    bound = O.w8_dequant_error_bound(A_vals, B, scale, zpv)
    assert_within(gotf, exact, bound, 7 if out == torch.bfloat16 else 23, kernel)


def test_per_tensor_fp32_workload_shape():
    w = W.w8_dequant_f32_64x256x192()
    check(dev(w.A), w.A, w.B, w.scale, w.zero_point, torch.float32, "w8_dequant_simt")


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (7, 33, 5), (65, 257, 130), (200, 96, 64)])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
def test_simt_shapes(M, K, N, zp):
    rng = np.random.default_rng(M + K + N)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    scale = rng.uniform(0.001, 0.05, N).astype(np.float32)
    z = None if zp is None else (np.array([3], np.int32) if zp == "tensor" else rng.integers(-9, 9, N).astype(np.int32))
    check(dev(A), A, B, scale, z, torch.float32, "w8_dequant_simt")


@pytest.mark.parametrize("M", [1, 2, 4, 5, 16])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_decode_gemv(M, zp, out):
    w = W.decode_gemv(M, K=1024, N=640, seed=M)
    rng = np.random.default_rng(M)
    z = None if zp is None else (np.array([-4], np.int32) if zp == "tensor" else rng.integers(-9, 9, 640).astype(np.int32))
    if M <= 2:
        kernel = "gemv_w8_pair_simt_f32x2"
    else:
        kernel = "gemv_w8_bf16_tma" if zp is None else "gemv_w8_bf16_tma_zp"
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, z, out, kernel)


@pytest.mark.parametrize("M,K,N", [(4, 1024, 200), (4, 1030, 256), (17, 512, 256)])
def test_decode_shapes_outside_gemv_fall_back_to_cuda_cores(M, K, N):
    w = W.decode_gemv(M, K=K, N=N, seed=1)
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, None, torch.bfloat16, "w8_dequant_simt")


def test_gemv_ragged_k_and_scalar_scale():
    w = W.decode_gemv(3, K=1000, N=384, seed=9)
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale[:1].copy(), None, torch.float32, "gemv_w8_bf16_tma")
    w = W.decode_gemv(2, K=1000, N=384, seed=9)
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale[:1].copy(), None, torch.float32, "gemv_w8_pair_simt_f32x2")


SIMT = "gemv_w8_pair_simt_f32x2"
F16 = "gemv_f16_prep+gemv_w8_f16_tma"   # with a workspace: activations pre-scaled to fp16


def bf16_rows(A32):
    """float32 values truncated to bf16: (exact values as float32, u16 bit patterns)."""
    bits = (np.ascontiguousarray(A32, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32), bits


@pytest.mark.parametrize("M", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_decode_gemv_with_workspace(M, zp, out):
    """With a workspace, 3 to 16 rows take the fp16 route; one or two rows keep
    the CUDA-core pair kernel (no workspace needed)."""
    w = W.decode_gemv(M, K=1024, N=640, seed=M + 30)
    rng = np.random.default_rng(M + 30)
    z = None if zp is None else (np.array([5], np.int32) if zp == "tensor" else rng.integers(-9, 9, 640).astype(np.int32))
    kernel = SIMT if M <= 2 else F16 + ("_zp" if zp else "")
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, z, out, kernel, workspace="auto")


@pytest.mark.parametrize("K", [8, 24, 1000, 1032, 4104])
def test_fp16_route_ragged_k(K):
    """K not a multiple of 16 or of the 256-deep stage: the prep's zero padding
    and the copies' zero fill meet at the tail."""
    w = W.decode_gemv(4, K=K, N=272, seed=K)
    z = np.arange(-8, 264, dtype=np.int32)[:272]
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, z, torch.float32, F16 + "_zp", workspace="auto")


def test_fp16_route_row_scales_span_the_bf16_range():
    """Rows whose magnitudes lie far outside fp16's range (2^-60 .. 2^100) and
    an all-zero row: each row's power-of-two scale keeps its values exact."""
    rng = np.random.default_rng(8)
    M, K, N = 7, 512, 256
    e = np.array([-60, -24, -3, 0, 17, 100, 0])[:, None]
    A32 = (W.normal_f32(rng, (M, K)) * np.exp2(e.astype(np.float64))).astype(np.float32)
    A32[6] = 0.0
    A, bits = bf16_rows(A32)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    scale = rng.uniform(0.001, 0.01, N).astype(np.float32)
    check(bf16_dev(bits), A, B, scale, np.array([-2], np.int32), torch.float32, F16 + "_zp", workspace="auto")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_decode_simt_bf16(M, zp, out):
    """One or two activation rows take the CUDA-core weight-streaming kernel (CTA pairs)."""
    w = W.decode_gemv(M, K=1024, N=640, seed=M + 11)
    rng = np.random.default_rng(M)
    z = None if zp is None else (np.array([-4], np.int32) if zp == "tensor" else rng.integers(-9, 9, 640).astype(np.int32))
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, z, out, SIMT, workspace=None)


@pytest.mark.parametrize("M,K,N", [(1, 4, 16), (2, 100, 16), (2, 1000, 4096), (1, 4100, 528), (1, 8192, 1040),
                                   (2, 64, 512), (1, 196, 28672)])
def test_decode_simt_fp32_activations_and_ragged_k(M, K, N):
    rng = np.random.default_rng(K + N)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    scale = rng.uniform(0.001, 0.05, N).astype(np.float32)
    z = rng.integers(-9, 9, N).astype(np.int32)
    check(dev(A), A, B, scale, z, torch.float32, SIMT, workspace="auto")
    check(dev(A), A, B, scale[:1].copy(), None, torch.bfloat16, SIMT, workspace="auto")


@pytest.mark.parametrize("M,workspace,kernel", [(2, None, SIMT), (4, "auto", F16)])
def test_decode_is_deterministic(M, workspace, kernel):
    w = W.decode_gemv(M, K=4096, N=2048, seed=5)
    outs = []
    for _ in range(3):
        C = q.qmm_w8_dequant(bf16_dev(w.A_bits), dev(w.W), dev(w.scale), None, out_dtype=torch.float32,
                             workspace=workspace)
        q.check_device_error()
        assert q.last_kernel() == kernel
        outs.append(host(C))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
