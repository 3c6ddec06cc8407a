"""Form (a) for large M on the tensor cores (bf16 copy of the int8 weight in a
workspace, SM-pair GEMM with one fp32 accumulation, scale/zero-point epilogue)
against the oracle's exact value, within 1e-3 * sum_k |a_k * scale*(b_k - zp)|
+ 1e-6 plus half an ulp of the output type; bf16 and fp32 activations (the
latter split into two bf16 parts along a doubled K)."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_within, bf16_bits_to_f64, bf16_dev, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")
PREFILL = "w8_bf16_prepass+gemm_tc05_pair_w8_bf16"


def check(A_dev, A_vals, B, scale, zp, out, kernel=PREFILL, workspace="auto"):
    zp_dev = None if zp is None else dev(zp.astype(np.int32))
    C = q.qmm_w8_dequant(A_dev, dev(B), dev(scale), zp_dev, out_dtype=out, workspace=workspace)
    q.check_device_error()
    assert q.last_kernel() == kernel
    got = host(C)
    gotf = bf16_bits_to_f64(got) if out == torch.bfloat16 else got.astype(np.float64)
    zpv = np.zeros(1, np.int32) if zp is None else zp
    exact = O.w8_dequant(A_vals, B, scale, zpv)
    bound = O.w8_dequant_error_bound(A_vals, B, scale, zpv)
    assert_within(gotf, exact, bound, 7 if out == torch.bfloat16 else 23, kernel)


def zero_point(kind, N, rng):
    if kind is None:
        return None
    return np.array([-4], np.int32) if kind == "tensor" else rng.integers(-9, 9, N).astype(np.int32)


@pytest.mark.parametrize("M,K,N", [(64, 1024, 640), (100, 512, 256), (300, 4096, 528), (1000, 1040, 1008)])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_bf16_activations(M, K, N, zp, out):
    w = W.decode_gemv(M, K=K, N=N, seed=M + N)
    rng = np.random.default_rng(M)
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, zero_point(zp, N, rng), out)


@pytest.mark.parametrize("M,K,N", [(64, 256, 192), (256, 1008, 272), (300, 2048, 400)])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
def test_fp32_activations_split_into_two_bf16_parts(M, K, N, zp):
    rng = np.random.default_rng(M + K)
    A = W.normal_f32(rng, (M, K))
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    scale = rng.uniform(0.001, 0.05, N).astype(np.float32)
    check(dev(A), A, B, scale, zero_point(zp, N, rng), torch.float32)


def test_scalar_scale_and_wide_dynamic_range():
    rng = np.random.default_rng(5)
    M, K, N = 128, 512, 256
    A = (W.normal_f32(rng, (M, K)) * np.exp2(rng.integers(-20, 20, (M, 1)))).astype(np.float32)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    check(dev(A), A, B, np.array([0.02], np.float32), np.array([3], np.int32), torch.float32)


@pytest.mark.parametrize("M,K,N,kernel", [(63, 256, 256, "w8_dequant_simt"), (128, 40, 256, "w8_dequant_simt"),
                                          (16, 1024, 640, "gemv_f16_prep+gemv_w8_f16_tma")])
def test_shapes_outside_the_prefill_path(M, K, N, kernel):
    w = W.decode_gemv(M, K=K, N=N, seed=3)
    assert q.qmm_w8_dequant_workspace_bytes(torch.bfloat16, M, K, N) == 0 or M <= 16
    check(bf16_dev(w.A_bits), w.A, w.W, w.scale, None, torch.bfloat16, kernel=kernel)
