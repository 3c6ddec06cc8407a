"""The five benchmark workloads at full size, through the same entry points and
launch configuration bench.py times, checked against the oracle: in full where
the oracle is cheap (DynamicQuantizeLinear, the small fp32 case), otherwise on
sampled rows or columns the oracle computes one by one."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, assert_within, bf16_bits_to_f64, bf16_dev, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")


def sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, size=k, replace=False))


@pytest.mark.parametrize("workspace,kernel", [("auto", "w8_bf16_prepass+gemm_tc05_pair_w8_bf16"),
                                              (None, "w8_dequant_simt")])
def test_w8_dequant_f32_64x256x192(workspace, kernel):
    w = W.w8_dequant_f32_64x256x192()
    C = q.qmm_w8_dequant(dev(w.A), dev(w.B), dev(w.scale), dev(w.zero_point), out_dtype=torch.float32,
                         workspace=workspace)
    q.check_device_error()
    assert q.last_kernel() == kernel
    exact = O.w8_dequant(w.A, w.B, w.scale, w.zero_point)
    bound = O.w8_dequant_error_bound(w.A, w.B, w.scale, w.zero_point)
    assert_within(host(C).astype(np.float64), exact, bound, 23, "w8 64x256x192")


@pytest.mark.parametrize("workspace,kernel", [("auto", "f16_prepass+gemm_tc05_pair_f16ops_a8w8"),
                                              (None, "gemm_tc05_pair_exact_a8w8")])
def test_a8w8_4096(workspace, kernel):
    w = W.a8w8_4096()
    C = q.qmm_a8w8(dev(w.A), dev(w.B), dev(w.act_scale), dev(w.weight_scale), out_dtype=torch.bfloat16,
                   workspace=workspace)
    q.check_device_error()
    assert q.last_kernel() == kernel
    got = host(C)
    rows = sample(4096, 40, 1)
    want = O.a8w8(w.A[rows], w.B, w.act_scale[rows], w.weight_scale, "bf16")
    assert_equal(got[rows], want, "a8w8 4096^3 sampled rows")


def test_a8w8_acc_decode_M16_8192x28672_b_trans():
    """16 rows on the tensor-core route at the decode size: 1024 sampled
    columns x all rows, bit-exact."""
    w = W.a8w8_acc(16, 8192, 28672, seed=0, b_trans=True)
    acc = torch.empty((16, 28672), dtype=torch.int32, device="cuda")
    C = q.qmm_a8w8_acc(dev(w.A), dev(w.B), dev(w.act_scale), dev(w.weight_scale), acc_in=dev(w.acc_in),
                       acc_out=acc, b_trans=True, out_dtype=torch.bfloat16)
    q.check_device_error()
    assert q.last_kernel() == "gemv_acc_prep+gemv_acc_a8w8_kmajor_tc"
    cols = np.sort(np.random.default_rng(16).choice(28672, 1024, replace=False))
    B = np.ascontiguousarray(w.B[cols].T)   # the sampled columns of the logical [K, N] weight
    want = O.a8w8_dequant_acc(w.acc_in[:, cols], w.A, B, w.act_scale, w.weight_scale[cols], "bf16")
    assert_equal(host(C)[:, cols], want, "decode accumulating A8W8, M = 16, sampled columns")
    want_acc = O.wrap_int32(w.acc_in[:, cols].astype(np.int64) + O.a8w8_acc(w.A, B).astype(np.int64))
    assert_equal(host(acc)[:, cols], want_acc, "decode accumulator, M = 16, sampled columns")


@pytest.mark.parametrize("b_trans", [False, True])
def test_a8w8_acc_decode_M1_8192x28672(b_trans):
    w = W.a8w8_acc(1, 8192, 28672, seed=0, b_trans=b_trans)
    C = q.qmm_a8w8_acc(dev(w.A), dev(w.B), dev(w.act_scale), dev(w.weight_scale), acc_in=dev(w.acc_in),
                       b_trans=b_trans, out_dtype=torch.bfloat16)
    q.check_device_error()
    assert q.last_kernel() == ("gemv_acc_a8w8_kmajor" if b_trans else "gemv_acc_a8w8_nmajor")
    B = np.ascontiguousarray(w.B.T) if b_trans else w.B
    want = O.a8w8_dequant_acc(w.acc_in, w.A, B, w.act_scale, w.weight_scale, "bf16")
    assert_equal(host(C), want, "decode accumulating A8W8, M = 1")


@pytest.mark.parametrize("packed", [False, True])
def test_dynamic_quantize_matmul_8192x4096x11008(packed):
    w = W.dql_matmul_integer_8192x4096x11008()
    rng = np.random.default_rng(9)
    w_scale = rng.uniform(0.001, 0.01, 11008).astype(np.float32)
    bias = rng.standard_normal(11008).astype(np.float32)
    if packed:   # the weight converted once, then the chain on it
        pw = q.dynamic_quantize_matmul_pack_weight(dev(w.B))
        C, ys, yz = q.dynamic_quantize_matmul_packed(dev(w.x), pw, dev(w_scale), dev(w.b_zp), dev(bias))
    else:
        C, ys, yz = q.dynamic_quantize_matmul(dev(w.x), dev(w.B), dev(w_scale), dev(w.b_zp), dev(bias))
    q.check_device_error()
    assert q.last_kernel() == ("dql_f16+gemm_tc05_pair_f16ops_matmul_integer_dequant"
                               + ("_packed" if packed else ""))
    rows = sample(8192, 24, 5)
    rows[:2] = [0, 8191]
    want, wys, wyz = O.dynamic_quantize_matmul(w.x, w.B, w_scale, w.b_zp, bias, rows=rows)
    assert float(ys.item()) == float(wys) and int(yz.item()) == int(wyz)
    assert_equal(host(C)[rows], want, "fused chain 8192x4096x11008, sampled rows")


@pytest.mark.parametrize("case", ["conv2d_3x3_8x256x56x56", "conv1d_k3_4x512x3000"])
def test_conv_integer_full_size(case):
    c = getattr(W, case)()
    y = q.conv_integer(dev(c.x), dev(c.w), dev(c.x_zp), dev(c.w_zp), pads=c.pads, strides=c.strides,
                       dilations=c.dilations, group=c.group)
    q.check_device_error()
    assert q.last_kernel() == "conv_f16_nhwc+gemm_tc05_pair_f16ops_conv_im2col"
    got = host(y)
    imgs = sample(c.x.shape[0], 2, 3)
    chans = sample(c.w.shape[0], 12, 4)
    chans[:2] = [0, c.w.shape[0] - 1]
    want = O.conv_integer(c.x[imgs], c.w[chans], c.x_zp, c.w_zp[chans], c.pads, c.strides, c.dilations, c.group)
    assert_equal(got[imgs][:, chans], want, f"{case}: sampled images and channels")


@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (True, True)])
def test_a8w8_acc_4096(a_trans, b_trans):
    w = W.a8w8_acc(4096, 4096, 4096, seed=0, a_trans=a_trans, b_trans=b_trans)
    acc = torch.empty((4096, 4096), dtype=torch.int32, device="cuda")
    C = q.qmm_a8w8_acc(dev(w.A), dev(w.B), dev(w.act_scale), dev(w.weight_scale), acc_in=dev(w.acc_in), acc_out=acc,
                       a_trans=a_trans, b_trans=b_trans, out_dtype=torch.bfloat16)
    q.check_device_error()
    assert q.last_kernel() == "f16_prepass+gemm_tc05_pair_f16ops_a8w8_acc"
    A = w.A.T if a_trans else w.A
    B = np.ascontiguousarray(w.B.T) if b_trans else w.B
    rows = sample(4096, 32, 2)
    A_r = np.ascontiguousarray(A[rows])
    want = O.a8w8_dequant_acc(w.acc_in[rows], A_r, B, w.act_scale[rows], w.weight_scale, "bf16")
    assert_equal(host(C)[rows], want, "a8w8_acc 4096^3 sampled rows")
    want_acc = O.wrap_int32(w.acc_in[rows].astype(np.int64) + O.a8w8_acc(A_r, B).astype(np.int64))
    assert_equal(host(acc)[rows], want_acc, "a8w8_acc 4096^3 accumulator, sampled rows")


@pytest.mark.parametrize("workspace,kernel", [("auto", "f16_prepass+gemm_tc05_pair_f16ops_matmul_integer"),
                                              (None, "gemm_tc05_pair_exact_matmul_integer")])
def test_dql_then_matmul_integer_8192x4096x11008(workspace, kernel):
    w = W.dql_matmul_integer_8192x4096x11008()
    y, s, zp, rs = q.dynamic_quantize_linear(dev(w.x), row_len=4096)
    assert q.last_kernel() == "dql_minmax+dql_quantize_rows"
    wy, ws, wzp = O.dynamic_quantize_linear(w.x)
    assert float(s.item()) == float(ws) and int(zp.item()) == int(wzp)
    assert_equal(host(y), wy, "DQL 8192x4096")
    assert_equal(host(rs), O.row_sums(wy, 4096), "DQL row sums")
    # the zero point stays on the device between the two calls
    C = q.matmul_integer(y, dev(w.B), a_zero_point=zp, b_zero_point=dev(w.b_zp), workspace=workspace)
    q.check_device_error()
    assert q.last_kernel() == kernel
    rows = sample(8192, 16, 2)
    want = O.matmul_integer(wy[rows], w.B, int(wzp), w.b_zp)
    assert_equal(host(C)[rows], want, "MatMulInteger 8192x4096x11008 sampled rows")


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("workspace", ["auto", None])
def test_decode_gemv_8192x28672(M, workspace):
    w = W.decode_gemv(M)
    C = q.qmm_w8_dequant(bf16_dev(w.A_bits), dev(w.W), dev(w.scale), None, out_dtype=torch.bfloat16,
                         workspace=workspace)
    q.check_device_error()
    if workspace == "auto" and M > 2:
        assert q.last_kernel() == "gemv_f16_prep+gemv_w8_f16_tma"
    else:
        assert q.last_kernel() == ("gemv_w8_pair_simt_f32x2" if M <= 2 else "gemv_w8_bf16_tma")
    got = bf16_bits_to_f64(host(C))
    cols = sample(28672, 1024, 3)
    zp0 = np.zeros(1, np.int32)
    Wc = np.ascontiguousarray(w.W[:, cols])
    exact = O.w8_dequant(w.A, Wc, w.scale[cols], zp0)
    bound = O.w8_dequant_error_bound(w.A, Wc, w.scale[cols], zp0)
    assert_within(got[:, cols], exact, bound, 7, f"GEMV M={M}")


def test_batched_matmul_integer_shared_b():
    w = W.batched_matmul_integer()
    C = q.matmul_integer(dev(w.A), dev(w.B), a_zero_point=dev(np.array([w.a_zp], np.int8)),
                         b_zero_point=dev(np.array([w.b_zp], np.int8)))
    q.check_device_error()
    assert q.last_kernel() == "f16_prepass+gemm_tc05_pair_f16ops_matmul_integer"
    assert C.shape == (8, 16, 512, 1024)
    got = host(C).reshape(-1, 1024)
    rows = sample(8 * 16 * 512, 48, 4)
    want = O.matmul_integer(w.A.reshape(-1, 1024)[rows], w.B, w.a_zp, w.b_zp)
    assert_equal(got[rows], want, "batched MatMulInteger sampled rows")
