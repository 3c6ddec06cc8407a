"""The decode routes captured into CUDA graphs: a decode loop replays one
captured call per layer, so each route must capture (the packed GEMV's
cluster launch with or without its prep kernel as a programmatic dependent,
the tensor-core accumulating decode behind its prep, the packed fused chain)
and replay exactly with new inputs written into the same buffers."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, assert_within, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")


def capture(call):
    """One warm-up call on a side stream (first-use set-up happens there),
    then the call captured into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    q.check_device_error()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        call()
    return g


@pytest.mark.parametrize("M,K,kernel", [(1, 2048, "gemv_w8_packed_rows_in_cta"),
                                        (4, 4608, "gemv_prep_rows+gemv_w8_packed")])
def test_captured_packed_decode_replays_with_new_activations(M, K, kernel):
    N = 1024
    w0 = W.decode_gemv(M, K=K, N=N, seed=70)
    packed = q.qmm_w8_pack_decode_weight(dev(w0.W))
    A = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    A.copy_(torch.from_numpy(w0.A_bits.view(np.int16)).view(torch.bfloat16))
    scale = dev(w0.scale)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(q.qmm_w8_dequant_packed_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    g = capture(lambda: q.qmm_w8_dequant_packed(A, packed, N, scale, out=out, workspace=ws))
    assert q.last_kernel() == kernel
    for seed in (71, 72):
        wn = W.decode_gemv(M, K=K, N=N, seed=seed)
        A.copy_(torch.from_numpy(wn.A_bits.view(np.int16)).view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        q.check_device_error()
        zp0 = np.zeros(1, np.int32)
        exact = O.w8_dequant(wn.A, w0.W, w0.scale, zp0)
        bound = O.w8_dequant_error_bound(wn.A, w0.W, w0.scale, zp0)
        assert_within(host(out).astype(np.float64), exact, bound, 23, f"graph replay {kernel} seed {seed}")


def test_captured_tensor_core_accumulating_decode_replays_exactly():
    M, K, N = 8, 2048, 512
    w0 = W.a8w8_acc(M, K, N, seed=80, b_trans=True)
    A, B, acc = dev(w0.A), dev(w0.B), dev(w0.acc_in)
    a_s, w_s = dev(w0.act_scale), dev(w0.weight_scale)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    acc_out = torch.empty((M, N), dtype=torch.int32, device="cuda")
    ws = torch.empty(q.qmm_a8w8_acc_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
    g = capture(lambda: q.qmm_a8w8_acc(A, B, a_s, w_s, acc_in=acc, acc_out=acc_out, b_trans=True, out=out,
                                       workspace=ws))
    assert q.last_kernel() == "gemv_acc_prep+gemv_acc_a8w8_kmajor_tc"
    Bl = np.ascontiguousarray(w0.B.T)
    for seed in (81, 82):
        wn = W.a8w8_acc(M, K, N, seed=seed, b_trans=True)
        A.copy_(dev(wn.A))
        acc.copy_(dev(wn.acc_in))
        g.replay()
        torch.cuda.synchronize()
        q.check_device_error()
        want_acc = O.wrap_int32(wn.acc_in.astype(np.int64) + O.a8w8_acc(wn.A, Bl).astype(np.int64))
        assert_equal(host(acc_out), want_acc, f"graph replay accumulator seed {seed}")
        assert_equal(host(out), O.a8w8_dequant_acc(wn.acc_in, wn.A, Bl, w0.act_scale, w0.weight_scale, "f32"),
                     f"graph replay seed {seed}")


def test_captured_packed_chain_replays_exactly():
    rng = np.random.default_rng(90)
    M, K, N = 300, 512, 256
    Wm = rng.integers(-128, 128, (K, N)).astype(np.int8)
    w_scale = rng.uniform(0.001, 0.01, N).astype(np.float32)
    w_zp = rng.integers(-128, 128, N).astype(np.int8)
    pw = q.dynamic_quantize_matmul_pack_weight(dev(Wm))
    x = dev(W.normal_f32(rng, (M, K)))
    ws_d, zp_d = dev(w_scale), dev(w_zp)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(q.dynamic_quantize_matmul_packed_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    res = {}

    def call():
        res["C"], res["ys"], res["yz"] = q.dynamic_quantize_matmul_packed(x, pw, ws_d, zp_d, out=out, workspace=ws)
    g = capture(call)
    assert q.last_kernel() == "dql_f16+gemm_tc05_pair_f16ops_matmul_integer_dequant_packed"
    for seed in (91, 92):
        xn = W.with_outliers(np.random.default_rng(seed), W.normal_f32(np.random.default_rng(seed), (M, K)),
                             0.001, 20.0)
        x.copy_(dev(xn))
        g.replay()
        torch.cuda.synchronize()
        q.check_device_error()
        want, wys, wyz = O.dynamic_quantize_matmul(xn, Wm, w_scale, w_zp, None)
        assert float(res["ys"].item()) == float(wys) and int(res["yz"].item()) == int(wyz)
        assert_equal(host(out), want, f"graph replay of the packed chain seed {seed}")
