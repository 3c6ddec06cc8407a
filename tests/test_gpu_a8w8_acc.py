"""The accumulating A8W8 (int32 accumulator input, a_trans / b_trans) against
the oracle, bit for bit: every layout of the operands on ragged shapes (M = 1
decode rows, K and N that are not multiples of 8 or 16, unaligned operand
pointers), int32 wrap-around of the accumulator, the raw accumulator output,
K-split chaining through acc_in / acc_out, in-place accumulation, the empty K,
scalar scales and argument errors."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

KERNEL = "f16_prepass+gemm_tc05_pair_f16ops_a8w8_acc"


def expected_kernel(M, K, N, b_trans):
    """Decode shapes (M <= 16) whose rows suit the weight-streaming kernels
    take them: with B stored [N,K], up to 3 rows on dp4a, 4..16 rows on the
    tensor cores."""
    if 1 <= M <= 16 and (K % 16 == 0 if b_trans else (K % 4 == 0 and N % 4 == 0)):
        if b_trans:
            return "gemv_acc_a8w8_kmajor" if M < 4 else "gemv_acc_prep+gemv_acc_a8w8_kmajor_tc"
        return "gemv_acc_a8w8_nmajor"
    return KERNEL


def logical(w):
    A = w.A.T if w.a_trans else w.A
    B = w.B.T if w.b_trans else w.B
    return np.ascontiguousarray(A), np.ascontiguousarray(B)


def want_acc(acc_in, A, B):
    return O.wrap_int32(acc_in.astype(np.int64) + O.a8w8_acc(A, B).astype(np.int64))


def run(w, out="f32", with_acc_in=True, with_acc_out=True, a=None, b=None):
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, None: None}[out]
    M, N = w.acc_in.shape
    acc_out = torch.empty((M, N), dtype=torch.int32, device="cuda") if with_acc_out else None
    C = q.qmm_a8w8_acc(dev(w.A) if a is None else a, dev(w.B) if b is None else b, dev(w.act_scale),
                       dev(w.weight_scale), acc_in=dev(w.acc_in) if with_acc_in else None, acc_out=acc_out,
                       a_trans=w.a_trans, b_trans=w.b_trans, out_dtype=dt)
    q.check_device_error()
    return (None if C is None else host(C)), (None if acc_out is None else host(acc_out))


SHAPES = [(1, 64, 256), (7, 33, 5), (300, 1040, 272), (257, 100, 129), (512, 4096, 1008), (130, 4104, 40),
          (640, 2064, 144)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (True, False), (False, True), (True, True)])
def test_acc_matches_oracle(M, K, N, a_trans, b_trans):
    w = W.a8w8_acc(M, K, N, seed=M + 3 * K + 5 * N, a_trans=a_trans, b_trans=b_trans)
    A, B = logical(w)
    for out in ("f32", "bf16"):
        C, acc = run(w, out)
        assert q.last_kernel() == expected_kernel(M, K, N, b_trans)
        tag = f"{M}x{K}x{N} a_trans={a_trans} b_trans={b_trans} {out}"
        assert_equal(C, O.a8w8_dequant_acc(w.acc_in, A, B, w.act_scale, w.weight_scale, out), tag)
        assert_equal(acc, want_acc(w.acc_in, A, B), "acc_out " + tag)


@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (True, True)])
def test_acc_wraps_modulo_2_32(a_trans, b_trans):
    """Accumulators spread over all of int32 plus products near the largest
    magnitude: many sums leave the int32 range and wrap."""
    M, K, N = 300, 4096, 272
    w = W.a8w8_acc(M, K, N, seed=9, a_trans=a_trans, b_trans=b_trans, acc_bound=2**31)
    w.A[...] = -128
    w.B[...] = np.where(np.arange(N) % 2 == 0, -128, 127)[None, :] if not b_trans else \
        np.where(np.arange(N) % 2 == 0, -128, 127)[:, None]
    A, B = logical(w)
    C, acc = run(w, "f32")
    want = want_acc(w.acc_in, A, B)
    wide = w.acc_in.astype(np.int64) + O.a8w8_acc(A, B).astype(np.int64)
    assert (wide != want).any(), "the case must wrap"
    assert_equal(acc, want, "wrapped accumulator")
    assert_equal(C, O.a8w8_dequant_acc(w.acc_in, A, B, w.act_scale, w.weight_scale, "f32"), "wrapped, scaled")


def test_acc_without_acc_in_is_a8w8():
    w = W.a8w8_acc(300, 1040, 272, seed=4)
    C, acc = run(w, "bf16", with_acc_in=False)
    assert_equal(C, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), "acc_in absent")
    assert_equal(acc, O.a8w8_acc(w.A, w.B), "acc_out without acc_in")


@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (True, False), (False, True)])
def test_k_split_chains_through_the_accumulator(a_trans, b_trans):
    """Part of K into acc_out only (no C), the rest with acc_in: the same
    accumulator and output as one call over the whole K, and as the oracle."""
    M, K, N, k1 = 384, 3000, 400, 1216
    w = W.a8w8_acc(M, K, N, seed=12)
    A, B = w.A, w.B
    part = lambda x, lo, hi, axis: np.ascontiguousarray(np.take(x, np.arange(lo, hi), axis=axis))
    A1, A2 = part(A, 0, k1, 1), part(A, k1, K, 1)
    B1, B2 = part(B, 0, k1, 0), part(B, k1, K, 0)
    store_a = (lambda x: np.ascontiguousarray(x.T)) if a_trans else (lambda x: x)
    store_b = (lambda x: np.ascontiguousarray(x.T)) if b_trans else (lambda x: x)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    assert q.qmm_a8w8_acc(dev(store_a(A1)), dev(store_b(B1)), acc_out=acc, a_trans=a_trans, b_trans=b_trans,
                          out_dtype=None) is None
    C = q.qmm_a8w8_acc(dev(store_a(A2)), dev(store_b(B2)), dev(w.act_scale), dev(w.weight_scale), acc_in=acc,
                       acc_out=acc, a_trans=a_trans, b_trans=b_trans, out_dtype=torch.float32)   # in place
    q.check_device_error()
    assert_equal(host(acc), O.a8w8_acc(A, B), "chained accumulator")
    assert_equal(host(C), O.a8w8(A, B, w.act_scale, w.weight_scale, "f32"), "chained output")


def test_empty_k_passes_the_accumulator_through():
    M, N = 70, 90
    w = W.a8w8_acc(M, 16, N, seed=2)
    A = torch.empty((M, 0), dtype=torch.int8, device="cuda")
    B = torch.empty((0, N), dtype=torch.int8, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C = q.qmm_a8w8_acc(A, B, dev(w.act_scale), dev(w.weight_scale), acc_in=dev(w.acc_in), acc_out=acc,
                       out_dtype=torch.float32)
    q.check_device_error()
    assert q.last_kernel() == "acc_passthrough"
    assert_equal(host(acc), w.acc_in, "K = 0 accumulator")
    empty = np.zeros((M, 0), np.int8), np.zeros((0, N), np.int8)
    assert_equal(host(C), O.a8w8_dequant_acc(w.acc_in, *empty, w.act_scale, w.weight_scale, "f32"), "K = 0 output")


def test_scalar_scales_and_unaligned_operands():
    M, K, N = 260, 203, 77
    w = W.a8w8_acc(M, K, N, seed=6, b_trans=True)
    A, B = logical(w)
    # operands one byte past a 16-byte boundary
    bufa = torch.empty(M * K + 1, dtype=torch.int8, device="cuda")
    bufb = torch.empty(N * K + 1, dtype=torch.int8, device="cuda")
    a = bufa[1:].view(M, K)
    b = bufb[1:].view(N, K)
    a.copy_(dev(w.A))
    b.copy_(dev(w.B))
    s_a, s_w = np.array([0.0125], np.float32), np.array([0.003], np.float32)
    C = q.qmm_a8w8_acc(a, b, dev(s_a), dev(s_w), acc_in=dev(w.acc_in), b_trans=True, out_dtype=torch.bfloat16)
    q.check_device_error()
    assert_equal(host(C), O.a8w8_dequant_acc(w.acc_in, A, B, s_a, s_w, "bf16"), "scalar scales, unaligned")


def test_argument_errors():
    A = torch.zeros((4, 8), dtype=torch.int8, device="cuda")
    B = torch.zeros((8, 4), dtype=torch.int8, device="cuda")
    with pytest.raises(ValueError):
        q.qmm_a8w8_acc(A, B, out_dtype=None)               # nothing to write
    with pytest.raises(ValueError):
        q.qmm_a8w8_acc(A, B.T.contiguous(), torch.ones(1, device="cuda"), torch.ones(1, device="cuda"),
                       b_trans=False)                     # inner dimensions differ
    need = q.qmm_a8w8_acc_workspace_bytes(4, 8, 4)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        q.qmm_a8w8_acc(A, B, torch.ones(1, device="cuda"), torch.ones(1, device="cuda"), workspace=small)


DECODE = [(1, 64, 256), (1, 4096, 1000), (2, 1040, 132), (5, 2048, 4), (8, 512, 520), (16, 1024, 264),
          (1, 8192, 4100), (9, 3088, 72), (16, 16, 100), (12, 4096, 2048)]


@pytest.mark.parametrize("M,K,N", DECODE)
@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (True, False), (False, True), (True, True)])
def test_decode_shapes_match_oracle(M, K, N, a_trans, b_trans):
    w = W.a8w8_acc(M, K, N, seed=7 * M + K + N, a_trans=a_trans, b_trans=b_trans)
    A, B = logical(w)
    C, acc = run(w, "bf16")
    assert q.last_kernel() == expected_kernel(M, K, N, b_trans)
    tag = f"decode {M}x{K}x{N} a_trans={a_trans} b_trans={b_trans}"
    assert_equal(acc, want_acc(w.acc_in, A, B), "acc_out " + tag)
    assert_equal(C, O.a8w8_dequant_acc(w.acc_in, A, B, w.act_scale, w.weight_scale, "bf16"), tag)


@pytest.mark.parametrize("b_trans", [False, True])
def test_decode_wraps_and_optional_operands(b_trans):
    """Extremes and int32-spanning accumulators (sums wrap); no acc_in; acc_out only."""
    M, K, N = 3, 8192, 512
    w = W.a8w8_acc(M, K, N, seed=4, b_trans=b_trans, acc_bound=2**31)
    w.A[...] = -128
    w.B[...] = -128
    A, B = logical(w)
    C, acc = run(w, "f32")
    assert q.last_kernel() == expected_kernel(M, K, N, b_trans)
    wide = w.acc_in.astype(np.int64) + O.a8w8_acc(A, B).astype(np.int64)
    assert (wide != want_acc(w.acc_in, A, B)).any(), "the case must wrap"
    assert_equal(acc, want_acc(w.acc_in, A, B), "wrapped decode accumulator")
    assert_equal(C, O.a8w8_dequant_acc(w.acc_in, A, B, w.act_scale, w.weight_scale, "f32"), "wrapped decode")
    C2, acc2 = run(w, "f32", with_acc_in=False)
    assert_equal(acc2, O.a8w8_acc(A, B), "decode without acc_in")
    acc3 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    assert q.qmm_a8w8_acc(dev(w.A), dev(w.B), acc_in=dev(w.acc_in), acc_out=acc3, b_trans=b_trans,
                          out_dtype=None) is None
    q.check_device_error()
    assert_equal(host(acc3), want_acc(w.acc_in, A, B), "decode, acc_out only")


@pytest.mark.parametrize("M", [4, 8, 16])
def test_decode_tensor_core_route_at_the_exactness_edge(M):
    """Every product -128 * -128 = 2^14, so each 1024-k fp32 partial sum of the
    tensor-core route is exactly 2^24; a mixed-sign half keeps the partials
    near the edge with both signs. Bit-exact against the oracle."""
    K, N = 4096, 256
    w = W.a8w8_acc(M, K, N, seed=M, b_trans=True, acc_bound=2**31)
    w.A[...] = -128
    w.B[...] = -128
    w.B[N // 2:, ::2] = 127   # columns of B stored [N,K]: alternate signs along k in the upper half
    A, B = logical(w)
    C, acc = run(w, "f32")
    assert q.last_kernel() == "gemv_acc_prep+gemv_acc_a8w8_kmajor_tc"
    assert_equal(acc, want_acc(w.acc_in, A, B), f"tensor-core decode accumulator M={M}")
    assert_equal(C, O.a8w8_dequant_acc(w.acc_in, A, B, w.act_scale, w.weight_scale, "f32"), f"M={M}")
