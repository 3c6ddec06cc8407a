"""A8W8 (form (b)) through the C ABI against the oracle, on small, ragged and
adversarial shapes. The GPU epilogue performs the same float32 steps in the
same order as the oracle, so outputs must match bit for bit; they must also lie
within the stated tolerance of the exact (float64) value."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, assert_within, bf16_bits_to_f64, dev, gemm_kernel, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

SHAPES = [(1, 16, 16), (3, 31, 7), (128, 64, 256), (129, 258, 200), (17, 1040, 300), (256, 4096, 512),
          (300, 2048, 272), (64, 128, 64)]


def run(A, B, a_s, w_s, out):
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = q.qmm_a8w8(dev(A), dev(B), dev(a_s), dev(w_s), out_dtype=dt, workspace=None)
    q.check_device_error()
    return host(C)


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_a8w8_matches_oracle(M, K, N, out):
    w = W.a8w8(M, K, N, seed=M * 7 + K * 3 + N)
    got = run(w.A, w.B, w.act_scale, w.weight_scale, out)
    assert q.last_kernel() == gemm_kernel("a8w8", M, K, N)
    want = O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, out)
    assert_equal(got, want, f"a8w8 {out} {M}x{K}x{N}")
    exact = O.a8w8_exact(w.A, w.B, w.act_scale, w.weight_scale)
    bound = O.a8w8_error_bound(w.A, w.B, w.act_scale, w.weight_scale)
    gotf = bf16_bits_to_f64(got) if out == "bf16" else got
    assert_within(gotf, exact, bound, 7 if out == "bf16" else 23, "a8w8 vs exact")


def test_a8w8_scalar_scales():
    w = W.a8w8(70, 96, 48, seed=3)
    a_s = np.array([0.0125], np.float32)
    w_s = np.array([0.003], np.float32)
    got = run(w.A, w.B, a_s, w_s, "f32")
    assert_equal(got, O.a8w8(w.A, w.B, a_s, w_s, "f32"), "scalar scales")


def test_a8w8_scale_orientation_square():
    """[M] scales rows and [N] scales columns even when M == N."""
    M = 256
    A = np.eye(M, dtype=np.int8)
    B = np.ones((M, M), np.int8)
    a_s = (np.arange(M, dtype=np.float32) + 1.0)
    w_s = np.float32(1.0) / (np.arange(M, dtype=np.float32) + 2.0)
    got = run(A, B, a_s, w_s.astype(np.float32), "f32")
    want = O.a8w8(A, B, a_s, w_s.astype(np.float32), "f32")
    assert_equal(got, want, "orientation")
    assert got[5, 0] == np.float32(np.float32(6.0) * w_s[0])


@pytest.mark.parametrize("pattern", ["all_min", "max_times_min", "alternating", "extremes_random"])
def test_a8w8_exact_at_chunk_edge(pattern):
    """Patterns whose K-chunk sums reach the 2^24 limit of exact fp32 accumulation."""
    M, K, N = 130, 4096, 272
    rng = np.random.default_rng(11)
    if pattern == "all_min":
        A = np.full((M, K), -128, np.int8)
        B = np.full((K, N), -128, np.int8)
    elif pattern == "max_times_min":
        A = np.full((M, K), 127, np.int8)
        B = np.full((K, N), -128, np.int8)
    elif pattern == "alternating":
        s = np.where(np.arange(K) % 2 == 0, 1, -1).astype(np.int16)
        A = np.tile((s * 127).astype(np.int8), (M, 1))
        B = np.tile((s * -128).astype(np.int8)[:, None], (1, N))
    else:
        A = rng.choice(np.array([-128, 127, -127, 126], np.int8), size=(M, K))
        B = rng.choice(np.array([-128, 127], np.int8), size=(K, N))
    a_s = np.ones(M, np.float32)
    w_s = np.ones(N, np.float32)
    got = run(A, B, a_s, w_s, "f32")
    assert_equal(got, O.a8w8(A, B, a_s, w_s, "f32"), pattern)


def test_a8w8_k_zero_gives_zeros():
    A = torch.empty((5, 0), dtype=torch.int8, device="cuda")
    B = torch.empty((0, 9), dtype=torch.int8, device="cuda")
    C = q.qmm_a8w8(A, B, torch.ones(5, device="cuda"), torch.ones(9, device="cuda"), out_dtype=torch.float32)
    assert q.last_kernel() == "memset_zero"
    assert torch.count_nonzero(C).item() == 0


def test_a8w8_more_chunks_than_default(monkeypatch):
    """A shorter chunk (more exact drains per tile) must give the same bits."""
    monkeypatch.setenv("QMM_CHUNK_K", "64")
    w = W.a8w8(200, 1000, 300, seed=5)
    got = run(w.A, w.B, w.act_scale, w.weight_scale, "bf16")
    assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), "chunk 64")
