"""The exact GEMM on SM pairs (M >= 256, 16-byte-aligned rows) against the
oracle: A8W8 bit for bit, MatMulInteger bit for bit, on the shapes where the
pair kernel differs from the single-SM one -- pair tiles whose odd CTA holds
no valid row or no valid column, K tails, the 2^24 chunk edge, many tiles per
pair (the column-sum exchange ring wraps), short forced chunks, batches and
int32 wrap-around."""
import numpy as np
import pytest

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

INFO = {"s8": (np.int8, -128, 127), "u8": (np.uint8, 0, 255)}
PAIR_A8W8 = "gemm_tc05_pair_exact_a8w8"
PAIR_MMI = "gemm_tc05_pair_exact_matmul_integer"


def rand(rng, dt, shape):
    t, lo, hi = INFO[dt]
    return rng.integers(lo, hi + 1, size=shape).astype(t)


def a8w8(A, B, a_s, w_s, out="f32"):
    import torch
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = q.qmm_a8w8(dev(A), dev(B), dev(a_s), dev(w_s), out_dtype=dt, workspace=None)
    q.check_device_error()
    return host(C)


def mmi(A, B, a_zp=None, b_zp=None):
    C = q.matmul_integer(dev(A), dev(B), None if a_zp is None else dev(a_zp), None if b_zp is None else dev(b_zp),
                         workspace=None)
    q.check_device_error()
    return host(C)


# (M, K, N): M % 256 in (0, 128] leaves the odd CTA of the last row tile without
# a valid row; N % 256 in (0, 128] leaves its B half without a valid column.
PAIR_SHAPES = [(256, 64, 256), (257, 128, 272), (384, 320, 400), (300, 4096, 528), (1000, 1040, 1008),
               (512, 16, 128), (640, 2064, 144)]


@pytest.mark.parametrize("M,K,N", PAIR_SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_pair_a8w8_matches_oracle(M, K, N, out):
    w = W.a8w8(M, K, N, seed=M + 3 * K + 7 * N)
    got = a8w8(w.A, w.B, w.act_scale, w.weight_scale, out)
    assert q.last_kernel() == PAIR_A8W8
    assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, out), f"pair a8w8 {out} {M}x{K}x{N}")


@pytest.mark.parametrize("adt,bdt", [("s8", "s8"), ("u8", "s8"), ("s8", "u8"), ("u8", "u8")])
@pytest.mark.parametrize("zp", ["none", "scalar", "vector", "a_only", "b_only"])
@pytest.mark.parametrize("M,K,N", [(260, 1040, 272), (513, 272, 400)])
def test_pair_matmul_integer_matches_oracle(adt, bdt, zp, M, K, N):
    rng = np.random.default_rng(M + K + N + len(zp) + 7 * len(adt + bdt))
    A, B = rand(rng, adt, (M, K)), rand(rng, bdt, (K, N))
    a_zp = b_zp = None
    if zp == "scalar":
        a_zp, b_zp = rand(rng, adt, (1,)), rand(rng, bdt, (1,))
    elif zp == "vector":
        a_zp, b_zp = rand(rng, adt, (M,)), rand(rng, bdt, (N,))
    elif zp == "a_only":
        a_zp = rand(rng, adt, (1,))
    elif zp == "b_only":
        b_zp = rand(rng, bdt, (N,))
    got = mmi(A, B, a_zp, b_zp)
    assert q.last_kernel() == PAIR_MMI
    want = O.matmul_integer(A, B, 0 if a_zp is None else a_zp, 0 if b_zp is None else b_zp)
    assert_equal(got, want, f"pair {adt}x{bdt} zp={zp} {M}x{K}x{N}")


@pytest.mark.parametrize("adt,bdt,a,b", [("s8", "s8", -128, -128), ("u8", "s8", 255, -128), ("u8", "u8", 255, 255),
                                         ("s8", "u8", -128, 255)])
def test_pair_exact_at_chunk_edge(adt, bdt, a, b):
    """Every K-chunk sum sits at the largest magnitude the fp32 accumulator holds exactly."""
    M, K, N = 260, 4096, 272
    A = np.full((M, K), a, INFO[adt][0])
    B = np.full((K, N), b, INFO[bdt][0])
    got = mmi(A, B)
    assert q.last_kernel() == PAIR_MMI
    assert (got == np.int64(a) * b * K).all()


def test_pair_a8w8_extremes_at_chunk_edge():
    rng = np.random.default_rng(11)
    M, K, N = 300, 4096, 272
    A = rng.choice(np.array([-128, 127, -127, 126], np.int8), size=(M, K))
    B = rng.choice(np.array([-128, 127], np.int8), size=(K, N))
    ones_m, ones_n = np.ones(M, np.float32), np.ones(N, np.float32)
    assert_equal(a8w8(A, B, ones_m, ones_n), O.a8w8(A, B, ones_m, ones_n, "f32"), "extremes")


def test_pair_column_sum_ring_wraps_over_many_tiles():
    """K = 48 (one stage per tile) and 512 pair tiles: each pair walks several
    tiles per slot of the column-sum exchange ring."""
    rng = np.random.default_rng(21)
    M, K, N = 4096, 48, 8192
    A, B = rand(rng, "u8", (M, K)), rand(rng, "s8", (K, N))
    a_zp, b_zp = rand(rng, "u8", (1,)), rand(rng, "s8", (N,))
    got = mmi(A, B, a_zp, b_zp)
    assert q.last_kernel() == PAIR_MMI
    rows = np.sort(rng.choice(M, 96, replace=False))
    rows[:2] = [0, M - 1]
    assert_equal(got[rows], O.matmul_integer(A[rows], B, a_zp, b_zp), "ring wrap, sampled rows")


def test_pair_more_chunks_than_default(monkeypatch):
    monkeypatch.setenv("QMM_CHUNK_K", "64")
    rng = np.random.default_rng(2)
    A, B = rand(rng, "u8", (300, 704)), rand(rng, "s8", (704, 96))
    a_zp, b_zp = rand(rng, "u8", (1,)), rand(rng, "s8", (96,))
    got = mmi(A, B, a_zp, b_zp)
    assert q.last_kernel() == PAIR_MMI
    assert_equal(got, O.matmul_integer(A, B, a_zp, b_zp), "pair chunk 64")
    w = W.a8w8(400, 1000 + 8, 300 + 4, seed=5)
    assert_equal(a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"),
                 O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), "pair a8w8 chunk 64")


def test_pair_shared_b_folded_batch_with_per_row_zero_point():
    rng = np.random.default_rng(4)
    A = rand(rng, "u8", (4, 300, 64))          # folded: M = 1200
    B = rand(rng, "s8", (64, 272))
    a_zp = rand(rng, "u8", (300,))             # per row m, the same in every batch
    b_zp = rand(rng, "s8", (272,))
    got = mmi(A, B, a_zp, b_zp)
    assert q.last_kernel() == PAIR_MMI
    assert_equal(got, O.matmul_integer(A, B, a_zp, b_zp), "folded batch, per-row a_zp")


def test_pair_batched_b():
    rng = np.random.default_rng(5)
    A = rand(rng, "s8", (3, 300, 64))
    B = rand(rng, "s8", (3, 64, 48))
    got = mmi(A, B, np.array([-3], np.int8), np.array([5], np.int8))
    assert q.last_kernel() == PAIR_MMI
    assert_equal(got, O.matmul_integer(A, B, -3, 5), "batched B")


def test_pair_wraps_modulo_2_32():
    K = 34816
    A = np.full((256, K), 255, np.uint8)
    B = np.full((K, 16), 255, np.uint8)
    got = mmi(A, B)
    assert q.last_kernel() == PAIR_MMI
    assert (got == 65025 * K - 2**32).all()
