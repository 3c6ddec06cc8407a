"""MatMulInteger (form (c)) through the C ABI against the oracle's direct
definition: int32 outputs must be bit-exact, including wrap-around."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, gemm_kernel, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

INFO = {"s8": (np.int8, -128, 127), "u8": (np.uint8, 0, 255)}


def rand(rng, dt, shape):
    t, lo, hi = INFO[dt]
    return rng.integers(lo, hi + 1, size=shape).astype(t)


def run(A, B, a_zp=None, b_zp=None):
    C = q.matmul_integer(dev(A), dev(B), None if a_zp is None else dev(a_zp), None if b_zp is None else dev(b_zp),
                         workspace=None)
    q.check_device_error()
    return host(C)


def oracle(A, B, a_zp, b_zp):
    return O.matmul_integer(A, B, 0 if a_zp is None else a_zp, 0 if b_zp is None else b_zp)


@pytest.mark.parametrize("adt,bdt", [("s8", "s8"), ("u8", "s8"), ("s8", "u8"), ("u8", "u8")])
@pytest.mark.parametrize("zp", ["none", "scalar", "vector", "a_only", "b_only"])
@pytest.mark.parametrize("M,K,N", [(5, 48, 32), (129, 259, 200), (200, 1040, 272)])
def test_matmul_integer_matches_oracle(adt, bdt, zp, M, K, N):
    rng = np.random.default_rng(M + K + N + len(zp))
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
    got = run(A, B, a_zp, b_zp)
    assert q.last_kernel() == gemm_kernel("matmul_integer", M, K, N)
    assert_equal(got, oracle(A, B, a_zp, b_zp), f"{adt}x{bdt} zp={zp} {M}x{K}x{N}")


def test_page_value_length_259():
    g = json.load(open(os.path.join(GOLDEN, "matmul_integer_u8_len259.json")))
    for N in (1, 16):
        A = np.full((1, g["K"]), g["a_value"], np.uint8)
        B = np.full((g["K"], N), g["b_value"], np.uint8)
        got = run(A, B)
        assert got.tolist() == [[g["expected"]] * N]


def test_wraps_modulo_2_32():
    K = 34816
    A = np.full((2, K), 255, np.uint8)
    B = np.full((K, 16), 255, np.uint8)
    got = run(A, B)
    assert (got == 65025 * K - 2**32).all()


@pytest.mark.parametrize("adt,bdt,a,b", [("s8", "s8", -128, -128), ("u8", "s8", 255, -128), ("u8", "u8", 255, 255),
                                         ("s8", "u8", -128, 255)])
def test_exact_at_chunk_edge(adt, bdt, a, b):
    """Each K-chunk sum sits at the largest magnitude the fp32 accumulator holds exactly."""
    M, K, N = 130, 4096, 272
    A = np.full((M, K), a, INFO[adt][0])
    B = np.full((K, N), b, INFO[bdt][0])
    got = run(A, B)
    assert (got == np.int64(a) * b * K).all()


def test_more_chunks_than_default(monkeypatch):
    monkeypatch.setenv("QMM_CHUNK_K", "64")
    rng = np.random.default_rng(2)
    A, B = rand(rng, "u8", (150, 700)), rand(rng, "s8", (700, 96))
    a_zp, b_zp = rand(rng, "u8", (1,)), rand(rng, "s8", (96,))
    assert_equal(run(A, B, a_zp, b_zp), oracle(A, B, a_zp, b_zp), "chunk 64")


def test_shared_rank2_b_folds_batch_into_m():
    rng = np.random.default_rng(3)
    A = rand(rng, "s8", (2, 3, 40, 64))
    B = rand(rng, "s8", (64, 48))
    a_zp = np.array([-5], np.int8)
    b_zp = np.array([7], np.int8)
    got = run(A, B, a_zp, b_zp)
    assert got.shape == (2, 3, 40, 48)
    assert_equal(got, oracle(A, B, a_zp, b_zp), "shared B")


def test_shared_b_with_per_row_zero_point():
    rng = np.random.default_rng(4)
    A = rand(rng, "u8", (4, 33, 64))
    B = rand(rng, "s8", (64, 32))
    a_zp = rand(rng, "u8", (33,))      # one per row m, the same in every batch
    got = run(A, B, a_zp, None)
    assert_equal(got, oracle(A, B, a_zp, None), "per-row a_zp across batches")


def test_batched_b_and_broadcast_a():
    rng = np.random.default_rng(5)
    A = rand(rng, "s8", (3, 33, 64))
    B = rand(rng, "s8", (3, 64, 48))
    assert_equal(run(A, B), oracle(A, B, None, None), "batched B")
    A1 = rand(rng, "u8", (1, 33, 64))
    got = run(A1, B, np.array([9], np.uint8), None)
    want = O.matmul_integer(np.broadcast_to(A1, (3, 33, 64)), B, 9, 0)
    assert_equal(got, want, "size-1 batch on A")


def test_size_one_b_batch_is_shared():
    rng = np.random.default_rng(6)
    A = rand(rng, "s8", (4, 20, 32))
    B = rand(rng, "s8", (1, 32, 16))
    assert_equal(run(A, B), oracle(A, B[0], None, None), "B batch of 1")


def test_k_zero_gives_zeros():
    A = torch.empty((2, 3, 0), dtype=torch.int8, device="cuda")
    B = torch.empty((0, 5), dtype=torch.int8, device="cuda")
    C = q.matmul_integer(A, B)
    assert q.last_kernel() == "memset_zero"
    assert C.shape == (2, 3, 5) and torch.count_nonzero(C).item() == 0


@pytest.mark.parametrize("adt,bdt", [("u8", "s8"), ("s8", "s8"), ("u8", "u8")])
def test_long_k_row_and_column_sums(adt, bdt):
    """K = 4160 (65 K-stages): the column sums are folded from 16-bit lanes several times per tile."""
    rng = np.random.default_rng(12)
    M, K, N = 130, 4160, 272
    A, B = rand(rng, adt, (M, K)), rand(rng, bdt, (K, N))
    if bdt == "s8":
        B[:, :16] = -128            # extreme column sums
    a_zp, b_zp = rand(rng, adt, (1,)), rand(rng, bdt, (N,))
    assert_equal(run(A, B, a_zp, b_zp), oracle(A, B, a_zp, b_zp), f"{adt}x{bdt} K=4160")
