"""The two-pass path (exact fp16 operand copies + row/column sums in a
workspace, then the SM-pair GEMM fed by TMA) against the oracle: A8W8 and
MatMulInteger bit for bit, on ragged pair tiles, the 2^24 chunk edge, many
tiles per pair, batches (folded, batched B, broadcast A) and int32 wrap-around;
plus the fall-back to the single-pass kernels and workspace validation."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, gemm_kernel, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

INFO = {"s8": (np.int8, -128, 127), "u8": (np.uint8, 0, 255)}
TWO_PASS_A8W8 = "f16_prepass+gemm_tc05_pair_f16ops_a8w8"
TWO_PASS_MMI = "f16_prepass+gemm_tc05_pair_f16ops_matmul_integer"


def rand(rng, dt, shape):
    t, lo, hi = INFO[dt]
    return rng.integers(lo, hi + 1, size=shape).astype(t)


def a8w8(A, B, a_s, w_s, out="f32", workspace="auto"):
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = q.qmm_a8w8(dev(A), dev(B), dev(a_s), dev(w_s), out_dtype=dt, workspace=workspace)
    q.check_device_error()
    return host(C)


def mmi(A, B, a_zp=None, b_zp=None, workspace="auto"):
    C = q.matmul_integer(dev(A), dev(B), None if a_zp is None else dev(a_zp), None if b_zp is None else dev(b_zp),
                         workspace=workspace)
    q.check_device_error()
    return host(C)


SHAPES = [(256, 64, 256), (257, 128, 272), (384, 320, 400), (300, 4096, 528), (1000, 1040, 1008), (512, 16, 128),
          (640, 2064, 144)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_two_pass_a8w8_matches_oracle(M, K, N, out):
    w = W.a8w8(M, K, N, seed=M + 5 * K + 3 * N)
    got = a8w8(w.A, w.B, w.act_scale, w.weight_scale, out)
    assert q.last_kernel() == TWO_PASS_A8W8
    assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, out), f"two-pass a8w8 {out} {M}x{K}x{N}")


def test_two_pass_a8w8_scalar_scales_and_chunk_edge():
    rng = np.random.default_rng(11)
    M, K, N = 300, 4096, 272
    A = rng.choice(np.array([-128, 127, -127, 126], np.int8), size=(M, K))
    B = rng.choice(np.array([-128, 127], np.int8), size=(K, N))
    one = np.ones(1, np.float32)
    assert_equal(a8w8(A, B, one, one), O.a8w8(A, B, one, one, "f32"), "extremes, scalar scales")
    A = np.full((M, K), -128, np.int8)
    B = np.full((K, N), -128, np.int8)
    assert (a8w8(A, B, one, one) == np.float32(16384 * K)).all()


def test_one_workspace_serves_calls_of_several_shapes():
    """A workspace of arbitrary bytes, reused by calls of other shapes."""
    shapes = [(1000, 1040, 1008), (1536, 192, 2000), (1000, 1040, 1008), (257, 128, 272)]
    need = max(q.qmm_a8w8_workspace_bytes(*s) for s in shapes)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    for i, (M, K, N) in enumerate(shapes):
        w = W.a8w8(M, K, N, seed=40 + i)
        got = a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16", workspace=ws)
        assert q.last_kernel() == TWO_PASS_A8W8
        assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), f"reused workspace {M}x{K}x{N}")


def test_captured_call_replays_exactly():
    """The two-pass call captured into a CUDA graph (the GEMM a programmatic
    dependent of the pre-pass inside the graph) replays exactly with new
    inputs."""
    M, K, N = 1000, 1040, 1008
    w1, w2 = W.a8w8(M, K, N, seed=50), W.a8w8(M, K, N, seed=51)
    A, B, a_s, w_s = dev(w1.A), dev(w1.B), dev(w1.act_scale), dev(w1.weight_scale)
    ws = torch.empty(q.qmm_a8w8_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        q.qmm_a8w8(A, B, a_s, w_s, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert q.last_kernel() == TWO_PASS_A8W8
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        q.qmm_a8w8(A, B, a_s, w_s, out=out, workspace=ws)
    assert q.last_kernel() == TWO_PASS_A8W8
    for w in (w2, w1, w2):
        A.copy_(dev(w.A))
        B.copy_(dev(w.B))
        a_s.copy_(dev(w.act_scale))
        w_s.copy_(dev(w.weight_scale))
        g.replay()
        torch.cuda.synchronize()
        q.check_device_error()
        assert_equal(host(out), O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), "graph replay")


def test_captured_matmul_integer_with_zero_points_replays_exactly():
    """With zero points the two conversions run on two streams (forked and
    joined with events); captured into a CUDA graph, the fork and join become
    graph edges and replays with new inputs stay exact."""
    rng = np.random.default_rng(17)
    M, K, N = 600, 512, 400
    A0, B0 = rand(rng, "u8", (M, K)), rand(rng, "s8", (K, N))
    a_zp, b_zp = rand(rng, "u8", (1,)), rand(rng, "s8", (N,))
    A, B, za, zb = dev(A0), dev(B0), dev(a_zp), dev(b_zp)
    out = torch.empty((M, N), dtype=torch.int32, device="cuda")
    ws = torch.empty(q.matmul_integer_workspace_bytes(1, M, K, N, 0, 0), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        q.matmul_integer(A, B, za, zb, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        q.matmul_integer(A, B, za, zb, out=out, workspace=ws)
    assert q.last_kernel() == TWO_PASS_MMI
    for seed in (1, 2):
        r = np.random.default_rng(seed)
        An, Bn = rand(r, "u8", (M, K)), rand(r, "s8", (K, N))
        A.copy_(dev(An))
        B.copy_(dev(Bn))
        g.replay()
        torch.cuda.synchronize()
        q.check_device_error()
        assert_equal(host(out), O.matmul_integer(An, Bn, a_zp, b_zp), f"graph replay {seed}")


@pytest.mark.parametrize("adt,bdt", [("s8", "s8"), ("u8", "s8"), ("s8", "u8"), ("u8", "u8")])
@pytest.mark.parametrize("zp", ["none", "scalar", "vector", "a_only", "b_only"])
@pytest.mark.parametrize("M,K,N", [(260, 1040, 272), (513, 272, 400)])
def test_two_pass_matmul_integer_matches_oracle(adt, bdt, zp, M, K, N):
    rng = np.random.default_rng(M + K + N + len(zp) + 11 * len(adt + bdt))
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
    assert q.last_kernel() == TWO_PASS_MMI
    want = O.matmul_integer(A, B, 0 if a_zp is None else a_zp, 0 if b_zp is None else b_zp)
    assert_equal(got, want, f"two-pass {adt}x{bdt} zp={zp} {M}x{K}x{N}")


@pytest.mark.parametrize("adt,bdt,a,b", [("s8", "s8", -128, -128), ("u8", "s8", 255, -128), ("u8", "u8", 255, 255),
                                         ("s8", "u8", -128, 255)])
def test_two_pass_exact_at_chunk_edge_with_sums(adt, bdt, a, b):
    M, K, N = 260, 4096, 272
    A = np.full((M, K), a, INFO[adt][0])
    B = np.full((K, N), b, INFO[bdt][0])
    za = np.array([3], INFO[adt][0])
    zb = np.array([5], INFO[bdt][0])
    got = mmi(A, B, za, zb)
    assert q.last_kernel() == TWO_PASS_MMI
    want = ((np.int64(a) - 3) * (np.int64(b) - 5) * K + 2**31) % 2**32 - 2**31
    assert (got == want).all()


def test_two_pass_many_tiles_per_pair():
    rng = np.random.default_rng(21)
    M, K, N = 4096, 48, 8192
    A, B = rand(rng, "u8", (M, K)), rand(rng, "s8", (K, N))
    a_zp, b_zp = rand(rng, "u8", (1,)), rand(rng, "s8", (N,))
    got = mmi(A, B, a_zp, b_zp)
    assert q.last_kernel() == TWO_PASS_MMI
    rows = np.sort(rng.choice(M, 96, replace=False))
    rows[:2] = [0, M - 1]
    assert_equal(got[rows], O.matmul_integer(A[rows], B, a_zp, b_zp), "many tiles, sampled rows")


def test_two_pass_more_chunks_than_default(monkeypatch):
    monkeypatch.setenv("QMM_CHUNK_K", "64")
    rng = np.random.default_rng(2)
    A, B = rand(rng, "u8", (300, 704)), rand(rng, "s8", (704, 96))
    a_zp, b_zp = rand(rng, "u8", (1,)), rand(rng, "s8", (96,))
    assert_equal(mmi(A, B, a_zp, b_zp), O.matmul_integer(A, B, a_zp, b_zp), "two-pass chunk 64")
    assert q.last_kernel() == TWO_PASS_MMI


def test_two_pass_folded_batch_batched_b_and_broadcast_a():
    rng = np.random.default_rng(4)
    A = rand(rng, "u8", (4, 300, 64))          # shared B: folded to M = 1200
    B = rand(rng, "s8", (64, 272))
    a_zp = rand(rng, "u8", (300,))
    b_zp = rand(rng, "s8", (272,))
    assert_equal(mmi(A, B, a_zp, b_zp), O.matmul_integer(A, B, a_zp, b_zp), "folded, per-row a_zp")
    assert q.last_kernel() == TWO_PASS_MMI
    A3 = rand(rng, "s8", (3, 300, 64))
    B3 = rand(rng, "s8", (3, 64, 48))
    assert_equal(mmi(A3, B3, np.array([-3], np.int8), np.array([5], np.int8)), O.matmul_integer(A3, B3, -3, 5),
                 "batched B")
    assert q.last_kernel() == TWO_PASS_MMI
    A1 = rand(rng, "u8", (1, 300, 64))          # one A for every batch of B
    got = mmi(A1, B3.view(np.int8), np.array([9], np.uint8), np.array([-2], np.int8))
    want = O.matmul_integer(np.broadcast_to(A1, (3, 300, 64)), B3, 9, -2)
    assert_equal(got, want, "broadcast A")
    assert q.last_kernel() == TWO_PASS_MMI


def test_two_pass_wraps_modulo_2_32():
    K = 34816
    A = np.full((256, K), 255, np.uint8)
    B = np.full((K, 16), 255, np.uint8)
    got = mmi(A, B)
    assert q.last_kernel() == TWO_PASS_MMI
    assert (got == 65025 * K - 2**32).all()


@pytest.mark.parametrize("M,K,N", [(100, 64, 64), (300, 40, 64), (300, 64, 40)])
def test_shapes_outside_the_two_pass_path_fall_back(M, K, N):
    w = W.a8w8(M, K, N, seed=7)
    assert q.qmm_a8w8_workspace_bytes(M, K, N) == 0
    got = a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16")
    assert q.last_kernel() == gemm_kernel("a8w8", M, K, N)
    assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), "fall-back")


def test_workspace_too_small_is_rejected():
    w = W.a8w8(256, 64, 256, seed=1)
    need = q.qmm_a8w8_workspace_bytes(256, 64, 256)
    assert need >= 2 * (256 * 64 + 64 * 256)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16", workspace=small)


def test_pack_then_packed_equals_one_call_and_reuses_the_pack():
    w = W.a8w8(512, 1024, 384, seed=3)
    A, B = dev(w.A), dev(w.B)
    ws = torch.empty(q.qmm_a8w8_workspace_bytes(512, 1024, 384), dtype=torch.uint8, device="cuda")
    q.qmm_a8w8_pack(A, B, ws)
    assert q.last_kernel() == "f16_prepass"
    for seed in (0, 1):
        rng = np.random.default_rng(seed)
        a_s = rng.uniform(0.005, 0.02, 512).astype(np.float32)
        w_s = rng.uniform(0.001, 0.01, 384).astype(np.float32)
        C = q.qmm_a8w8_packed(512, 1024, 384, dev(a_s), dev(w_s), ws)
        q.check_device_error()
        assert q.last_kernel() == "gemm_tc05_pair_f16ops_a8w8"
        assert_equal(host(C), O.a8w8(w.A, w.B, a_s, w_s, "bf16"), f"packed, scales {seed}")


def test_pack_rejects_shapes_outside_the_path():
    A = torch.zeros((100, 64), dtype=torch.int8, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        q.qmm_a8w8_pack(A, B, ws)
