"""Decode form (a) on a weight packed once (qmm_w8_pack_decode_weight +
qmm_w8_dequant_packed) against the oracle, through the C ABI: within the
stated bound (1e-3 * sum_k |a_k * scale_n * (b_k - zp_n)| + 1e-6, plus half an
ulp of the output type) for 1..16 rows, ragged K and N (the packed layout pads
both), zero-point modes, both output types, K split over clusters, the full
8192 x 28672 decode shape, rows spanning the bf16 range, and determinism."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_within, bf16_bits_to_f64, bf16_dev, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")


def kernel_name(M, K, zp):
    """Rows whose fp16 copy (row pitch K rounded to 16, plus 16) fits
    16.5 KiB are prepared inside each CTA; otherwise by a prep kernel."""
    Kp = -(-K // 16) * 16
    if M <= 8 and M * (Kp + 16) * 2 <= 16 * 1024 + 512:
        base = "gemv_w8_packed_rows_in_cta"
    else:
        base = "gemv_prep_rows+gemv_w8_packed" + ("_m16" if M > 8 else "")
    return base + ("_zp" if zp else "")


def run(A_bits, A_vals, B, scale, zp, out, cols=None):
    M, K = A_bits.shape
    N = B.shape[1]
    packed = q.qmm_w8_pack_decode_weight(dev(B))
    assert q.last_kernel() == "gemv_w8_pack"
    C = q.qmm_w8_dequant_packed(bf16_dev(A_bits), packed, N, dev(scale), None if zp is None else dev(zp),
                                out_dtype=out)
    q.check_device_error()
    assert q.last_kernel() == kernel_name(M, K, zp is not None)
    got = host(C)
    gotf = bf16_bits_to_f64(got) if out == torch.bfloat16 else got.astype(np.float64)
    zpv = np.zeros(1, np.int32) if zp is None else zp
    if cols is not None:
        B = np.ascontiguousarray(B[:, cols])
        scale = scale[cols] if scale.size > 1 else scale
        zpv = zpv[cols] if zpv.size > 1 else zpv
        gotf = gotf[:, cols]
    exact = O.w8_dequant(A_vals, B, scale, zpv)
    bound = O.w8_dequant_error_bound(A_vals, B, scale, zpv)
    assert_within(gotf, exact, bound, 7 if out == torch.bfloat16 else 23, kernel_name(M, K, zp is not None))
    return C


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 16])
@pytest.mark.parametrize("zp", [None, "tensor", "column"])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_packed_decode_rows_zero_points_outputs(M, zp, out):
    w = W.decode_gemv(M, K=1024, N=640, seed=M + 60)
    rng = np.random.default_rng(M + 60)
    z = None if zp is None else (np.array([-3], np.int32) if zp == "tensor" else rng.integers(-9, 9, 640).astype(np.int32))
    run(w.A_bits, w.A, w.W, w.scale, z, out)


@pytest.mark.parametrize("K,N", [(8, 8), (24, 72), (1000, 200), (1032, 1000), (4104, 136), (8192, 640), (2056, 4096)])
def test_packed_decode_ragged_shapes(K, N):
    """K not a multiple of 16 and N not a multiple of 64: the packed layout's
    zero padding (a biased 0) and the prep's zero rows meet at the edges."""
    w = W.decode_gemv(5, K=K, N=N, seed=K + N)
    z = np.arange(-5, N - 5, dtype=np.int32) % 11 - 5
    run(w.A_bits, w.A, w.W, w.scale, z, torch.float32)


@pytest.mark.parametrize("M,K,N", [(1, 8192, 640), (2, 4096, 640), (4, 2056, 136), (3, 16384, 192),
                                   (8, 1024, 256), (8, 8192, 640), (5, 8192, 1024), (2, 8192, 640)])
def test_packed_decode_split_k_and_both_preps(M, K, N):
    """Few slabs, so K is split over a cluster (up to 8 CTAs): with the rows
    prepared inside each CTA (every CTA scales by the whole row's maximum and
    keeps only its K range) and, for rows too large for that, by the prep
    kernel."""
    w = W.decode_gemv(M, K=K, N=N, seed=M * 7 + K)
    z = (np.arange(N, dtype=np.int32) % 7) - 3
    run(w.A_bits, w.A, w.W, w.scale, z, torch.float32)


def test_packed_decode_scalar_scale_and_row_range():
    """A scalar scale, and rows whose magnitudes lie far outside fp16's range
    (2^-60 .. 2^100) plus an all-zero row: each row's power-of-two scale keeps
    its values exact."""
    rng = np.random.default_rng(8)
    M, K, N = 7, 512, 256
    e = np.array([-60, -24, -3, 0, 17, 100, 0])[:, None]
    A32 = (W.normal_f32(rng, (M, K)) * np.exp2(e.astype(np.float64))).astype(np.float32)
    A32[6] = 0.0
    bits = (A32.view(np.uint32) >> 16).astype(np.uint16)
    A = (bits.astype(np.uint32) << 16).view(np.float32)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    run(bits, A, B, np.array([0.02], np.float32), np.array([2], np.int32), torch.float32)


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("zp", [False, True])
def test_packed_decode_8192x28672(M, zp):
    """The decode workload at full size, 1024 sampled columns x all rows; with
    a per-column zero point too (the row sums come from one more MMA per step)."""
    w = W.decode_gemv(M)
    cols = np.random.default_rng(M).choice(28672, 1024, replace=False)
    z = ((np.arange(28672, dtype=np.int32) * 7) % 15 - 7) if zp else None
    run(w.A_bits, w.A, w.W, w.scale, z, torch.bfloat16, cols=cols)


def test_packed_decode_is_deterministic_and_reuses_the_pack():
    w = W.decode_gemv(4, K=4096, N=2048, seed=5)
    packed = q.qmm_w8_pack_decode_weight(dev(w.W))
    outs = []
    for _ in range(3):
        C = q.qmm_w8_dequant_packed(bf16_dev(w.A_bits), packed, 2048, dev(w.scale), out_dtype=torch.float32)
        q.check_device_error()
        outs.append(host(C))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    # same bits as a fresh pack of the same weight
    again = q.qmm_w8_pack_decode_weight(dev(w.W))
    torch.cuda.synchronize()
    assert torch.equal(packed, again)


def test_packed_decode_rejects_bad_arguments():
    A = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    W8 = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    packed = q.qmm_w8_pack_decode_weight(W8)
    s = torch.ones(64, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError):   # 17 rows: outside the decode path
        q.qmm_w8_dequant_packed(torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda"), packed, 64, s)
    with pytest.raises(q.QmmError):   # packed buffer too short for N = 128
        q.qmm_w8_dequant_packed(A, packed, 128, torch.ones(128, dtype=torch.float32, device="cuda"))
    with pytest.raises(q.QmmError):   # K not a multiple of 8
        q.qmm_w8_pack_decode_weight(torch.zeros((12, 64), dtype=torch.int8, device="cuda"))
