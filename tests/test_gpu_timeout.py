"""The failure path of the kernels' bounded waits, run on the GPU without any
fault: a host-side test hook makes one SM pair of the two-pass A8W8 GEMM skip
the arrival and the copies of its first operand stage, so that pair's MMA
issuer waits for data that never comes. The wait must run out after the short
limit given, the error word must name the site, the pair must unwind (drain,
free its tensor memory, return) while every other pair finishes its tiles, and
the context must stay usable: the next ordinary call is bit-exact.

Pattern of ROCm hip-ep PR #1248 ("What", last paragraph): errors are cleared
before a launch and read back after it, here through qmm_check_device_error.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import qmm_oracle as O
from _helpers import dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

SITE_FULL = 0x401          # the MMA issuer's wait for an operand stage
SENTINEL = 0x7FC1          # a bf16 NaN no result can take


def _stall_fn():
    f = q.lib().qmm_test_a8w8_packed_stall
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, ctypes.c_int, vp, ctypes.c_size_t, ctypes.c_uint64, vp]
    f.restype = ctypes.c_int
    return f


def _problem(seed, M=1024, K=1024, N=1024):
    rng = np.random.default_rng(seed)
    A = rng.integers(-127, 128, (M, K), dtype=np.int8)
    B = rng.integers(-127, 128, (K, N), dtype=np.int8)
    a_s = rng.uniform(0.005, 0.02, M).astype(np.float32)
    w_s = rng.uniform(0.001, 0.01, N).astype(np.float32)
    return A, B, a_s, w_s


def test_stalled_pair_times_out_unwinds_and_the_next_call_is_exact():
    A, B, a_s, w_s = _problem(3)
    M, K = A.shape
    N = B.shape[1]
    Ad, Bd, asd, wsd = dev(A), dev(B), dev(a_s), dev(w_s)
    ws = torch.empty(q.qmm_a8w8_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
    q.qmm_a8w8_pack(Ad, Bd, ws)
    C = torch.full((M, N), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    lib = q.lib()
    assert lib.qmm_check_device_error(stream) == q.QMM_OK   # nothing pending before the stall
    st = _stall_fn()(M, K, N, ctypes.c_void_p(asd.data_ptr()), M, ctypes.c_void_p(wsd.data_ptr()), N,
                     ctypes.c_void_p(C.data_ptr()), q.QMM_BF16, ctypes.c_void_p(ws.data_ptr()),
                     ws.numel(), 1_000_000, stream)
    assert st == q.QMM_OK, lib.qmm_status_string(st)
    # the kernel returned (the synchronisation inside the check finishes) and reported the site
    assert lib.qmm_check_device_error(stream) == q.QMM_ERR_TIMEOUT
    assert lib.qmm_last_device_error() == SITE_FULL
    assert lib.qmm_check_device_error(stream) == q.QMM_OK    # the word was cleared
    want = O.a8w8(A, B, a_s, w_s, "bf16")
    got = host(C).view(np.uint16)
    # the stalled pair's first tile (rows 0..255, at least columns 0..223) was never written ...
    assert (got[:256, :224] == SENTINEL).all()
    # ... and every other pair finished its tiles exactly
    assert np.array_equal(got[256:], want[256:])
    assert np.array_equal(got[:, 256:], want[:, 256:])
    # the context is usable: an ordinary call afterwards is bit-exact everywhere
    C2 = q.qmm_a8w8(Ad, Bd, asd, wsd, out_dtype=torch.bfloat16, workspace=ws)
    q.check_device_error()
    assert np.array_equal(host(C2).view(np.uint16), want)


def test_stall_hook_rejects_limits_outside_its_range():
    f = _stall_fn()
    for lim in (0, 999, 100_000_001):
        assert f(1024, 1024, 1024, None, 1, None, 1, None, q.QMM_BF16, None, 0, lim, None) == q.QMM_ERR_INVALID_ARG
