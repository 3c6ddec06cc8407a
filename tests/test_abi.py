"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/qmm.h declares, and rejects malformed arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\([^;{]*\)\s*;", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def qmm():
    import quantized_int8_matmul_gb300 as q
    return q


def test_header_declares_the_four_forms():
    names = declared_functions()
    for fn in ("qmm_w8_dequant", "qmm_a8w8", "matmul_integer", "dynamic_quantize_linear"):
        assert fn in names


def test_library_exports_every_declared_symbol(qmm):
    lib = ctypes.CDLL(qmm.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_library_is_built_for_sm_103a_only(qmm):
    from quantized_int8_matmul_gb300 import _build
    assert _build.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings_and_version(qmm):
    lib = qmm.lib()
    assert lib.qmm_abi_version() == 1
    assert lib.qmm_status_string(0) == b"QMM_OK"
    assert lib.qmm_status_string(4) == b"QMM_ERR_TIMEOUT"
    assert lib.qmm_status_string(99) == b"QMM_UNKNOWN_STATUS"


def test_dql_workspace_size_is_a_device_independent_bound(qmm):
    f = qmm.dynamic_quantize_linear_workspace_bytes
    assert f(0) == 8 and f(1) == 8
    assert f(32768 * 3) == 24
    assert f(8192 * 4096) == 8 * 1024          # capped at 1024 partials
    assert f(10**12) == 8 * 1024


# Malformed calls fail validation on the host and enqueue nothing, so they run without a GPU.
P = ctypes.c_void_p(16)   # a non-null stand-in pointer; never dereferenced on these paths


def test_w8_dequant_rejects_bad_arguments(qmm):
    lib = qmm.lib()
    ok_args = dict(A=P, a=0, B=P, M=4, K=8, N=8, s=P, sc=1, z=None, zc=0, C=P, c=0, st=None)

    def call(**kw):
        a = {**ok_args, **kw}
        return lib.qmm_w8_dequant(a["A"], a["a"], a["B"], a["M"], a["K"], a["N"], a["s"], a["sc"], a["z"],
                                  a["zc"], a["C"], a["c"], a["st"])

    assert call(a=2) == qmm.QMM_ERR_INVALID_ARG          # int8 activations are not form (a)
    assert call(c=4) == qmm.QMM_ERR_INVALID_ARG          # int32 output
    assert call(M=-1) == qmm.QMM_ERR_INVALID_ARG
    assert call(K=2**31) == qmm.QMM_ERR_INVALID_ARG
    assert call(sc=3) == qmm.QMM_ERR_INVALID_ARG          # scale count neither 1 nor N
    assert call(zc=1, z=None) == qmm.QMM_ERR_INVALID_ARG  # zero point count without pointer
    assert call(zc=5) == qmm.QMM_ERR_INVALID_ARG
    assert call(s=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(M=0) == qmm.QMM_OK                        # empty output: nothing to do


def test_a8w8_rejects_bad_arguments(qmm):
    lib = qmm.lib()

    def call(M=4, K=8, N=8, ac=1, wc=1, c=1, A=P, C=P):
        return lib.qmm_a8w8(A, P, M, K, N, P, ac, P, wc, C, c, None)

    assert call(ac=3) == qmm.QMM_ERR_INVALID_ARG
    assert call(wc=2) == qmm.QMM_ERR_INVALID_ARG
    assert call(c=2) == qmm.QMM_ERR_INVALID_ARG
    assert call(A=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(C=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(N=-5) == qmm.QMM_ERR_INVALID_ARG
    assert call(N=0) == qmm.QMM_OK


def test_matmul_integer_rejects_bad_arguments(qmm):
    lib = qmm.lib()

    def call(ad=3, bd=2, batch=1, M=4, K=8, N=8, sa=0, sb=0, az=None, azc=0, bz=None, bzc=0, C=P):
        return lib.matmul_integer(P, ad, P, bd, batch, M, K, N, sa, sb, az, azc, bz, bzc, C, None)

    assert call(ad=0) == qmm.QMM_ERR_INVALID_ARG          # float A
    assert call(bd=4) == qmm.QMM_ERR_INVALID_ARG
    assert call(sa=-1) == qmm.QMM_ERR_INVALID_ARG
    assert call(azc=1) == qmm.QMM_ERR_INVALID_ARG         # count without pointer
    assert call(az=P, azc=3) == qmm.QMM_ERR_INVALID_ARG   # neither 1 nor M
    assert call(bz=P, bzc=4) == qmm.QMM_ERR_INVALID_ARG   # neither 1 nor N
    assert call(batch=2**20, M=2**12) == qmm.QMM_ERR_UNSUPPORTED   # batch*M beyond int32
    assert call(batch=0) == qmm.QMM_OK


def test_dql_rejects_bad_arguments(qmm):
    lib = qmm.lib()
    ws = ctypes.c_void_p(4096)

    def call(n=100, x=P, y=P, rs=None, rl=0, w=ws, wb=8):
        return lib.dynamic_quantize_linear(x, n, y, P, P, rs, rl, w, wb, None)

    assert call(n=-1) == qmm.QMM_ERR_INVALID_ARG
    assert call(x=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(w=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(w=ctypes.c_void_p(4100)) == qmm.QMM_ERR_INVALID_ARG     # workspace not 16-byte aligned
    assert call(n=10**7, wb=8) == qmm.QMM_ERR_INVALID_ARG                # workspace too small
    assert call(rs=P, rl=7) == qmm.QMM_ERR_INVALID_ARG                   # 100 % 7 != 0
    assert call(rs=P, rl=0) == qmm.QMM_ERR_INVALID_ARG


def test_a8w8_host_workspace_holds_the_operands_and_the_two_pass_workspace(qmm):
    lib = qmm.lib()
    M, K, N = 4096, 4096, 4096
    host = lib.qmm_a8w8_host_workspace_bytes(M, K, N, M, N, qmm.QMM_BF16)
    operands = M * K + K * N + 4 * (M + N) + 2 * M * N
    assert host >= operands + lib.qmm_a8w8_workspace_bytes(M, K, N)
    # outside the two-pass path: the device copies only
    small = lib.qmm_a8w8_host_workspace_bytes(100, 64, 64, 1, 1, qmm.QMM_F32)
    assert 100 * 64 + 64 * 64 + 4 * 100 * 64 <= small < 100 * 64 + 64 * 64 + 4 * 100 * 64 + 6 * 256
    assert lib.qmm_a8w8_host_workspace_bytes(M, K, N, M, N, 7) == 0      # not an output type
    assert lib.qmm_a8w8_host_workspace_bytes(0, K, N, 1, 1, qmm.QMM_BF16) == 0


def test_a8w8_host_rejects_bad_arguments(qmm):
    lib = qmm.lib()
    ws = ctypes.c_void_p(4096)

    def call(M=4, K=8, N=8, ac=1, wc=1, c=1, A=P, C=P, w=ws, wb=1 << 20):
        return lib.qmm_a8w8_host(A, P, M, K, N, P, ac, P, wc, C, c, w, wb, None)

    assert call(ac=3) == qmm.QMM_ERR_INVALID_ARG
    assert call(wc=2) == qmm.QMM_ERR_INVALID_ARG
    assert call(c=2) == qmm.QMM_ERR_INVALID_ARG
    assert call(A=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(C=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(w=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(w=ctypes.c_void_p(4100)) == qmm.QMM_ERR_INVALID_ARG      # workspace not 16-byte aligned
    assert call(wb=64) == qmm.QMM_ERR_INVALID_ARG                        # workspace too small
    assert call(N=0) == qmm.QMM_OK


def _i64s(*v):
    return (ctypes.c_int64 * len(v))(*v)


def test_conv_workspace_follows_the_route(qmm):
    """Groups of whole 64-channel blocks take the implicit GEMM, whose workspace
    holds the fp16 NHWC input and weight only; other shapes hold the im2col
    matrix, which is larger by about the kernel's tap count."""
    lib = qmm.lib()
    pads, strides, dils = _i64s(1, 1, 1, 1), _i64s(1, 1), _i64s(1, 1)
    N, C, H, W, M = 8, 256, 56, 56, 256
    implicit = lib.conv_integer_workspace_bytes(N, C, H, W, M, 3, 3, pads, strides, dils, 1)
    assert 2 * (N * H * W * C + M * C * 9) <= implicit < 2 * (N * H * W * C + M * C * 9) + 1024
    # 48 channels per group: not whole 64-channel blocks -> the im2col matrix (9x the input in fp16)
    im2col = lib.conv_integer_workspace_bytes(N, 48, H, W, M, 3, 3, pads, strides, dils, 1)
    assert im2col >= 2 * N * 48 * 9 * H * W
    # an output row that is not a 16-byte multiple (oH*oW % 4 != 0) also takes the im2col route
    odd = lib.conv_integer_workspace_bytes(1, 64, 5, 5, 8, 3, 3, pads, strides, dils, 1)
    assert odd >= 2 * 64 * 9 * 25


def test_w8_dequant_workspace_follows_the_route(qmm):
    lib = qmm.lib()
    K, N = 8192, 28672
    kp = (K + 15) // 16 * 16
    for M in (3, 4, 16):   # decode rows, bf16: the GEMV's fp16 activations and row scales
        b = lib.qmm_w8_dequant_workspace_bytes(qmm.QMM_BF16, M, K, N)
        assert 2 * M * kp <= b <= 2 * M * kp + 512
    for M in (1, 2):       # one or two rows keep the CUDA-core kernel: no workspace
        assert lib.qmm_w8_dequant_workspace_bytes(qmm.QMM_BF16, M, K, N) == 0
    assert lib.qmm_w8_dequant_workspace_bytes(qmm.QMM_F32, 4, K, N) == 0     # fp32 decode rows
    assert lib.qmm_w8_dequant_workspace_bytes(qmm.QMM_BF16, 4, K + 4, N) == 0  # K % 8 != 0
    # prefill (M >= 64): the exact bf16 weight copy
    assert lib.qmm_w8_dequant_workspace_bytes(qmm.QMM_BF16, 4096, K, N) >= 2 * K * N


def test_decode_pack_sizes_follow_the_layout(qmm):
    """The packed decode weight: K padded to 16-row steps, N to 64-column
    slabs; shapes outside the path (K or N not a multiple of 8) give 0."""
    lib = qmm.lib()
    assert lib.qmm_w8_decode_pack_bytes(8192, 28672) == 8192 * 28672
    assert lib.qmm_w8_decode_pack_bytes(1000, 200) == 1008 * 256
    assert lib.qmm_w8_decode_pack_bytes(1000, 100) == 0
    assert lib.qmm_w8_decode_pack_bytes(12, 64) == 0
    assert lib.qmm_w8_dequant_packed_workspace_bytes(4, 8192) >= 8 * 8192 * 2
    assert lib.qmm_w8_dequant_packed_workspace_bytes(9, 8192) >= 16 * 8192 * 2
    assert lib.qmm_w8_dequant_packed_workspace_bytes(17, 8192) == 0


def test_packed_chain_sizes_and_host_checks(qmm):
    """The chain's packed weight holds the fp16 copy (pitch N rounded to 8)
    and N column sums; the packed call's workspace holds no weight, and the
    host rejects a short or null packed buffer before any launch."""
    lib = qmm.lib()
    assert lib.dynamic_quantize_matmul_weight_bytes(4096, 11008) >= 4096 * 11008 * 2 + 11008 * 4
    assert lib.dynamic_quantize_matmul_weight_bytes(100, 5) >= 100 * 8 * 2 + 5 * 4
    assert lib.dynamic_quantize_matmul_weight_bytes(0, 5) == 0
    full = lib.dynamic_quantize_matmul_workspace_bytes(512, 4096, 11008)
    act = lib.dynamic_quantize_matmul_packed_workspace_bytes(512, 4096)
    assert act >= 512 * 4096 * 2 and full - act >= 4096 * 11008 * 2
    P = ctypes.c_void_p(256)
    need = lib.dynamic_quantize_matmul_weight_bytes(8, 3)
    ws = lib.dynamic_quantize_matmul_packed_workspace_bytes(4, 8)

    def call(packed=P, pb=need, wdt=qmm.QMM_S8, w=P, wb=ws):
        return lib.dynamic_quantize_matmul_packed(P, 4, 8, packed, pb, wdt, 3, P, 1, None, 0, None, P, None, None,
                                                  w, wb, None)
    assert call(pb=need - 1) == qmm.QMM_ERR_INVALID_ARG
    assert call(packed=None) == qmm.QMM_ERR_INVALID_ARG
    assert call(wdt=qmm.QMM_F32) == qmm.QMM_ERR_INVALID_ARG
    assert call(wb=ws - 1) == qmm.QMM_ERR_INVALID_ARG
    assert lib.dynamic_quantize_matmul_pack_weight(P, qmm.QMM_U8, 8, 3, P, need - 1, None) == qmm.QMM_ERR_INVALID_ARG
