"""Python binding of the GB300 integer-quantised matmul library (libqmm.so).

Argument marshalling only: each function checks dtypes/shapes of torch
tensors, passes raw device pointers, sizes and the current CUDA stream to the
C ABI of the same name (include/qmm.h), and raises ``QmmError`` on a non-OK
status. Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback. Output tensors are allocated with torch
when the caller does not pass one (device memory is PyTorch's job here).

If the shared library is missing it is built from ``csrc/`` with nvcc on
first import; if that fails the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple

import torch

from . import _build

QMM_OK, QMM_ERR_INVALID_ARG, QMM_ERR_UNSUPPORTED, QMM_ERR_CUDA, QMM_ERR_TIMEOUT = range(5)
QMM_F32, QMM_BF16, QMM_S8, QMM_U8, QMM_S32 = range(5)

_TORCH_TO_QMM = {
    torch.float32: QMM_F32,
    torch.bfloat16: QMM_BF16,
    torch.int8: QMM_S8,
    torch.uint8: QMM_U8,
    torch.int32: QMM_S32,
}


class QmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == QMM_ERR_CUDA:
            detail = f" (cudaError {_lib.qmm_last_cuda_error()})"
        if status == QMM_ERR_TIMEOUT:
            detail = f" (device error site 0x{_lib.qmm_last_device_error():x})"
        super().__init__(f"{fn}: {_lib.qmm_status_string(status).decode()}{detail}")


def _load() -> ctypes.CDLL:
    path = _build.build()
    lib = ctypes.CDLL(path)
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.qmm_w8_dequant.argtypes = [vp, ci, vp, i64, i64, i64, vp, i64, vp, i64, vp, ci, vp]
    lib.qmm_w8_dequant_workspace_bytes.argtypes = [ci, i64, i64, i64]
    lib.qmm_w8_dequant_workspace_bytes.restype = ctypes.c_size_t
    lib.qmm_w8_dequant_ws.argtypes = [vp, ci, vp, i64, i64, i64, vp, i64, vp, i64, vp, ci, vp, ctypes.c_size_t, vp]
    lib.qmm_a8w8.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, i64, vp, ci, vp]
    lib.matmul_integer.argtypes = [vp, ci, vp, ci, i64, i64, i64, i64, i64, i64, vp, i64, vp, i64, vp, vp]
    sz = ctypes.c_size_t
    lib.qmm_a8w8_workspace_bytes.argtypes = [i64, i64, i64]
    lib.qmm_a8w8_workspace_bytes.restype = sz
    lib.qmm_a8w8_ws.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, i64, vp, ci, vp, sz, vp]
    lib.qmm_a8w8_acc_workspace_bytes.argtypes = [i64, i64, i64]
    lib.qmm_a8w8_acc_workspace_bytes.restype = sz
    lib.qmm_a8w8_acc.argtypes = [vp, ci, vp, ci, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, ci, vp, sz, vp]
    lib.conv_integer_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64, i64, vp, vp, vp, i64]
    lib.conv_integer_workspace_bytes.restype = sz
    lib.conv_integer.argtypes = [vp, ci, vp, ci, i64, i64, i64, i64, i64, i64, i64, vp, vp, vp, i64, vp, vp, i64,
                                 vp, vp, sz, vp]
    lib.dynamic_quantize_matmul_workspace_bytes.argtypes = [i64, i64, i64]
    lib.dynamic_quantize_matmul_workspace_bytes.restype = sz
    lib.dynamic_quantize_matmul.argtypes = [vp, i64, i64, vp, ci, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp, sz, vp]
    lib.dynamic_quantize_matmul_weight_bytes.argtypes = [i64, i64]
    lib.dynamic_quantize_matmul_weight_bytes.restype = sz
    lib.dynamic_quantize_matmul_pack_weight.argtypes = [vp, ci, i64, i64, vp, sz, vp]
    lib.dynamic_quantize_matmul_packed_workspace_bytes.argtypes = [i64, i64]
    lib.dynamic_quantize_matmul_packed_workspace_bytes.restype = sz
    lib.dynamic_quantize_matmul_packed.argtypes = [vp, i64, i64, vp, sz, ci, i64, vp, i64, vp, i64, vp, vp, vp, vp,
                                                   vp, sz, vp]
    lib.qmm_a8w8_pack.argtypes = [vp, vp, i64, i64, i64, vp, sz, vp]
    lib.qmm_a8w8_packed.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, ci, vp, sz, vp]
    lib.qmm_a8w8_host_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, ci]
    lib.qmm_a8w8_host_workspace_bytes.restype = sz
    lib.qmm_a8w8_host.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, i64, vp, ci, vp, sz, vp]
    lib.matmul_integer_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64]
    lib.matmul_integer_workspace_bytes.restype = sz
    lib.matmul_integer_ws.argtypes = [vp, ci, vp, ci, i64, i64, i64, i64, i64, i64, vp, i64, vp, i64, vp, vp, sz, vp]
    lib.dynamic_quantize_linear_workspace_bytes.argtypes = [i64]
    lib.dynamic_quantize_linear_workspace_bytes.restype = ctypes.c_size_t
    lib.dynamic_quantize_linear.argtypes = [vp, i64, vp, vp, vp, vp, i64, vp, ctypes.c_size_t, vp]
    for fn in ("qmm_w8_dequant", "qmm_w8_dequant_ws", "qmm_a8w8", "qmm_a8w8_ws", "qmm_a8w8_pack", "qmm_a8w8_packed", "matmul_integer",
               "matmul_integer_ws", "dynamic_quantize_linear"):
        getattr(lib, fn).restype = ci
    lib.qmm_status_string.argtypes = [ci]
    lib.qmm_status_string.restype = ctypes.c_char_p
    lib.qmm_last_kernel.restype = ctypes.c_char_p
    lib.qmm_last_cuda_error.restype = ci
    lib.qmm_last_device_error.restype = ctypes.c_uint
    lib.qmm_check_device_error.argtypes = [vp]
    lib.qmm_check_device_error.restype = ci
    lib.qmm_num_sms.restype = ci
    lib.qmm_abi_version.restype = ci
    lib.qmm_w8_decode_pack_bytes.argtypes = [i64, i64]
    lib.qmm_w8_decode_pack_bytes.restype = sz
    lib.qmm_w8_pack_decode_weight.argtypes = [vp, i64, i64, vp, sz, vp]
    lib.qmm_w8_pack_decode_weight.restype = ci
    lib.qmm_w8_dequant_packed_workspace_bytes.argtypes = [i64, i64]
    lib.qmm_w8_dequant_packed_workspace_bytes.restype = sz
    lib.qmm_w8_dequant_packed.argtypes = [vp, i64, i64, i64, vp, sz, vp, i64, vp, i64, vp, ci, vp, sz, vp]
    lib.qmm_w8_dequant_packed.restype = ci
    lib.qmm_int8_mma_peak_launch.argtypes = [ci, ctypes.POINTER(ctypes.c_double), vp]
    lib.qmm_int8_mma_peak_launch.restype = ci
    return lib


_lib = _load()
LIB_PATH = _build.LIB_PATH


def lib() -> ctypes.CDLL:
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != QMM_OK:
        raise QmmError(fn, status)


def _need(t, dtypes, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def qmm_w8_pack_decode_weight(W, packed=None, stream=None):
    """Re-lay a frozen int8 weight W [K, N] once for the decode GEMV (same bytes, padded)."""
    _need(W, (torch.int8,), "W")
    K, N = W.shape
    nbytes = int(_lib.qmm_w8_decode_pack_bytes(K, N))
    if nbytes == 0:
        raise QmmError("qmm_w8_pack_decode_weight", QMM_ERR_UNSUPPORTED)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _check("qmm_w8_pack_decode_weight",
           _lib.qmm_w8_pack_decode_weight(_ptr(W), K, N, _ptr(packed), packed.numel(), _stream(stream)))
    return packed


def qmm_w8_dequant_packed(A, packed, N, scale, zero_point=None, out=None, out_dtype=torch.bfloat16,
                          workspace=None, stream=None):
    """Decode form (a), C = scale * (A @ W - zp * rowsum(A)), on a weight packed
    by qmm_w8_pack_decode_weight; A bf16 [M, K], 1 <= M <= 16."""
    _need(A, (torch.bfloat16,), "A")
    _need(scale, (torch.float32,), "scale")
    M, K = A.shape
    zc = 0
    if zero_point is not None:
        _need(zero_point, (torch.int32,), "zero_point")
        zc = zero_point.numel()
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    _need(out, (torch.float32, torch.bfloat16), "out")
    nbytes = int(_lib.qmm_w8_dequant_packed_workspace_bytes(M, K))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=A.device)
    st = _lib.qmm_w8_dequant_packed(_ptr(A), M, K, N, _ptr(packed), packed.numel(), _ptr(scale), scale.numel(),
                                    _ptr(zero_point), zc, _ptr(out), _TORCH_TO_QMM[out.dtype], _ptr(workspace),
                                    workspace.numel(), _stream(stream))
    _check("qmm_w8_dequant_packed", st)
    return out


def qmm_w8_dequant_packed_workspace_bytes(M: int, K: int) -> int:
    return int(_lib.qmm_w8_dequant_packed_workspace_bytes(M, K))


def int8_mma_peak_launch(iters: int, stream=None) -> float:
    """Enqueue the int8 warp-MMA throughput kernel (a measurement aid) and
    return the integer operations it performs; time it with CUDA events."""
    ops = ctypes.c_double(0.0)
    _check("qmm_int8_mma_peak_launch", _lib.qmm_int8_mma_peak_launch(int(iters), ctypes.byref(ops), _stream(stream)))
    return ops.value


def last_kernel() -> str:
    """Name of the kernel(s) the last successful call on this thread launched."""
    return _lib.qmm_last_kernel().decode()


def check_device_error(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a timed-out wait."""
    _check("qmm_check_device_error", _lib.qmm_check_device_error(_stream(stream)))


def qmm_w8_dequant_workspace_bytes(a_dtype, M: int, K: int, N: int) -> int:
    return int(_lib.qmm_w8_dequant_workspace_bytes(_TORCH_TO_QMM[a_dtype], M, K, N))


def qmm_w8_dequant(A, B, scale, zero_point=None, out=None, out_dtype=torch.float32, stream=None, workspace="auto"):
    """Form (a): C = scale_n * (A @ B - zp_n * rowsum(A)); A f32/bf16 [M,K], B int8 [K,N].

    workspace: "auto" (default) or a device tensor of at least
    qmm_w8_dequant_workspace_bytes(A.dtype, M, K, N) bytes runs large M on the
    SM-pair tensor-core GEMM (bf16 weight copy in the workspace) where it
    applies; None keeps the GEMV / CUDA-core kernels."""
    _need(A, (torch.float32, torch.bfloat16), "A")
    _need(B, (torch.int8,), "B")
    _need(scale, (torch.float32,), "scale")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    zp_count = 0
    if zero_point is not None:
        _need(zero_point, (torch.int32,), "zero_point")
        zp_count = zero_point.numel()
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    _need(out, (torch.float32, torch.bfloat16), "out")
    ws, wsb = _workspace(workspace, qmm_w8_dequant_workspace_bytes(A.dtype, M, K, N), A.device)
    if ws is None:
        st = _lib.qmm_w8_dequant(_ptr(A), _TORCH_TO_QMM[A.dtype], _ptr(B), M, K, N, _ptr(scale), scale.numel(),
                                 _ptr(zero_point), zp_count, _ptr(out), _TORCH_TO_QMM[out.dtype], _stream(stream))
        _check("qmm_w8_dequant", st)
    else:
        st = _lib.qmm_w8_dequant_ws(_ptr(A), _TORCH_TO_QMM[A.dtype], _ptr(B), M, K, N, _ptr(scale), scale.numel(),
                                    _ptr(zero_point), zp_count, _ptr(out), _TORCH_TO_QMM[out.dtype], _ptr(ws), wsb,
                                    _stream(stream))
        _check("qmm_w8_dequant_ws", st)
    return out


def _workspace(ws, nbytes, device):
    """None -> no workspace; "auto" -> a fresh uint8 buffer of nbytes (torch's
    caching allocator); a tensor -> used as is. Returns (tensor or None, bytes)."""
    if ws is None or nbytes == 0:
        return None, 0
    if isinstance(ws, str):
        if ws != "auto":
            raise ValueError("workspace must be None, 'auto' or a device tensor")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def qmm_a8w8_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(_lib.qmm_a8w8_workspace_bytes(M, K, N))


def matmul_integer_workspace_bytes(batch, M, K, N, a_batch_stride, b_batch_stride) -> int:
    return int(_lib.matmul_integer_workspace_bytes(batch, M, K, N, a_batch_stride, b_batch_stride))


def qmm_a8w8(A, B, act_scale, weight_scale, out=None, out_dtype=torch.bfloat16, stream=None, workspace="auto"):
    """Form (b): C = out(f32(A @ B) * act_scale[m] * weight_scale[n]); A, B int8.

    workspace: "auto" (default) or a device tensor of at least
    qmm_a8w8_workspace_bytes(M, K, N) bytes runs the two-pass path (fp16
    operand copies, then the SM-pair GEMM) where it applies; None runs the
    single-pass kernels."""
    _need(A, (torch.int8,), "A")
    _need(B, (torch.int8,), "B")
    _need(act_scale, (torch.float32,), "act_scale")
    _need(weight_scale, (torch.float32,), "weight_scale")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    _need(out, (torch.float32, torch.bfloat16), "out")
    ws, wsb = _workspace(workspace, qmm_a8w8_workspace_bytes(M, K, N), A.device)
    if ws is None:
        st = _lib.qmm_a8w8(_ptr(A), _ptr(B), M, K, N, _ptr(act_scale), act_scale.numel(), _ptr(weight_scale),
                           weight_scale.numel(), _ptr(out), _TORCH_TO_QMM[out.dtype], _stream(stream))
        _check("qmm_a8w8", st)
    else:
        st = _lib.qmm_a8w8_ws(_ptr(A), _ptr(B), M, K, N, _ptr(act_scale), act_scale.numel(), _ptr(weight_scale),
                              weight_scale.numel(), _ptr(out), _TORCH_TO_QMM[out.dtype], _ptr(ws), wsb,
                              _stream(stream))
        _check("qmm_a8w8_ws", st)
    return out


def qmm_a8w8_pack(A, B, workspace, stream=None):
    """First pass of qmm_a8w8's two-pass path: fp16 copies of A and B into workspace."""
    _need(A, (torch.int8,), "A")
    _need(B, (torch.int8,), "B")
    M, K = A.shape
    N = B.shape[1]
    st = _lib.qmm_a8w8_pack(_ptr(A), _ptr(B), M, K, N, _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream))
    _check("qmm_a8w8_pack", st)


def _need_host(t, dtypes, name):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def qmm_a8w8_host_workspace_bytes(M, K, N, act_count, w_count, out_dtype=torch.bfloat16) -> int:
    return int(_lib.qmm_a8w8_host_workspace_bytes(M, K, N, act_count, w_count, _TORCH_TO_QMM[out_dtype]))


def qmm_a8w8_host(A, B, act_scale, weight_scale, out=None, out_dtype=torch.bfloat16, stream=None,
                  workspace="auto"):
    """qmm_a8w8 on host (CPU) tensors: the copies to and from the GPU are
    pipelined with the computation (row panels of A). Pinned host tensors let
    the copies run asynchronously; the result is complete once `stream` (the
    current CUDA stream by default) has finished. workspace: "auto" or a CUDA
    uint8 tensor of at least qmm_a8w8_host_workspace_bytes(...) bytes."""
    _need_host(A, (torch.int8,), "A")
    _need_host(B, (torch.int8,), "B")
    _need_host(act_scale, (torch.float32,), "act_scale")
    _need_host(weight_scale, (torch.float32,), "weight_scale")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, pin_memory=True)
    _need_host(out, (torch.float32, torch.bfloat16), "out")
    nbytes = qmm_a8w8_host_workspace_bytes(M, K, N, act_scale.numel(), weight_scale.numel(), out.dtype)
    ws, wsb = _workspace(workspace, nbytes, torch.device("cuda", torch.cuda.current_device()))
    st = _lib.qmm_a8w8_host(_ptr(A), _ptr(B), M, K, N, _ptr(act_scale), act_scale.numel(), _ptr(weight_scale),
                            weight_scale.numel(), _ptr(out), _TORCH_TO_QMM[out.dtype], _ptr(ws), wsb,
                            _stream(stream))
    _check("qmm_a8w8_host", st)
    return out


def qmm_a8w8_packed(M, K, N, act_scale, weight_scale, workspace, out=None, out_dtype=torch.bfloat16, stream=None):
    """Second pass: the SM-pair GEMM and fused scaling on operands packed by qmm_a8w8_pack."""
    _need(act_scale, (torch.float32,), "act_scale")
    _need(weight_scale, (torch.float32,), "weight_scale")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=workspace.device)
    _need(out, (torch.float32, torch.bfloat16), "out")
    st = _lib.qmm_a8w8_packed(M, K, N, _ptr(act_scale), act_scale.numel(), _ptr(weight_scale), weight_scale.numel(),
                              _ptr(out), _TORCH_TO_QMM[out.dtype], _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check("qmm_a8w8_packed", st)
    return out


def qmm_a8w8_acc_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(_lib.qmm_a8w8_acc_workspace_bytes(M, K, N))


def qmm_a8w8_acc(A, B, act_scale=None, weight_scale=None, acc_in=None, acc_out=None, a_trans=False, b_trans=False,
                 out=None, out_dtype=torch.bfloat16, stream=None, workspace="auto"):
    """Accumulating A8W8: acc = acc_in + A @ B (int32, wrapping), then
    C = out(f32(acc) * act_scale[m] * weight_scale[n]).

    A is [M, K] ([K, M] with a_trans), B is [K, N] ([N, K] with b_trans), both
    int8; acc_in / acc_out optional int32 [M, N] (acc_out receives acc and may
    be acc_in). out_dtype None (and no out) writes only acc_out and returns None."""
    _need(A, (torch.int8,), "A")
    _need(B, (torch.int8,), "B")
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    K, M = A.shape if a_trans else A.shape[::-1]
    N, K2 = B.shape if b_trans else B.shape[::-1]
    if K2 != K:
        raise ValueError("inner dimensions differ")
    for t, name in ((acc_in, "acc_in"), (acc_out, "acc_out")):
        if t is not None:
            _need(t, (torch.int32,), name)
            if tuple(t.shape) != (M, N):
                raise ValueError(f"{name} must be [{M}, {N}]")
    if out is None and out_dtype is not None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if out is not None:
        _need(out, (torch.float32, torch.bfloat16), "out")
        _need(act_scale, (torch.float32,), "act_scale")
        _need(weight_scale, (torch.float32,), "weight_scale")
    elif acc_out is None:
        raise ValueError("nothing to write: give out_dtype/out or acc_out")
    ws, wsb = _workspace(workspace, qmm_a8w8_acc_workspace_bytes(M, K, N), A.device)
    st = _lib.qmm_a8w8_acc(_ptr(A), int(bool(a_trans)), _ptr(B), int(bool(b_trans)), M, K, N, _ptr(acc_in),
                           _ptr(acc_out), _ptr(act_scale) if out is not None else None,
                           act_scale.numel() if out is not None else 0,
                           _ptr(weight_scale) if out is not None else None,
                           weight_scale.numel() if out is not None else 0, _ptr(out),
                           _TORCH_TO_QMM[out.dtype] if out is not None else 0, _ptr(ws), wsb, _stream(stream))
    _check("qmm_a8w8_acc", st)
    return out


def _conv_geometry(x_shape, w_shape, pads, strides, dilations):
    """(N, C, H, W), (M, Cg, kH, kW) and the ctypes int64 arrays of the 2-D
    geometry; a rank-3 NCL problem becomes NC1L (unit spatial row)."""
    if len(x_shape) == 3:
        if len(w_shape) != 3:
            raise ValueError("a rank-3 input takes a rank-3 weight")
        pads = [0, 0] if pads is None else list(pads)
        strides = [1] if strides is None else list(strides)
        dilations = [1] if dilations is None else list(dilations)
        if len(pads) != 2 or len(strides) != 1 or len(dilations) != 1:
            raise ValueError("rank 3: pads [begin, end], one stride, one dilation")
        x4 = (x_shape[0], x_shape[1], 1, x_shape[2])
        w4 = (w_shape[0], w_shape[1], 1, w_shape[2])
        pads, strides, dilations = [0, pads[0], 0, pads[1]], [1, strides[0]], [1, dilations[0]]
    elif len(x_shape) == 4:
        if len(w_shape) != 4:
            raise ValueError("a rank-4 input takes a rank-4 weight")
        x4, w4 = tuple(x_shape), tuple(w_shape)
        pads = [0, 0, 0, 0] if pads is None else list(pads)
        strides = [1, 1] if strides is None else list(strides)
        dilations = [1, 1] if dilations is None else list(dilations)
        if len(pads) != 4 or len(strides) != 2 or len(dilations) != 2:
            raise ValueError("rank 4: pads [top, left, bottom, right], strides and dilations (h, w)")
    else:
        raise ValueError("ConvInteger takes rank-3 (NCL) or rank-4 (NCHW) inputs")
    arr = lambda v: (ctypes.c_int64 * len(v))(*[int(t) for t in v])  # noqa: E731
    return x4, w4, (pads, strides, dilations), (arr(pads), arr(strides), arr(dilations))


def conv_integer_workspace_bytes(x_shape, w_shape, pads=None, strides=None, dilations=None, group=1) -> int:
    x4, w4, _, (p, st, dl) = _conv_geometry(x_shape, w_shape, pads, strides, dilations)
    return int(_lib.conv_integer_workspace_bytes(*x4, w4[0], w4[2], w4[3], p, st, dl, group))


def conv_integer(x, w, x_zero_point=None, w_zero_point=None, pads=None, strides=None, dilations=None, group=1,
                 out=None, stream=None, workspace="auto"):
    """ConvInteger: y = conv(x - x_zp, w - w_zp) in int32 (wrapping), x [N,C,H,W]
    or [N,C,L], w [M,C/group,kH,kW] or [M,C/group,k], both uint8 or int8;
    x_zero_point one value (x's dtype), w_zero_point one or M values (w's
    dtype); pads in ONNX order ([top, left, bottom, right] / [begin, end])."""
    _need(x, (torch.int8, torch.uint8), "x")
    _need(w, (torch.int8, torch.uint8), "w")
    x4, w4, (pads_, strides_, dils_), (p, st, dl) = _conv_geometry(tuple(x.shape), tuple(w.shape), pads, strides,
                                                                   dilations)
    N, C, H, Wd = x4
    M, Cg, kH, kW = w4
    if Cg * group != C or M % group != 0:
        raise ValueError("channels do not divide into the groups")
    xzp = wzp = None
    if x_zero_point is not None:
        _need(x_zero_point, (x.dtype,), "x_zero_point")
        if x_zero_point.numel() != 1:
            raise ValueError("x_zero_point must be a scalar")
        xzp = x_zero_point
    if w_zero_point is not None:
        _need(w_zero_point, (w.dtype,), "w_zero_point")
        if w_zero_point.numel() not in (1, M):
            raise ValueError("w_zero_point must have 1 or M values")
        wzp = w_zero_point
    if min(strides_) >= 1 and min(dils_) >= 1:
        oH = max((H + pads_[0] + pads_[2] - dils_[0] * (kH - 1) - 1) // strides_[0] + 1, 0)
        oW = max((Wd + pads_[1] + pads_[3] - dils_[1] * (kW - 1) - 1) // strides_[1] + 1, 0)
    else:
        oH = oW = 0   # the library rejects the geometry
    shape = (N, M, oW) if x.dim() == 3 else (N, M, oH, oW)
    if out is None:
        out = torch.empty(shape, dtype=torch.int32, device=x.device)
    _need(out, (torch.int32,), "out")
    if tuple(out.shape) != shape:
        raise ValueError(f"out must be {shape}")
    ws, wsb = _workspace(workspace, conv_integer_workspace_bytes(tuple(x.shape), tuple(w.shape), pads, strides,
                                                                 dilations, group), x.device)
    st_ = _lib.conv_integer(_ptr(x), _TORCH_TO_QMM[x.dtype], _ptr(w), _TORCH_TO_QMM[w.dtype], N, C, H, Wd, M, kH, kW,
                            p, st, dl, group, _ptr(xzp), _ptr(wzp), 0 if wzp is None else wzp.numel(), _ptr(out),
                            _ptr(ws), wsb, _stream(stream))
    _check("conv_integer", st_)
    return out


def dynamic_quantize_matmul_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(_lib.dynamic_quantize_matmul_workspace_bytes(M, K, N))


def dynamic_quantize_matmul(x, W, w_scale, w_zero_point=None, bias=None, out=None, stream=None, workspace="auto"):
    """DynamicQuantizeLinear(x) -> MatMulInteger(y, W, y_zp, w_zp) -> fp32 cast,
    times y_scale * w_scale[n], plus bias[n]: C float32 [M, N] from x float32
    [M, K] and W int8/uint8 [K, N]. Returns (C, y_scale [1], y_zero_point [1])."""
    _need(x, (torch.float32,), "x")
    _need(W, (torch.int8, torch.uint8), "W")
    _need(w_scale, (torch.float32,), "w_scale")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[0]:
        raise ValueError("x [M, K] and W [K, N] expected")
    M, K = x.shape
    N = W.shape[1]
    if w_scale.numel() not in (1, N):
        raise ValueError("w_scale must have 1 or N values")
    if w_zero_point is not None:
        _need(w_zero_point, (W.dtype,), "w_zero_point")
        if w_zero_point.numel() not in (1, N):
            raise ValueError("w_zero_point must have 1 or N values")
    if bias is not None:
        _need(bias, (torch.float32,), "bias")
        if bias.numel() != N:
            raise ValueError("bias must have N values")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, (torch.float32,), "out")
    ys = torch.empty(1, dtype=torch.float32, device=x.device)
    yz = torch.empty(1, dtype=torch.uint8, device=x.device)
    ws, wsb = _workspace(workspace, dynamic_quantize_matmul_workspace_bytes(M, K, N), x.device)
    st = _lib.dynamic_quantize_matmul(_ptr(x), M, K, _ptr(W), _TORCH_TO_QMM[W.dtype], N, _ptr(w_scale),
                                      w_scale.numel(), _ptr(w_zero_point),
                                      0 if w_zero_point is None else w_zero_point.numel(), _ptr(bias), _ptr(out),
                                      _ptr(ys), _ptr(yz), _ptr(ws), wsb, _stream(stream))
    _check("dynamic_quantize_matmul", st)
    return out, ys, yz


class DqmPackedWeight(NamedTuple):
    """A weight packed once for dynamic_quantize_matmul_packed: the device
    buffer (exact fp16 copy and column sums) and the extents and dtype it was
    packed with."""
    buf: torch.Tensor
    K: int
    N: int
    dtype: torch.dtype


def dynamic_quantize_matmul_weight_bytes(K: int, N: int) -> int:
    return int(_lib.dynamic_quantize_matmul_weight_bytes(K, N))


def dynamic_quantize_matmul_packed_workspace_bytes(M: int, K: int) -> int:
    return int(_lib.dynamic_quantize_matmul_packed_workspace_bytes(M, K))


def dynamic_quantize_matmul_pack_weight(W, packed=None, stream=None) -> DqmPackedWeight:
    """Pack a frozen int8/uint8 weight W [K, N] once for the fused chain."""
    _need(W, (torch.int8, torch.uint8), "W")
    if W.dim() != 2:
        raise ValueError("W [K, N] expected")
    K, N = W.shape
    nbytes = dynamic_quantize_matmul_weight_bytes(K, N)
    if nbytes == 0:
        raise QmmError("dynamic_quantize_matmul_pack_weight", QMM_ERR_INVALID_ARG)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _check("dynamic_quantize_matmul_pack_weight",
           _lib.dynamic_quantize_matmul_pack_weight(_ptr(W), _TORCH_TO_QMM[W.dtype], K, N, _ptr(packed),
                                                    packed.numel() * packed.element_size(), _stream(stream)))
    return DqmPackedWeight(packed, K, N, W.dtype)


def dynamic_quantize_matmul_packed(x, weight: DqmPackedWeight, w_scale, w_zero_point=None, bias=None, out=None,
                                   stream=None, workspace="auto"):
    """dynamic_quantize_matmul on a weight packed by
    dynamic_quantize_matmul_pack_weight: the same results, bit for bit."""
    _need(x, (torch.float32,), "x")
    _need(w_scale, (torch.float32,), "w_scale")
    M, K = x.shape if x.dim() == 2 else (None, None)
    if M is None or K != weight.K:
        raise ValueError("x [M, K] expected, K as packed")
    N = weight.N
    if w_scale.numel() not in (1, N):
        raise ValueError("w_scale must have 1 or N values")
    zc = 0
    if w_zero_point is not None:
        _need(w_zero_point, (weight.dtype,), "w_zero_point")
        zc = w_zero_point.numel()
    if bias is not None:
        _need(bias, (torch.float32,), "bias")
        if bias.numel() != N:
            raise ValueError("bias must have N values")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(out, (torch.float32,), "out")
    ys = torch.empty(1, dtype=torch.float32, device=x.device)
    yz = torch.empty(1, dtype=torch.uint8, device=x.device)
    nbytes = dynamic_quantize_matmul_packed_workspace_bytes(M, K)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    if workspace is None:
        raise ValueError("the packed chain needs a workspace")
    buf = weight.buf
    st = _lib.dynamic_quantize_matmul_packed(_ptr(x), M, K, _ptr(buf), buf.numel() * buf.element_size(),
                                             _TORCH_TO_QMM[weight.dtype], N, _ptr(w_scale), w_scale.numel(),
                                             _ptr(w_zero_point), zc, _ptr(bias), _ptr(out), _ptr(ys), _ptr(yz),
                                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                                             _stream(stream))
    _check("dynamic_quantize_matmul_packed", st)
    return out, ys, yz


def matmul_integer(A, B, a_zero_point=None, b_zero_point=None, out=None, stream=None, workspace="auto"):
    """Form (c): int32 C = (A - a_zp) @ (B - b_zp), A [...,M,K], B [K,N] (shared) or [...,K,N].

    workspace: as for qmm_a8w8 (None: single pass; "auto" or a tensor: two-pass
    path with precomputed row/column sums where it applies)."""
    _need(A, (torch.int8, torch.uint8), "A")
    _need(B, (torch.int8, torch.uint8), "B")
    if A.dim() < 2 or A.dim() > 4 or B.dim() < 2 or B.dim() > 4:
        raise ValueError("MatMulInteger takes ranks 2 to 4")
    M, K = A.shape[-2:]
    K2, N = B.shape[-2:]
    if K2 != K:
        raise ValueError("inner dimensions differ")
    a_batch = A.shape[:-2]
    b_batch = B.shape[:-2]
    shared_b = all(d == 1 for d in b_batch)
    batch_shape = torch.broadcast_shapes(a_batch, b_batch)
    batch = 1
    for d in batch_shape:
        batch *= d
    if shared_b:
        b_stride = 0
    elif tuple(b_batch) == tuple(batch_shape):
        b_stride = K * N
    else:
        raise ValueError("B batch dims must be all 1 or equal to the result's batch dims")
    a_count = 1
    for d in a_batch:
        a_count *= d
    if a_count == 1:
        a_stride = 0
    elif tuple(a_batch) == tuple(batch_shape):
        a_stride = M * K
    else:
        raise ValueError("A batch dims must be all 1 or equal to the result's batch dims")
    az = bz = 0
    if a_zero_point is not None:
        _need(a_zero_point, (A.dtype,), "a_zero_point")
        az = a_zero_point.numel()
    if b_zero_point is not None:
        _need(b_zero_point, (B.dtype,), "b_zero_point")
        bz = b_zero_point.numel()
    if out is None:
        out = torch.empty((*batch_shape, M, N), dtype=torch.int32, device=A.device)
    _need(out, (torch.int32,), "out")
    ws, wsb = _workspace(workspace, matmul_integer_workspace_bytes(batch, M, K, N, a_stride, b_stride), A.device)
    if ws is None:
        st = _lib.matmul_integer(_ptr(A), _TORCH_TO_QMM[A.dtype], _ptr(B), _TORCH_TO_QMM[B.dtype], batch, M, K, N,
                                 a_stride, b_stride, _ptr(a_zero_point), az, _ptr(b_zero_point), bz, _ptr(out),
                                 _stream(stream))
        _check("matmul_integer", st)
    else:
        st = _lib.matmul_integer_ws(_ptr(A), _TORCH_TO_QMM[A.dtype], _ptr(B), _TORCH_TO_QMM[B.dtype], batch, M, K,
                                    N, a_stride, b_stride, _ptr(a_zero_point), az, _ptr(b_zero_point), bz,
                                    _ptr(out), _ptr(ws), wsb, _stream(stream))
        _check("matmul_integer_ws", st)
    return out


def dynamic_quantize_linear_workspace_bytes(n: int) -> int:
    return int(_lib.dynamic_quantize_linear_workspace_bytes(n))


def dynamic_quantize_linear(x, row_len=None, workspace=None, y=None, stream=None):
    """Form (d): (y uint8, y_scale f32[1], y_zero_point u8[1][, row_sums int32]) of float32 x.

    With row_len, also returns the sum of each run of row_len elements of y."""
    _need(x, (torch.float32,), "x")
    n = x.numel()
    dev = x.device
    if y is None:
        y = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    y_scale = torch.empty(1, dtype=torch.float32, device=dev)
    y_zp = torch.empty(1, dtype=torch.uint8, device=dev)
    ws_bytes = dynamic_quantize_linear_workspace_bytes(n)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    row_sums = None
    rl = 0
    if row_len is not None:
        rl = int(row_len)
        row_sums = torch.empty(n // rl if rl > 0 else 0, dtype=torch.int32, device=dev)
    st = _lib.dynamic_quantize_linear(_ptr(x), n, _ptr(y), _ptr(y_scale), _ptr(y_zp), _ptr(row_sums), rl,
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream))
    _check("dynamic_quantize_linear", st)
    if row_sums is not None:
        return y, y_scale, y_zp, row_sums
    return y, y_scale, y_zp


def num_sms() -> int:
    return int(_lib.qmm_num_sms())


__all__ = [
    "qmm_w8_dequant", "qmm_a8w8", "qmm_a8w8_acc", "matmul_integer", "conv_integer", "dynamic_quantize_matmul",
    "dynamic_quantize_matmul_pack_weight", "dynamic_quantize_matmul_packed", "DqmPackedWeight",
    "dynamic_quantize_linear",
    "dynamic_quantize_linear_workspace_bytes", "last_kernel", "check_device_error", "QmmError", "lib",
    "num_sms", "LIB_PATH",
]
