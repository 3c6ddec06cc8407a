"""dynamic_quantize_linear_noalloc: the DynamicQuantizeLinear entry point for
callers that cannot allocate device memory (a plugin inside a framework that
owns all device memory, an engine with memory fixed at start-up, a thread that
must not call cudaMalloc). It keeps its partials in a fixed array inside the
library instead of a caller workspace, so these tests check, through the C
ABI, that two calls in a row give exactly what the workspace entry point gives
-- the second call must not be affected by what the first left in the shared
array -- and that both equal the CPU oracle byte for byte. This file is
collected last on purpose."""
import ctypes
import json
import os

import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")


def _fn():
    f = q.lib().dynamic_quantize_linear_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [vp, i64, vp, vp, vp, vp, i64, vp]
    f.restype = ctypes.c_int
    return f


def noalloc(x, row_len=None):
    n = x.numel()
    y = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty(1, dtype=torch.float32, device=x.device)
    zp = torch.empty(1, dtype=torch.uint8, device=x.device)
    rs = None if row_len is None else torch.empty(n // row_len, dtype=torch.int32, device=x.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = _fn()(ctypes.c_void_p(x.data_ptr()), n, ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(s.data_ptr()),
               ctypes.c_void_p(zp.data_ptr()), None if rs is None else ctypes.c_void_p(rs.data_ptr()),
               0 if row_len is None else row_len, stream)
    assert st == 0, q.lib().qmm_status_string(st)
    return y, s, zp, rs


def inputs():
    rng = np.random.default_rng(21)
    big = W.with_outliers(rng, W.normal_f32(rng, (4096, 4096)), 0.001, 20.0)   # 512 partials
    small = np.float32(0.01) * W.normal_f32(rng, (37, 1000))                  # 2 partials, narrow range
    return torch.from_numpy(big).cuda(), torch.from_numpy(small).cuda()


def check_oracle(x, y, s, zp, rs=None, row_len=None):
    """The bytes, the scale's bits, the zero point (and the row sums) equal the oracle's."""
    xh = x.cpu().numpy()
    wy, ws, wzp = O.dynamic_quantize_linear(xh)
    assert s.cpu().numpy().view(np.uint32)[0] == np.float32(ws).view(np.uint32)
    assert int(zp.item()) == int(wzp)
    assert np.array_equal(y.cpu().numpy().reshape(-1), wy.reshape(-1))
    if rs is not None:
        assert np.array_equal(rs.cpu().numpy(), O.row_sums(wy.reshape(-1), row_len))


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    xs = inputs()
    got = [noalloc(x) for x in xs]           # two no-alloc calls back to back
    torch.cuda.synchronize()
    for x, (y, s, zp, _) in zip(xs, got):
        wy, ws, wzp = q.dynamic_quantize_linear(x)
        torch.cuda.synchronize()
        assert torch.equal(s, ws) and torch.equal(zp, wzp)
        assert torch.equal(y, wy)
        check_oracle(x, y, s, zp)


def test_ties_to_even_through_the_no_alloc_entry_point():
    """The page's ties-to-even rule on the zero point (-lo/scale = 2.5 -> 2) and
    on the quotients, after a large call has filled the shared array."""
    big, _ = inputs()
    noalloc(big)
    with open(os.path.join(os.path.dirname(__file__), "golden", "dql_ties.json")) as f:
        g = json.load(f)
    x = torch.tensor(g["x"], dtype=torch.float32, device="cuda")
    y, s, zp, _ = noalloc(x)
    torch.cuda.synchronize()
    assert y.cpu().tolist() == g["y"] and int(zp.item()) == g["zero_point"] and float(s.item()) == g["scale"]
    check_oracle(x, y, s, zp)


def test_two_calls_in_a_row_with_row_sums():
    xs = inputs()
    got = [noalloc(x, row_len=x.shape[1]) for x in xs]
    torch.cuda.synchronize()
    for x, (y, s, zp, rs) in zip(xs, got):
        wy, ws, wzp, wrs = q.dynamic_quantize_linear(x, row_len=x.shape[1])
        torch.cuda.synchronize()
        assert torch.equal(s, ws) and torch.equal(zp, wzp)
        assert torch.equal(y, wy) and torch.equal(rs, wrs)
        check_oracle(x, y, s, zp, rs, x.shape[1])


def test_rejects_malformed_arguments():
    x = torch.zeros(10, device="cuda")
    f = _fn()
    p = ctypes.c_void_p(x.data_ptr())
    assert f(p, -1, p, p, p, None, 0, None) == q.QMM_ERR_INVALID_ARG
    assert f(None, 10, p, p, p, None, 0, None) == q.QMM_ERR_INVALID_ARG
    assert f(p, 10, p, p, p, p, 3, None) == q.QMM_ERR_INVALID_ARG     # 10 % 3 != 0
