"""A8W8 from host buffers (qmm_a8w8_host): the copies in and out overlap the
GEMMs (2 x 2 blocks from 512 rows and 1024 columns on, with pitched copies of
B's column panels and C's blocks; row panels below that); the result must be
bit-identical to the oracle and to the device-pointer call, with ragged last
panels, both output types, scalar scales, pageable host memory, back-to-back
calls on one workspace, and the shapes outside the two-pass path."""
import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, gemm_kernel, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")

PIPELINED = "h2d_pipelined+f16_prepass+gemm_tc05_pair_f16ops_a8w8"
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def host_call(w, out, pinned=True, workspace="auto", act=None, wsc=None):
    act = w.act_scale if act is None else act
    wsc = w.weight_scale if wsc is None else wsc
    ts = [torch.from_numpy(np.ascontiguousarray(a)) for a in (w.A, w.B, act, wsc)]
    if pinned:
        ts = [t.pin_memory() for t in ts]
    C = q.qmm_a8w8_host(*ts, out_dtype=DT[out], workspace=workspace)
    torch.cuda.synchronize()
    q.check_device_error()
    return host(C)


@pytest.mark.parametrize("M,K,N", [(2600, 128, 4096), (1000, 1040, 1008), (256, 64, 256), (1000, 1040, 1040),
                                   (600, 2064, 1024)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_host_pipeline_matches_oracle(M, K, N, out):
    w = W.a8w8(M, K, N, seed=M + K + N)
    got = host_call(w, out)
    assert q.last_kernel() == PIPELINED
    assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, out), f"host A8W8 {out} {M}x{K}x{N}")


def test_host_pipeline_equals_device_call_and_reuses_its_workspace():
    M, K, N = 2600, 192, 4096
    ws = torch.empty(q.qmm_a8w8_host_workspace_bytes(M, K, N, M, N), dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        w = W.a8w8(M, K, N, seed=seed)
        got = host_call(w, "bf16", workspace=ws)
        ref = host(q.qmm_a8w8(dev(w.A), dev(w.B), dev(w.act_scale), dev(w.weight_scale), out_dtype=torch.bfloat16))
        assert np.array_equal(got, ref), f"host call differs from the device call (seed {seed})"


def test_host_pipeline_scalar_scales_and_pageable_memory():
    w = W.a8w8(1300, 96, 4096, seed=9)
    one = np.array([0.0125], np.float32)
    got = host_call(w, "f32", pinned=False, act=one, wsc=one)
    assert q.last_kernel() == PIPELINED
    assert_equal(got, O.a8w8(w.A, w.B, one, one, "f32"), "scalar scales, pageable host buffers")


@pytest.mark.parametrize("M,K,N", [(100, 64, 64), (300, 40, 64)])
def test_host_call_outside_the_two_pass_path(M, K, N):
    w = W.a8w8(M, K, N, seed=3)
    got = host_call(w, "bf16")
    assert q.last_kernel() == gemm_kernel("a8w8", M, K, N)
    assert_equal(got, O.a8w8(w.A, w.B, w.act_scale, w.weight_scale, "bf16"), "host call, single-pass kernel")


def test_host_call_rejects_device_tensors_and_small_workspace():
    w = W.a8w8(256, 64, 256, seed=4)
    with pytest.raises(ValueError):
        q.qmm_a8w8_host(dev(w.A), torch.from_numpy(w.B), torch.from_numpy(w.act_scale),
                        torch.from_numpy(w.weight_scale))
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        q.qmm_a8w8_host(*(torch.from_numpy(np.ascontiguousarray(a)) for a in (w.A, w.B, w.act_scale,
                                                                           w.weight_scale)), workspace=small)
