"""DynamicQuantizeLinear (form (d)) through the C ABI: the uint8 output, the
scale and the zero point must equal the oracle's bit for bit (every float step
is one IEEE operation in the same precision on both sides)."""
import json
import os

import numpy as np
import pytest
import torch

import qmm_workloads as W
from oracle import qmm_oracle as O
from _helpers import assert_equal, dev, host

pytestmark = pytest.mark.gpu
q = pytest.importorskip("quantized_int8_matmul_gb300")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(x, row_len=None):
    r = q.dynamic_quantize_linear(dev(x), row_len=row_len)
    torch.cuda.synchronize()
    return [host(t) for t in r]


def check(x, what):
    y, s, zp = run(x)
    wy, ws, wzp = O.dynamic_quantize_linear(x)
    assert s.view(np.uint32)[0] == np.float32(ws).view(np.uint32), f"{what}: scale {s[0]!r} vs {ws!r}"
    assert int(zp[0]) == int(wzp), f"{what}: zero point"
    assert_equal(y.reshape(-1), wy.reshape(-1), what)


@pytest.mark.parametrize("name", ["dql_all_zero.json", "dql_hand_worked.json", "dql_ties.json"])
def test_golden(name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    x = np.array(g["x"], np.float32)
    y, s, zp = run(x)
    assert y.tolist() == g["y"] and int(zp[0]) == g["zero_point"]
    if "scale" in g:
        assert float(s[0]) == g["scale"]
    else:
        assert int(s.view(np.uint32)[0]) == g["scale_f32_bits"]


def test_golden_one_sided():
    for c in json.load(open(os.path.join(GOLDEN, "dql_one_sided.json")))["cases"]:
        y, _, zp = run(np.array(c["x"], np.float32))
        assert y.tolist() == c["y"] and int(zp[0]) == c["zero_point"]


@pytest.mark.parametrize("n", [1, 3, 4, 1000, 65537, 1000003])
def test_random_with_outliers(n):
    rng = np.random.default_rng(n)
    x = W.with_outliers(rng, W.normal_f32(rng, (n,)), 0.001, 20.0)
    check(x, f"n={n}")


def test_nonnegative_and_nonpositive_inputs():
    rng = np.random.default_rng(1)
    x = np.abs(W.normal_f32(rng, (50000,)))
    check(x, "non-negative")
    check(-x, "non-positive")


def test_misaligned_input_takes_the_scalar_path():
    rng = np.random.default_rng(2)
    base = torch.from_numpy(W.normal_f32(rng, (40001,))).cuda()
    xs = base[1:]                       # 4-byte offset: not 16-byte aligned
    y, s, zp = q.dynamic_quantize_linear(xs)
    wy, ws, wzp = O.dynamic_quantize_linear(xs.cpu().numpy())
    assert float(s.item()) == float(ws) and int(zp.item()) == int(wzp)
    assert_equal(host(y), wy, "misaligned")


def test_row_sums():
    rng = np.random.default_rng(3)
    x = W.with_outliers(rng, W.normal_f32(rng, (96, 1000)), 0.001, 20.0)
    y, s, zp, rs = run(x, row_len=1000)
    wy, ws, wzp = O.dynamic_quantize_linear(x)
    assert_equal(y, wy, "y")
    assert_equal(rs, O.row_sums(wy, 1000), "row sums")
    assert q.last_kernel() == "dql_minmax+dql_quantize_rows"


def test_empty_input():
    x = torch.empty(0, dtype=torch.float32, device="cuda")
    y, s, zp = q.dynamic_quantize_linear(x)
    assert float(s.item()) == 1.0 and int(zp.item()) == 0 and y.numel() == 0


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_quotients_near_halfway(seed):
    """x/scale lands within a few ulps of k + 1/2: the rounded quotient decides the byte."""
    rng = np.random.default_rng(100 + seed)
    lo, hi = -np.float32(rng.uniform(0.1, 50)), np.float32(rng.uniform(0.1, 50))
    scale = np.float32(np.float32(hi - lo) / np.float32(255))
    k = rng.integers(-200, 200, 200000).astype(np.float32)
    base = ((k + np.float32(0.5)) * scale).astype(np.float32)
    ulps = rng.integers(-3, 4, base.size).astype(np.int32)
    x = (base.view(np.int32) + ulps).view(np.float32)
    x = np.clip(x, lo, hi).astype(np.float32)
    x[:2] = [lo, hi]
    check(x, f"near-halfway seed={seed}")


@pytest.mark.parametrize("log2_scale", [-125, -112, -101, -99, 60])
def test_quotients_near_halfway_at_extreme_scales(log2_scale):
    """Ranges around 255 * 2^log2_scale: scales whose reciprocal is above 2^100
    are divided by IEEE division, the rest by the corrected reciprocal; either
    way every byte, the scale and the zero point equal the oracle's."""
    rng = np.random.default_rng(200 - log2_scale)
    width = np.float32(np.ldexp(255.0 * rng.uniform(1.0, 1.9), log2_scale))
    lo = -np.float32(width * np.float32(rng.uniform(0.2, 0.8)))
    hi = np.float32(width + lo)
    scale = np.float32(np.float32(hi - lo) / np.float32(255))
    k = rng.integers(-250, 250, 100000).astype(np.float64)
    base = ((k + 0.5) * np.float64(scale)).astype(np.float32)
    x = (base.view(np.int32) + rng.integers(-3, 4, base.size).astype(np.int32)).view(np.float32)
    x = np.clip(x, lo, hi).astype(np.float32)
    x[:2] = [lo, hi]
    check(x, f"near-halfway 2^{log2_scale}")
