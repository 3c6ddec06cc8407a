"""Helpers for the GPU parity tests: moving arrays between numpy and the device,
and the elementwise tolerance checks. No method arithmetic lives here."""
import numpy as np
import torch


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def half_ulp(x: np.ndarray, mant_bits: int) -> np.ndarray:
    """Half a unit in the last place of |x| for a binary format with `mant_bits`
    stored mantissa bits (bf16: 7, f32: 23): the rounding any output cast may add."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - mant_bits - 1).astype(np.int64))


def assert_within(got: np.ndarray, exact: np.ndarray, bound: np.ndarray, out_mant_bits: int, what: str):
    err = np.abs(got.astype(np.float64) - exact)
    allowed = bound + half_ulp(exact, out_mant_bits)
    bad = err > allowed
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r}, exact {exact[tuple(i)]!r}, allowed {allowed[tuple(i)]!r}")


def assert_equal(got: np.ndarray, want: np.ndarray, what: str):
    if got.shape != want.shape:
        raise AssertionError(f"{what}: shape {got.shape} != {want.shape}")
    bad = got != want
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} elements differ; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r}, want {want[tuple(i)]!r}")


def gemm_kernel(form: str, M: int, K: int, N: int) -> str:
    """Name of the exact-GEMM kernel the library is expected to launch: the SM-pair
    kernel for 16-byte-aligned rows and M >= 256 (M after folding a batch), the
    single-SM TMA kernel for other aligned shapes, the byte-wise one otherwise."""
    vec = K % 16 == 0 and N % 16 == 0
    if vec and M >= 256:
        return f"gemm_tc05_pair_exact_{form}"
    return f"gemm_tc05_exact_{form}" + ("" if vec else "_bytewise")
