"""Shared test helpers: moving seeded numpy inputs to the device and back."""
import numpy as np
import torch


def dev():
    return torch.device("cuda:0")


def bf16_dev(a_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).to(dev())


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_bf16_values(u: np.ndarray) -> np.ndarray:
    """Float64 values of BF16 bit patterns read back from the device (decoded
    here, so that no device output passes through the oracle)."""
    bits = np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def np_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bf16_ulp(ref_f64: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |ref| (2^-7 relative, subnormal floor)."""
    a = np.abs(np.asarray(ref_f64, dtype=np.float64))
    _, e = np.frexp(a)
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def assert_bf16_within_one_ulp(got_u16, exact_f64, what=""):
    """BF16 output within 1 BF16 ulp of the correctly rounded exact result."""
    from oracle import nvfp4_moe_oracle as O
    ref = O.bf16_to_f32(O.f64_to_bf16(exact_f64)).astype(np.float64)
    got = gpu_bf16_values(got_u16)
    ulp = np.maximum(bf16_ulp(ref), bf16_ulp(got))
    bad = np.abs(got - ref) > ulp
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside 1 BF16 ulp; worst " \
        f"{np.abs(got - ref)[bad].max() if bad.any() else 0}"


def assert_fp32_within_bound(got_f32, exact_f64, abs_sum, what=""):
    """|y_gpu - y| <= 2^-20 * sum_k |a_k b_k|."""
    err = np.abs(np.asarray(got_f32, dtype=np.float64) - exact_f64)
    lim = 2.0 ** -20 * abs_sum
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond 2^-20 sum|ab|; worst ratio " \
        f"{(err / np.maximum(abs_sum, 1e-300)).max() * 2**20:.3f} x bound"
