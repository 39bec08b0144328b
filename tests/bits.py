"""Bit-pattern conversions for tests (numpy / torch views, no normalization math).

These are independent of the oracle's own IEEE helpers: binary16 goes through
numpy's float16 type, bfloat16 through a 16-bit shift into binary32 or through
torch's bfloat16 type.
"""
import numpy as np
import torch


def f16_bits_to_f64(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):  # NaN payloads widen as NaN
        return b.view(np.float32).astype(np.float64)


def bits_to_f64(dt, a):
    if dt == 0:
        return np.asarray(a, np.float32).astype(np.float64)
    if dt == 1:
        return f16_bits_to_f64(a)
    return bf16_bits_to_f64(a)


def torch_to_np(t: torch.Tensor):
    """CPU tensor -> numpy array in the oracle's convention (f32 or raw uint16)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def np_to_torch(a, dtype: torch.dtype):
    a = np.ascontiguousarray(a)
    if dtype == torch.float32:
        return torch.from_numpy(a.astype(np.float32))
    return torch.from_numpy(a.view(np.int16).copy()).view(dtype)


def dt_code(dtype: torch.dtype) -> int:
    return {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[dtype]


def f64_to_bits_numpy_f16(v):
    """Independent RN-even double -> binary16 (numpy's conversion)."""
    with np.errstate(over="ignore", invalid="ignore"):  # out of range rounds to infinity
        return np.asarray(v, np.float64).astype(np.float16).view(np.uint16)


def f32_to_bits_torch_bf16(v):
    """Independent RN-even binary32 -> bfloat16 (torch's conversion)."""
    t = torch.from_numpy(np.asarray(v, np.float32).copy()).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def ordered(dt, bits):
    """Map bit patterns to integers whose order is the numeric order (ulp distance)."""
    if dt == 0:
        i = np.asarray(bits, np.float32).view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    i = np.asarray(bits, np.uint16).astype(np.int64)
    return np.where(i & 0x8000, -(i & 0x7FFF), i)


def ulp_diff(dt, a, b):
    return np.abs(ordered(dt, a) - ordered(dt, b))
