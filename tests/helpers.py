"""Small conversions shared by the tests (no arithmetic of the forward here)."""
from __future__ import annotations

import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """A CPU numpy view of a tensor's bits: bf16 -> uint16, e4m3 -> uint8, others as is."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def bf16_from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.bfloat16)


def e4m3_from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn)


def f64(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> float64 values (exact)."""
    return bf16_from_bits(b).double().numpy()


def rms(a: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def parse_golden(path) -> list[str]:
    return [ln.split("#", 1)[0].strip() for ln in open(path) if ln.split("#", 1)[0].strip()]


def dev_bf16(b: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bits (uint16) -> a bf16 tensor on the device."""
    return bf16_from_bits(b).to(device)


def dev_e4m3(b: np.ndarray, device="cuda") -> torch.Tensor:
    return e4m3_from_bits(b).to(device)


def sentinel_like(shape, dtype, device="cuda") -> torch.Tensor:
    """A tensor whose every byte is 0xA5, to detect writes past the valid rows."""
    t = torch.empty(shape, dtype=dtype, device=device)
    t.view(torch.uint8).fill_(0xA5)
    return t


def is_sentinel(t: torch.Tensor) -> bool:
    return bool((t.contiguous().view(torch.uint8) == 0xA5).all())


def e4m3_step_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in code steps between e4m3 codes of the same sign (large if signs differ)."""
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    same = ((a & 0x80) == (b & 0x80)) | ((a & 0x7F) == 0) | ((b & 0x7F) == 0)
    mag = np.abs((a & 0x7F) - (b & 0x7F))
    return np.where(same, mag, 1000)
