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


def bf16_step(v: np.ndarray) -> np.ndarray:
    """One bf16 step (unit in the last place) at each value."""
    a = np.abs(np.asarray(v, np.float64))
    return np.exp2(np.floor(np.log2(np.where(a > 0, a, 1e-38))) - 7)


def assert_forward_close(got: np.ndarray, exp: np.ndarray, tol: float, label: str = "") -> dict:
    """The end-to-end output bound against the oracle: every element within
    tol * rms(exp) plus one bf16 step of its expected value, and the strict
    bound tol * rms(exp) met on at least 99.9% of the elements.  The achieved
    figures are printed and, when the environment names a file in
    MOE_PARITY_LOG, appended to it as one JSON line."""
    import json
    import os

    got = np.asarray(got, np.float64)
    exp = np.asarray(exp, np.float64)
    err = np.abs(got - exp)
    r = rms(exp)
    bound = tol * r
    strict = err <= bound
    stats = {"label": label, "elements": int(err.size), "tol_rms": tol,
             "max_err_rms": float(err.max() / r) if err.size and r > 0 else 0.0,
             "strict_fraction": float(strict.mean()) if err.size else 1.0,
             "over_strict": int((~strict).sum()), "exact_fraction": float((err == 0).mean()) if err.size else 1.0}
    print(f"parity {label}: max|err| = {stats['max_err_rms']:.4f} rms (bound {tol:g}); strict bound on "
          f"{stats['strict_fraction']:.6f} of {stats['elements']} elements ({stats['over_strict']} above it); "
          f"bit-identical {stats['exact_fraction']:.4f}")
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(stats) + "\n")
    msg = f"{label}: max|err| {stats['max_err_rms']:.4f} rms; strict bound met on {stats['strict_fraction']:.5f}"
    assert np.all(err <= bound + bf16_step(exp)), msg
    assert stats["strict_fraction"] >= 0.999, msg
    return stats
