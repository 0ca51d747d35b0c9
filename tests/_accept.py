"""Acceptance bound for floating-point parity and shared test helpers.

Per element: |C - C_ref| <= 4e-3 * |C_ref| + 1e-5 * T, where C_ref is the
oracle's fp64 value and T = sum_k |sA*A*sB*B| its magnitude sum.  The first
term covers the bf16 output rounding (at most 2^-9 relative) and the second the
fp32 accumulation over K.
"""
import numpy as np
import torch

REL = 4e-3
ABS_T = 1e-5


def bf16_to_f64(c: torch.Tensor) -> np.ndarray:
    return c.float().cpu().numpy().astype(np.float64)


# what -> (worst, mean, elements) of |C - C_ref| / bound, for the session summary
REPORT: dict = {}


def check(C_gpu: np.ndarray, C_ref: np.ndarray, T: np.ndarray, what: str = ""):
    err = np.abs(C_gpu - C_ref)
    bound = REL * np.abs(C_ref) + ABS_T * T
    bad = ~(err <= bound)
    r = err / np.maximum(bound, 1e-300)
    ratio = float(np.max(r)) if err.size else 0.0
    if err.size:
        REPORT[what] = (ratio, float(np.mean(r)), int(err.size))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = [f"{what}: {int(bad.sum())}/{bad.size} elements outside the bound; worst ratio {ratio:.3g}"]
        for i in idx:
            i = tuple(i)
            msg.append(f"  at {i}: gpu={C_gpu[i]!r} ref={C_ref[i]!r} T={T[i]!r}")
        raise AssertionError("\n".join(msg))
    return ratio
