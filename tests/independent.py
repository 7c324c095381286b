"""Independent restatements used only to pin the oracle.

These are deliberately different algorithms from the oracle's: the encoders
here are exhaustive nearest-value searches over the golden code tables
(every code's distance computed, the minimum taken, ties broken toward the
even code), vectorised in numpy; e4m3 and bf16 conversions come from torch's
own casts.  The oracle never imports this module.
"""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str):
    """Rows of a golden text fixture as lists of strings (comments dropped)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def e2m1_table() -> np.ndarray:
    """float64[16]: value of each e2m1 code, from the MX golden table."""
    t = np.zeros(16, np.float64)
    for code, val in read_golden("e2m1_values.txt"):
        t[int(code, 16)] = float(val)
    return t


def e4m3_table() -> np.ndarray:
    """float64[256]: value of each e4m3 code, from torch's float8_e4m3fn."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _nearest_even(x: np.ndarray, mags: np.ndarray) -> np.ndarray:
    """Index of the nearest magnitude for each |x| (exhaustive), ties to the
    even index; values above the largest magnitude take the largest."""
    a = np.abs(x.astype(np.float64))[:, None]
    d = np.abs(a - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    is_best = d == best
    # among the tied minima prefer an even index (there are at most two)
    even = is_best & (np.arange(mags.size)[None, :] % 2 == 0)
    idx = np.where(even.any(axis=1), even.argmax(axis=1), is_best.argmax(axis=1))
    idx = np.where(a[:, 0] >= mags[-1], mags.size - 1, idx)
    return idx


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Brute-force e2m1 round-to-nearest-even with satfinite (finite x)."""
    x = np.asarray(x, np.float32).ravel()
    mags = e2m1_table()[:8]
    out = np.empty(x.size, np.uint8)
    for s in range(0, x.size, 1 << 20):      # bound the [n, 8] temporaries
        xs = x[s:s + (1 << 20)]
        out[s:s + xs.size] = _nearest_even(xs, mags).astype(np.uint8) | (np.signbit(xs).astype(np.uint8) << 3)
    return out


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Brute-force e4m3 round-to-nearest-even with satfinite (finite x)."""
    x = np.asarray(x, np.float32).ravel()
    mags = e4m3_table()[:127]
    out = np.empty(x.size, np.uint8)
    for s in range(0, x.size, 1 << 16):      # bound the [n, 127] temporaries
        xs = x[s:s + (1 << 16)]
        idx = _nearest_even(xs, mags)
        out[s:s + xs.size] = idx.astype(np.uint8) | (np.signbit(xs).astype(np.uint8) << 7)
    return out


def torch_e4m3_bits(x_f32: torch.Tensor) -> torch.Tensor:
    """torch's float32 -> float8_e4m3fn cast, as uint8 bits (no saturation:
    |x| >= 464 gives NaN)."""
    return x_f32.to(torch.float8_e4m3fn).view(torch.uint8)


def torch_bf16_bits(x_f32: torch.Tensor) -> np.ndarray:
    return x_f32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """[..., n] bytes -> [..., 2n] codes, low nibble first."""
    lo = packed & 0x0F
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
