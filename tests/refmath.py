"""Independent checkers used to pin the oracle.

Nothing here shares code with ``oracle/`` or with the CUDA library.  The helpers
are brute force or exact-rational definitions, or call library routines:

* ``fp8_code_values(fmt)``: the value of every fp8 code as decoded by torch's
  float8 dtypes (a library routine).
* ``fp8_nearest(x, fmt)``: round-to-nearest-even with saturation by brute force
  -- for every input, the finite code at the smallest distance, the even
  mantissa on a tie, the sign of the input on zero, 0x7F for any NaN.
* ``bf16_round_exact(x)``: the bf16 value nearest to each double, found by
  comparing exact rationals (``fractions.Fraction``) against neighbouring bf16
  candidates; ties go to the even pattern.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

BF16, FP8_E4M3, FP8_E5M2 = 0, 1, 2
_TORCH_FP8 = {FP8_E4M3: torch.float8_e4m3fn, FP8_E5M2: torch.float8_e5m2}
FP8_MAX = {FP8_E4M3: 448.0, FP8_E5M2: 57344.0}


def fp8_code_values(fmt: int) -> np.ndarray:
    """float64 value of each of the 256 codes, decoded by torch."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(_TORCH_FP8[fmt]).to(torch.float64).numpy()


def fp8_nearest(x: np.ndarray, fmt: int) -> np.ndarray:
    """Brute-force RNE-saturating fp8 encoding of float values (any float dtype)."""
    x = np.asarray(x, dtype=np.float64).ravel()
    vals = fp8_code_values(fmt)
    pos_codes = np.array([c for c in range(128) if np.isfinite(vals[c])], dtype=np.int64)
    pos_vals = vals[pos_codes]  # ascending, 0 first
    out = np.empty(x.shape, np.uint8)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    # Beyond the largest finite code the nearest code is that code; clamping at
    # twice its value keeps every distance below exact in float64.
    a_fin = np.where(nan, 0.0, np.minimum(a, 2.0 * pos_vals[-1]))
    chunk = 1 << 14
    for s in range(0, a.size, chunk):
        aa = a_fin[s:s + chunk, None]
        d = np.abs(aa - pos_vals[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # prefer the even code among tied candidates (mantissa LSB is bit 0)
        even = (pos_codes[None, :] & 1) == 0
        pick_even = cand & even
        has_even = pick_even.any(axis=1)
        idx = np.where(has_even, pick_even.argmax(axis=1), cand.argmax(axis=1))
        out[s:s + chunk] = pos_codes[idx].astype(np.uint8)
    out = np.where(sign, out | 0x80, out).astype(np.uint8)
    out = np.where(nan, 0x7F, out).astype(np.uint8)  # canonical NaN code
    return out


def bf16_bits_value(b: int) -> float:
    return float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])


def bf16_round_exact(x) -> np.ndarray:
    """Nearest-even bf16 bit pattern of each double, by exact rational comparison."""
    x = np.asarray(x, dtype=np.float64).ravel()
    out = np.empty(x.shape, np.uint16)
    for i, v in enumerate(x.tolist()):
        if v != v:
            out[i] = 0x7FC0 | (0x8000 if np.signbit(x[i]) else 0)
            continue
        sgn = 0x8000 if np.signbit(x[i]) else 0
        a = abs(v)
        if a == 0.0:
            out[i] = sgn
            continue
        f32 = np.float32(a)
        base = int(np.array([f32], dtype=np.float32).view(np.uint32)[0] >> 16)
        fa = Fraction(a)
        best = None
        for b in range(max(base - 2, 0), min(base + 3, 0x7F81)):
            if b == 0x7F80:  # infinity is never the nearest for the inputs used here
                continue
            db = abs(Fraction(bf16_bits_value(b)) - fa)
            if best is None or db < best[0] or (db == best[0] and (b & 1) == 0):
                best = (db, b)
        out[i] = sgn | best[1]
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def fp8_widen_to_bf16(codes: np.ndarray, fmt: int) -> np.ndarray:
    """fp8 -> bf16 through torch (fp8 -> fp32 -> bf16; exact for finite codes)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(_TORCH_FP8[fmt])
    return t.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def ulp_diff_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in units of bf16 ordering (same-sign monotone bit distance)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a) - key(b))


def ulp_diff_fp8(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x80, -(x & 0x7F), x & 0x7F)
    return np.abs(key(a) - key(b))
