"""Pins for the oracle's RMSNorm, neox RoPE and cos/sin table.

The grouped insert can apply RMSNorm to kv_c (one weight row per layer) and a
RoPE rotation to k_pe (the same positions for every layer) before converting
("PR #50585 [K3 Perf] Optimize k3 dspark fused kv", Source snippets:
_precompute_fused_context_kv).  Checked here against closed forms, invariants,
exact rationals and library routines (torch's rms_norm, numpy's complex
multiply), not against a retyped copy of the oracle's formula.
"""
import math

import numpy as np
import pytest
import torch

import refmath as R


def bf16(x):
    return R.bf16_round_exact(np.asarray(x, np.float64))


def test_rmsnorm_constant_row_closed_form(orc):
    gamma = bf16(np.ones(512))
    for c in [1.0, -1.0, 0.0625, -3.5, 100.0, 0.25]:
        x = bf16(np.full(512, c))
        cval = R.bf16_to_f64(x[:1])[0]
        y = orc.rms_norm_row(x, gamma, 1e-6)
        expect = bf16([cval / math.sqrt(cval * cval + float(np.float32(1e-6)))])[0]
        assert (y == expect).all(), (c, hex(y[0]), hex(expect))
        # |c| >= 1/16 normalises to exactly +-1
        assert y[0] == (0x3F80 if c > 0 else 0xBF80)


def test_rmsnorm_single_nonzero_closed_form(orc):
    rng = np.random.default_rng(0)
    for _ in range(20):
        k = int(rng.integers(0, 512))
        a = bf16([rng.standard_normal() * 4])[0]
        av = R.bf16_to_f64(np.array([a], np.uint16))[0]
        gamma = bf16(1.0 + 0.1 * rng.standard_normal(512))
        gk = R.bf16_to_f64(gamma[k:k + 1])[0]
        x = np.zeros(512, np.uint16)
        x[k] = a
        y = orc.rms_norm_row(x, gamma, 1e-6)
        eps = float(np.float32(1e-6))
        expect = bf16([av * math.sqrt(512) / math.sqrt(av * av + 512 * eps) * gk])[0]
        assert y[k] == expect
        others = np.delete(y, k)
        assert (others & 0x7FFF == 0).all()  # zeros (sign follows gamma)


def test_rmsnorm_scale_invariant_without_eps(orc):
    rng = np.random.default_rng(1)
    x = bf16(rng.standard_normal(512))
    gamma = bf16(1 + 0.1 * rng.standard_normal(512))
    y = orc.rms_norm_row(x, gamma, 0.0)
    for k in (-8, 3, 17):
        xs = bf16(R.bf16_to_f64(x) * 2.0 ** k)  # exact power-of-two scaling
        np.testing.assert_array_equal(orc.rms_norm_row(xs, gamma, 0.0), y)


def test_rmsnorm_matches_torch_library(orc):
    """torch.nn.functional.rms_norm in float64, rounded exactly to bf16."""
    rng = np.random.default_rng(2)
    for row in range(8):
        x = bf16(rng.standard_normal(512) * (0.1 + row))
        gamma = bf16(1 + 0.1 * rng.standard_normal(512))
        y = orc.rms_norm_row(x, gamma, 1e-6)
        eps = float(np.float32(1e-6))
        ref = torch.nn.functional.rms_norm(
            torch.from_numpy(R.bf16_to_f64(x))[None], (512,),
            torch.from_numpy(R.bf16_to_f64(gamma)), eps)[0].numpy()
        np.testing.assert_array_equal(y, bf16(ref))


def test_rope_table_closed_forms(orc):
    P = 256
    t = orc.rope_cos_sin_cache(P, 64, 10000.0)
    # position 0: no rotation
    np.testing.assert_array_equal(t[0, :32], np.ones(32, np.float32))
    np.testing.assert_array_equal(t[0, 32:], np.zeros(32, np.float32))
    # cos^2 + sin^2 = 1 within fp32 rounding
    n = t[:, :32].astype(np.float64) ** 2 + t[:, 32:].astype(np.float64) ** 2
    assert np.abs(n - 1).max() < 4e-7
    # i = 0 has frequency 1 and i = 16 has frequency 10000^(-1/2) = 1/100
    p = np.arange(P)
    assert np.abs(t[:, 0] - np.cos(p)).max() <= 6e-8
    assert np.abs(t[:, 32] - np.sin(p)).max() <= 6e-8
    assert np.abs(t[:, 16] - np.cos(p / 100.0)).max() <= 6e-8
    assert np.abs(t[:, 48] - np.sin(p / 100.0)).max() <= 6e-8


def test_rope_table_frequencies_are_geometric(orc):
    """At position 1 the angles are the frequencies: 1, r, r^2, ... with
    r^32 = 1/10000 (exponent -2i/64, base 10000)."""
    t = orc.rope_cos_sin_cache(2, 64, 10000.0)
    theta = np.arctan2(t[1, 32:].astype(np.float64), t[1, :32].astype(np.float64))
    assert abs(theta[0] - 1.0) < 1e-7
    ratios = theta[1:] / theta[:-1]
    assert np.abs(ratios - 10000.0 ** (-1 / 32)).max() < 2e-6
    assert abs(theta[31] / theta[0] - 10000.0 ** (-31 / 32)) < 1e-6


def test_rope_table_angle_addition(orc):
    t = orc.rope_cos_sin_cache(32768, 64, 10000.0).astype(np.float64)
    rng = np.random.default_rng(3)
    a = rng.integers(0, 16384, 200)
    b = rng.integers(0, 16384, 200)
    ca, sa, cb, sb = t[a, :32], t[a, 32:], t[b, :32], t[b, 32:]
    c_sum = ca * cb - sa * sb
    s_sum = sa * cb + ca * sb
    assert np.abs(c_sum - t[a + b, :32]).max() < 2e-7
    assert np.abs(s_sum - t[a + b, 32:]).max() < 2e-7


def test_rope_identity_at_position_zero(orc):
    rng = np.random.default_rng(4)
    x = bf16(rng.standard_normal(64))
    t = orc.rope_cos_sin_cache(1, 64, 10000.0)
    np.testing.assert_array_equal(orc.rope_neox_row(x, np.ascontiguousarray(t[0])), x)


def test_rope_matches_complex_multiply(orc):
    """Neox pairs (i, i+32) rotate like the complex number x_i + j x_{i+32}
    multiplied by cos + j sin (numpy complex128)."""
    rng = np.random.default_rng(5)
    table = orc.rope_cos_sin_cache(32768, 64, 10000.0)
    for pos in rng.integers(0, 32768, 50):
        x = bf16(rng.standard_normal(64))
        cs = np.ascontiguousarray(table[pos])
        y = orc.rope_neox_row(x, cs)
        xv = R.bf16_to_f64(x)
        z = (xv[:32] + 1j * xv[32:]) * (cs[:32].astype(np.float64) + 1j * cs[32:].astype(np.float64))
        np.testing.assert_array_equal(y[:32], bf16(z.real))
        np.testing.assert_array_equal(y[32:], bf16(z.imag))
        # the pair norm is preserved up to bf16 rounding
        yv = R.bf16_to_f64(y)
        n0 = xv[:32] ** 2 + xv[32:] ** 2
        n1 = yv[:32] ** 2 + yv[32:] ** 2
        assert np.all(np.abs(np.sqrt(n1) - np.sqrt(n0)) <= 2 ** -7 * np.sqrt(n0) + 1e-30)


def test_rope_quarter_turn(orc):
    """cos = 0, sin = 1 maps (x1, x2) to (-x2, x1) exactly."""
    rng = np.random.default_rng(6)
    x = bf16(rng.standard_normal(64))
    cs = np.concatenate([np.zeros(32), np.ones(32)]).astype(np.float32)
    y = orc.rope_neox_row(x, cs)
    np.testing.assert_array_equal(y[:32], x[32:] ^ 0x8000)
    np.testing.assert_array_equal(y[32:], x[:32])
