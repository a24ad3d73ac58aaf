"""Pins for the oracle's element codecs (bf16, fp8 e4m3fn / e5m2).

The fp8 conversion is the per-element step of the grouped insert ("PR #55356
[Kimi Perf] Group fp8 mla cache insertion", Source snippets: the
scaled_convert branch) and of the fp8 pack ("PR #51772 [Attention][MLA] Fuse
Kimi-K3 chunked-context K/V packing", Implementation item 1).  The oracle's
encoder is checked against: the OCP OFP8 special values and hand-worked ties
(tests/golden), torch's decode of all 256 codes, a brute-force nearest-code
search over all 2^16 bf16 inputs (at scale 1 and at the workloads' scales),
torch's own cast on its non-overflow domain, and decode/encode round trips.
"""
import os

import numpy as np
import pytest
import torch

import refmath as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ofp8_bf16_values.txt")
FMT = {"e4m3": R.FP8_E4M3, "e5m2": R.FP8_E5M2}


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        fmt, kind, value, code = line.split()[:4]
        rows.append((fmt, kind, float(value), int(code, 16)))
    return rows


def all_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    return bits.view(np.float32)


def test_golden_special_values_and_ties(orc):
    rows = _golden_rows()
    assert len(rows) > 40
    for fmt, kind, value, code in rows:
        if fmt == "bf16":
            assert orc.bf16_from_f64(value) == code, (value, hex(code))
            continue
        f = FMT[fmt]
        if kind == "dec":
            got = orc.fp8_to_f64(code, f)
            if np.isnan(value):
                assert np.isnan(got), (fmt, hex(code))
            else:
                assert got == value, (fmt, hex(code), got, value)
        else:
            assert orc.fp8_from_f32(value, f) == code, (fmt, value, hex(code))


@pytest.mark.parametrize("fmt", [R.FP8_E4M3, R.FP8_E5M2])
def test_decode_matches_torch_all_codes(orc, fmt):
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.fp8_decode(codes, fmt)
    lib = R.fp8_code_values(fmt)
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    np.testing.assert_array_equal(mine[ok], lib[ok])
    # signed zeros decode with their sign
    assert np.signbit(mine[0x80]) and not np.signbit(mine[0])


@pytest.mark.parametrize("fmt", [R.FP8_E4M3, R.FP8_E5M2])
@pytest.mark.parametrize("scale", [1.0, 0.005, 0.0123, 0.02, 0.01])
def test_encode_exhaustive_bf16_vs_brute_force(orc, fmt, scale):
    """All 2^16 bf16 patterns, divided by the scale in fp32, against the
    brute-force nearest finite code (ties to even, saturating)."""
    x = all_bf16_as_f32()
    q = (x / np.float32(scale)).astype(np.float32)  # IEEE fp32 division
    mine = orc.fp8_encode(q, fmt)
    ref = R.fp8_nearest(q, fmt)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, [(float(q[i]), hex(mine[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("fmt", [R.FP8_E4M3, R.FP8_E5M2])
def test_encode_matches_torch_cast_below_overflow(orc, fmt):
    """torch's CPU cast is RNE but not saturating: it agrees with the oracle on
    every input below the overflow midpoint and differs (NaN / inf) above."""
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    mine = orc.fp8_encode(x, fmt)
    tdt = torch.float8_e4m3fn if fmt == R.FP8_E4M3 else torch.float8_e5m2
    lib = torch.from_numpy(x.copy()).to(tdt).view(torch.uint8).numpy()
    limit = 464.0 if fmt == R.FP8_E4M3 else 61440.0
    below = np.abs(x) <= (limit if fmt == R.FP8_E4M3 else limit - 1)
    np.testing.assert_array_equal(mine[below], lib[below])
    above = np.abs(x) > limit
    assert above.any()
    maxcode = 0x7E if fmt == R.FP8_E4M3 else 0x7B
    np.testing.assert_array_equal(mine[above] & 0x7F, np.full(above.sum(), maxcode, np.uint8))
    assert (lib[above] & 0x7F != maxcode).all()  # the documented divergence


@pytest.mark.parametrize("fmt", [R.FP8_E4M3, R.FP8_E5M2])
def test_decode_encode_round_trip(orc, fmt):
    for c in range(256):
        v = orc.fp8_to_f64(c, fmt)
        if np.isnan(v):
            assert orc.fp8_from_f32(v, fmt) == 0x7F
            continue
        if np.isinf(v):
            continue
        assert orc.fp8_from_f32(v, fmt) == c, (fmt, hex(c), v)


@pytest.mark.parametrize("fmt", [R.FP8_E4M3, R.FP8_E5M2])
def test_encode_monotone_and_sign_symmetric(orc, fmt):
    x = np.sort(np.abs(all_bf16_as_f32()[np.isfinite(all_bf16_as_f32())]))
    codes = orc.fp8_encode(x, fmt).astype(np.int32)
    assert (np.diff(codes) >= 0).all()
    neg = orc.fp8_encode(-x, fmt)
    np.testing.assert_array_equal(neg, (codes | 0x80).astype(np.uint8))


def test_nan_encodes_to_the_canonical_nan_code(orc):
    for fmt in (R.FP8_E4M3, R.FP8_E5M2):
        assert orc.fp8_from_f32(float("nan"), fmt) == 0x7F
        assert orc.fp8_from_f32(-float("nan"), fmt) == 0x7F


def test_bf16_from_f32_matches_torch(orc):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    extra = np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.3895313892515355e38,
                      1e-40, -1e-40, 9.2e-41, 65504.0], np.float32)
    x = np.concatenate([x, extra])
    mine = orc.bf16_from_f32_array(x)
    lib = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, lib)


def test_bf16_from_f64_exact_rational(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000)),
        # exact midpoints between neighbouring bf16 values (ties) and near-ties
        (1.0 + (2 * rng.integers(0, 128, 500) + 1) / 256.0) * np.exp2(rng.integers(-10, 10, 500)),
        (1.0 + (2 * rng.integers(0, 128, 500) + 1) / 256.0 + 1e-12) * np.exp2(rng.integers(-10, 10, 500)),
        np.array([1e-39, -3e-39, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135]),
    ])
    mine = orc.bf16_from_f64_array(x)
    ref = R.bf16_round_exact(x)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, [(x[i], hex(mine[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("fmt", [R.FP8_E4M3, R.FP8_E5M2])
def test_fp8_widening_to_bf16_is_exact(orc, fmt):
    """fp8 -> bf16 without a scale: bit-equal to torch's fp8 -> fp32 -> bf16 cast
    for every finite code, and value-preserving."""
    ref = R.fp8_widen_to_bf16(np.arange(256, dtype=np.uint8), fmt)
    vals = R.fp8_code_values(fmt)
    for c in range(256):
        got = orc.bf16_from_fp8(c, fmt)
        if np.isnan(vals[c]):
            assert got & 0x7FFF == 0x7FC0 and (got >> 15) == (c >> 7)
            continue
        assert got == ref[c], (hex(c), hex(got), hex(ref[c]))
        assert R.bf16_to_f64(np.array([got], np.uint16))[0] == vals[c]
