"""Pins for the oracle's fp16 support: the pack's fp16 inputs ("PR #51772
[Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing", Review: the fused
kernel is tested with bf16 and fp16 inputs) and the gather's exact widening of
fp8 into an fp16 kv_b_proj input (Implementation item 5: the cast to the
kv_b_proj input dtype).

* binary16 decode of all 2^16 patterns against numpy's float16;
* binary16 encode against numpy's correctly rounded float64 -> float16 cast on
  random doubles over the whole range, plus hand-worked ties, the overflow
  threshold 65520 and the subnormal ties (IEEE 754 binary16);
* fp8 -> fp16 widening of all 256 codes of both formats against torch;
* the pack with fp16 inputs: a concatenation of the input bits for fp16
  output, the brute-force fp8 encoder of value / scale for fp8 output, an fp8
  k_pe widened exactly into an fp16 key;
* the gather into fp16 rows: the widening applied to the raw gather.
"""
import numpy as np
import pytest
import torch

import refmath as R
from pack_mla_cache_gb300 import workloads as W

ENTRY = 576
F16 = 3


def test_decode_all_patterns_matches_numpy(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_encode_matches_numpy_correct_rounding(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, 20000)),
        rng.uniform(-70000, 70000, 5000),
        rng.uniform(-2.0 ** -14, 2.0 ** -14, 5000),
    ])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([orc.f16_from_f64(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3C00), (-2.0, 0xC000), (65504.0, 0x7BFF), (65519.99, 0x7BFF),
    (65520.0, 0x7C00), (-65520.0, 0xFC00), (1e10, 0x7C00),
    (1 + 2.0 ** -11, 0x3C00),            # tie between 1 and 1 + 2^-10 -> even (1)
    (1 + 3 * 2.0 ** -11, 0x3C02),        # tie between 1 + 2^-10 and 1 + 2^-9 -> even
    (2.0 ** -14, 0x0400), (2.0 ** -24, 0x0001),
    (2.0 ** -25, 0x0000),                # tie between 0 and the smallest subnormal -> 0
    (3 * 2.0 ** -25, 0x0002),            # tie between 1 and 2 subnormal quanta -> 2
    (-0.0, 0x8000), (float("inf"), 0x7C00), (float("-inf"), 0xFC00),
])
def test_encode_worked_values(orc, x, bits):
    assert orc.f16_from_f64(x) == bits


def test_encode_nan_keeps_sign(orc):
    assert orc.f16_from_f64(float("nan")) == 0x7E00
    assert orc.f16_from_f64(-float("nan")) == 0xFE00


@pytest.mark.parametrize("fmt", [1, 2])
def test_fp8_widening_matches_torch(orc, fmt):
    t = {1: torch.float8_e4m3fn, 2: torch.float8_e5m2}[fmt]
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(t).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    vals = R.fp8_code_values(fmt)
    for c in range(256):
        got = orc.f16_from_fp8(c, fmt)
        if np.isnan(vals[c]):
            assert got == (0x8000 if c & 0x80 else 0) | 0x7E00
        else:
            assert got == ref[c], hex(c)


def _f16_heads(T, H, seed):
    rng = np.random.default_rng(seed)
    kvb = (rng.standard_normal((T, H * 256 + 64)) * 4).astype(np.float16).view(np.uint16)
    return np.ascontiguousarray(kvb)


@pytest.mark.parametrize("H", [1, 3, 16])
def test_fp16_pack_is_a_concat_of_the_input_bits(orc, H):
    T = 29
    kvb = _f16_heads(T, H, H)
    rs = kvb.shape[1]
    kpe = _f16_heads(T, 1, 99)[:, :64].copy()
    key, v = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, kpe, 64, F16, T, H, 128,
                                 64, 128, F16, in_dtype=F16)
    heads = kvb[:, : H * 256].reshape(T, H, 256)
    np.testing.assert_array_equal(key[:, :, :128], heads[:, :, :128])
    np.testing.assert_array_equal(key[:, :, 128:], np.broadcast_to(kpe[:, None], (T, H, 64)))
    np.testing.assert_array_equal(v, heads[:, :, 128:])


@pytest.mark.parametrize("fmt", [1, 2])
def test_fp16_to_fp8_pack_equals_brute_force_encoder(orc, fmt):
    T, H, scale = 23, 4, 0.03
    kvb = _f16_heads(T, H, 5)
    rs = kvb.shape[1]
    kpe = _f16_heads(T, 1, 6)[:, :64].copy()
    key, v = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, kpe, 64, F16, T, H, 128,
                                 64, 128, fmt, out_scale=scale, in_dtype=F16)
    heads = kvb[:, : H * 256].reshape(T, H, 256).view(np.float16).astype(np.float32)
    enc = lambda a: R.fp8_nearest((a / np.float32(scale)).astype(np.float32), fmt).reshape(a.shape)
    np.testing.assert_array_equal(key[:, :, :128], enc(heads[:, :, :128]))
    np.testing.assert_array_equal(v, enc(heads[:, :, 128:]))
    pe = enc(kpe.view(np.float16).astype(np.float32))
    np.testing.assert_array_equal(key[:, :, 128:], np.broadcast_to(pe[:, None], (T, H, 64)))


def test_fp8_kpe_widens_into_an_fp16_key(orc):
    T, H = 17, 3
    kvb = _f16_heads(T, H, 7)
    rs = kvb.shape[1]
    kpe = np.random.default_rng(8).integers(0, 256, size=(T, 64)).astype(np.uint8)
    key, _ = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, kpe, 64, 1, T, H, 128,
                                 64, 128, F16, in_dtype=F16)
    lut = np.array([orc.f16_from_fp8(c, 1) for c in range(256)], np.uint16)
    np.testing.assert_array_equal(key[:, :, 128:], np.broadcast_to(lut[kpe][:, None], (T, H, 64)))


@pytest.mark.parametrize("fmt", [1, 2])
def test_gather_widens_into_fp16_rows(orc, fmt):
    pw = W.pack_workload(num_tokens=640, chunk=640, num_blocks=16, block_size=64, seed=9,
                         cache_dtype=fmt)
    nb, B = pw.num_blocks, pw.block_size
    cu, st = np.array([0, 600], np.int32), np.array([33], np.int32)
    raw = np.zeros((600, ENTRY), np.uint8)
    assert orc.context_gather(pw.cache, fmt, nb, B, B * ENTRY, ENTRY, ENTRY, pw.block_table, cu,
                              st, raw, fmt) == 0
    out = np.zeros((600, ENTRY), np.uint16)
    assert orc.context_gather(pw.cache, fmt, nb, B, B * ENTRY, ENTRY, ENTRY, pw.block_table, cu,
                              st, out, F16) == 0
    lut = np.array([orc.f16_from_fp8(c, fmt) for c in range(256)], np.uint16)
    np.testing.assert_array_equal(out, lut[raw])
