"""Pins for the oracle's scaled dequantising gather and its pack with k_pe read
from the paged cache.

* Scaled widening: the exact value of every fp8 code (decoded by torch) times
  the scale as a numpy float32 product, rounded to bf16 by exact rational
  comparison; the closed form for power-of-two scales (no rounding at all);
  scale 1 reduces to torch's exact widening; NaN, infinity and overflow rules.
* Scaled gather: element-wise the scalar rule applied to the raw gather, and
  the rows numpy fancy indexing selects.
* Paged pack ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V
  packing", Implementation item 1: k_pe still in the cache layout): equal to
  the raw gather of full rows followed by the pack of the workspace's k_pe, and
  to numpy fancy indexing of the cache; rows it cannot find leave the key's
  rope slice untouched.
"""
import math

import numpy as np
import pytest

import refmath as R
from pack_mla_cache_gb300 import workloads as W

ENTRY = 576


def _bits_f32(x) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


# ------------------------------------------------------------ scaled widening
@pytest.mark.parametrize("fmt", [1, 2])
def test_scale_one_is_the_exact_widening(orc, fmt):
    vals = R.fp8_code_values(fmt)
    torch_bits = R.fp8_widen_to_bf16(np.arange(256, dtype=np.uint8), fmt)
    for c in range(256):
        got = orc.bf16_from_fp8_scaled(c, fmt, 1.0)
        if np.isnan(vals[c]):
            assert got == (0x8000 if c & 0x80 else 0) | 0x7FC0, hex(c)
        else:
            assert got == torch_bits[c], hex(c)


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("scale", [0.01, 0.0173, 0.3, 3.7, 123456.7, 1e-30, 2.5e-38, 7e-41])
def test_scaled_widening_is_one_fp32_product_then_bf16(orc, fmt, scale):
    vals = R.fp8_code_values(fmt)
    fin = np.isfinite(vals)
    prod = (vals[fin].astype(np.float32) * np.float32(scale)).astype(np.float32)
    expect = R.bf16_round_exact(prod.astype(np.float64))
    got = np.array([orc.bf16_from_fp8_scaled(c, fmt, scale) for c in np.flatnonzero(fin)],
                   np.uint16)
    np.testing.assert_array_equal(got, expect)


@pytest.mark.parametrize("fmt", [1, 2])
def test_product_is_rounded_to_fp32_before_bf16(orc, fmt):
    """Cases where rounding the exact product straight to bf16 differs from
    rounding it first to fp32 (the fp32 product lands on a bf16 tie): the
    oracle follows the fp32 product."""
    vals = R.fp8_code_values(fmt)
    codes = np.flatnonzero(np.isfinite(vals) & (vals != 0))
    rng = np.random.default_rng(123)
    scales = rng.uniform(0.001, 0.05, 200000).astype(np.float32)
    hits = []
    for c in codes[::3]:
        p64 = vals[c] * scales.astype(np.float64)  # exact: 4 x 24 significant bits
        p32 = p64.astype(np.float32)
        tie = (p32.view(np.uint32) & 0xFFFF) == 0x8000
        idx = np.flatnonzero(tie & (p32.astype(np.float64) != p64))
        for i in idx[:4]:
            via32 = int(R.bf16_round_exact([float(p32[i])])[0])
            direct = int(R.bf16_round_exact([float(p64[i])])[0])
            if via32 != direct:  # the tie went to even, away from the exact product
                hits.append((int(c), float(scales[i]), via32))
    assert len(hits) >= 10
    for c, sc, via32 in hits:
        assert orc.bf16_from_fp8_scaled(c, fmt, sc) == via32


@pytest.mark.parametrize("fmt,k_range", [(1, range(-120, 101, 7)), (2, range(-110, 101, 9))])
def test_power_of_two_scale_is_exact(orc, fmt, k_range):
    """v * 2^k has at most 4 significant bits and stays in the normal or
    bf16-representable subnormal range here, so the result is exact: the top
    half of the fp32 value, whose low half is zero."""
    vals = R.fp8_code_values(fmt)
    for k in k_range:
        for c in range(256):
            if not np.isfinite(vals[c]):
                continue
            exact = math.ldexp(float(vals[c]), k)
            b = _bits_f32(exact)
            assert b & 0xFFFF == 0 and float(np.float32(exact)) == exact
            assert orc.bf16_from_fp8_scaled(c, fmt, math.ldexp(1.0, k)) == b >> 16, (k, hex(c))


def test_nan_infinity_and_overflow_rules(orc):
    # NaN codes keep their sign at any scale
    for fmt, nans in ((1, [0x7F, 0xFF]), (2, [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF])):
        for c in nans:
            for sc in (0.5, 0.0, float("inf")):
                assert orc.bf16_from_fp8_scaled(c, fmt, sc) == (0x8000 if c & 0x80 else 0) | 0x7FC0
    # e5m2 infinities scale to infinities; times zero they are the positive NaN
    assert orc.bf16_from_fp8_scaled(0x7C, 2, 0.01) == 0x7F80
    assert orc.bf16_from_fp8_scaled(0xFC, 2, 0.01) == 0xFF80
    assert orc.bf16_from_fp8_scaled(0xFC, 2, 0.0) == 0x7FC0
    # a NaN scale gives the positive NaN for every non-NaN code
    assert orc.bf16_from_fp8_scaled(0x38, 1, float("nan")) == 0x7FC0
    # fp32 overflow of the product is an infinity of the code's sign
    assert orc.bf16_from_fp8_scaled(0x7B, 2, 2.0 ** 120) == 0x7F80
    assert orc.bf16_from_fp8_scaled(0xFB, 2, 2.0 ** 120) == 0xFF80
    # a negative scale flips the sign; zero codes keep the product's sign
    assert orc.bf16_from_fp8_scaled(0x38, 1, -2.0) == 0xC000  # 1.0 * -2
    assert orc.bf16_from_fp8_scaled(0x00, 1, -2.0) == 0x8000
    assert orc.bf16_from_fp8_scaled(0x80, 1, 2.0) == 0x8000


# ------------------------------------------------------------- scaled gather
def _two_seq_layout(pw):
    table = np.stack([pw.block_table[0, :16], pw.block_table[0, 16:32]]).astype(np.int32)
    starts = np.array([100, 0], np.int32)
    cu = np.array([0, 600, 850], np.int32)
    return table, starts, cu


@pytest.mark.parametrize("fmt", [1, 2])
def test_scaled_gather_is_the_scalar_rule_on_the_raw_gather(orc, fmt):
    pw = W.pack_workload(num_tokens=2048, chunk=2048, num_blocks=40, block_size=64, seed=7,
                         cache_dtype=fmt)
    nb, B = pw.num_blocks, pw.block_size
    table, starts, cu = _two_seq_layout(pw)
    raw = np.zeros((850, ENTRY), np.uint8)
    err_raw = orc.context_gather(pw.cache, fmt, nb, B, B * ENTRY, ENTRY, ENTRY, table, cu,
                                 starts, raw, fmt)
    out = np.full((850, ENTRY), 0x1234, np.uint16)
    scale = 0.0173
    err = orc.context_gather_scaled(pw.cache, fmt, nb, B, B * ENTRY, ENTRY, ENTRY, table, cu,
                                    starts, out, scale)
    assert err == err_raw == 0
    # every code through the scalar rule, by a lookup table of all 256 codes
    lut = np.array([orc.bf16_from_fp8_scaled(c, fmt, scale) for c in range(256)], np.uint16)
    np.testing.assert_array_equal(out, lut[raw])
    # and the rows are those numpy fancy indexing selects
    cache3 = pw.cache.reshape(nb, B, ENTRY)
    rows = []
    for s in range(2):
        p = starts[s] + np.arange(cu[s + 1] - cu[s])
        rows.append(cache3[table[s, p // B], p % B])
    np.testing.assert_array_equal(raw, np.concatenate(rows))


def test_scaled_gather_bad_block_is_skipped_and_reported(orc):
    pw = W.pack_workload(num_tokens=128, chunk=128, num_blocks=4, block_size=64, seed=8)
    table = np.array([[1, 9]], np.int32)
    out = np.full((128, ENTRY), 0x3333, np.uint16)
    err = orc.context_gather_scaled(pw.cache, 1, 4, 64, 64 * ENTRY, ENTRY, ENTRY, table,
                                    np.array([0, 128], np.int32), np.array([0], np.int32), out,
                                    0.5)
    assert err == orc.ERR_BLOCK_OOB
    assert (out[64:] == 0x3333).all() and (out[:64] != 0x3333).any()


# --------------------------------------------------------------- paged pack
def _paged_case(cache_dtype, T=300, H=16, seed=10):
    pw = W.pack_workload(num_tokens=2048, chunk=2048, num_blocks=40, block_size=64,
                         num_heads=H, seed=seed, cache_dtype=cache_dtype)
    # three sequences with unaligned starts; their chunk tokens fill [0, T)
    bt = pw.block_table[0]
    table = np.stack([bt[0:6], bt[6:12], bt[12:18]]).astype(np.int32)
    starts = np.array([37, 0, 130], np.int32)
    cu = np.array([0, 120, 200, T], np.int32)
    kvb = W.pack_workload(num_tokens=T, chunk=T, num_blocks=8, num_heads=H, seed=seed + 1).kv_b_proj[0]
    return pw, table, starts, cu, kvb


@pytest.mark.parametrize("cache_dtype,out_dtype", [(1, 1), (1, 0), (2, 2), (2, 0), (0, 0), (0, 1)])
def test_paged_pack_equals_gather_then_pack(orc, cache_dtype, out_dtype):
    T, H = 300, 16
    pw, table, starts, cu, kvb = _paged_case(cache_dtype, T, H)
    nb, B, rs = pw.num_blocks, pw.block_size, kvb.shape[1]
    ws = np.zeros((T, ENTRY), np.uint16 if cache_dtype == 0 else np.uint8)
    assert orc.context_gather(pw.cache, cache_dtype, nb, B, B * ENTRY, ENTRY, ENTRY, table, cu,
                              starts, ws, cache_dtype) == 0
    key_ref, v_ref = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256,
                                         np.ascontiguousarray(ws[:, 512:]), 64, cache_dtype, T, H,
                                         128, 64, 128, out_dtype=out_dtype, out_scale=0.01)
    key, v, err = orc.context_kv_pack_paged(kvb, rs, 256, kvb[:, 128:], rs, 256, pw.cache,
                                            cache_dtype, nb, B, B * ENTRY, ENTRY, 512, table, cu,
                                            starts, T, H, 128, 64, 128, out_dtype, 0.01)
    assert err == 0
    np.testing.assert_array_equal(key, key_ref)
    np.testing.assert_array_equal(v, v_ref)
    if out_dtype == cache_dtype:  # the rope slice is the cache's bytes themselves
        cache3 = pw.cache.reshape(nb, B, ENTRY)
        for s in range(3):
            p = starts[s] + np.arange(cu[s + 1] - cu[s])
            pe = cache3[table[s, p // B], p % B, 512:]
            np.testing.assert_array_equal(key[cu[s]:cu[s + 1], :, 128:],
                                          np.broadcast_to(pe[:, None], (len(p), H, 64)))


def test_paged_pack_unfound_rows_keep_the_rope_slice(orc):
    T, H = 120, 3
    pw, table, starts, cu, kvb = _paged_case(1, T, H)
    nb, B, rs = pw.num_blocks, pw.block_size, kvb.shape[1]
    cu = np.array([5, 70, 100, 110], np.int32)  # tokens 0-4 and 110-119 owned by no sequence
    table = table.copy()
    table[1, 1] = nb + 3  # sequence 1 (positions 0-29 of block index 0) is fine...
    starts = np.array([37, 50, 130], np.int32)  # ...but from position 64 on it uses index 1
    init = np.full((T, H, 192), 0x5A, np.uint8)
    key, v, err = orc.context_kv_pack_paged(kvb, rs, 256, kvb[:, 128:], rs, 256, pw.cache, 1, nb,
                                            B, B * ENTRY, ENTRY, 512, table, cu, starts, T, H,
                                            128, 64, 128, 1, 0.01, key_init=init)
    assert err == orc.ERR_BLOCK_OOB
    bad = list(range(0, 5)) + list(range(70 + 14, 100)) + list(range(110, 120))
    good = [t for t in range(T) if t not in bad]
    assert (key[bad][:, :, 128:] == 0x5A).all()
    assert (key[good][:, :, 128:] != 0x5A).any()
    # k_nope and V are written for every token
    ref_key, ref_v = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256,
                                         np.zeros((T, 64), np.uint8), 64, 1, T, H, 128, 64, 128,
                                         out_dtype=1, out_scale=0.01)
    np.testing.assert_array_equal(key[:, :, :128], ref_key[:, :, :128])
    np.testing.assert_array_equal(v, ref_v)
