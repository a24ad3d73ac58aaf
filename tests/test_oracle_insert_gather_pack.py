"""Pins for the oracle's grouped insert, context gather and K/V pack.

* Grouped insert ("PR #55356 [Kimi Perf] Group fp8 mla cache insertion",
  Source snippets and test_concat_and_cache_mla_grouped): checked against a
  numpy scatter written from the page's index arithmetic, the brute-force fp8
  encoder, per-layer equivalence, the shared (aliased) slot mapping, the -1
  padding slot and out-of-range slots.
* Gather and pack ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context
  K/V packing", Implementation items 1-2 and Source snippets): checked against
  numpy fancy indexing, the insert -> gather round trip, torch's exact fp8 ->
  bf16 widening, and the step-by-step gather -> cast -> concat -> cast chain.
"""
import numpy as np
import pytest

import refmath as R
from pack_mla_cache_gb300 import workloads as W

ENTRY = 576


def _rows_expected_bf16(wl, layer):
    """Expected [kv_c | k_pe] rows of one layer as uint16 (raw insert)."""
    return np.concatenate([wl.kv_c[layer], wl.k_pe[layer]], axis=1)


def _numpy_scatter(cache, rows, slots, block_size, block_stride, entry_stride):
    nb = cache.size // block_stride
    view = np.lib.stride_tricks.as_strided(
        cache, shape=(nb, block_size, ENTRY),
        strides=(block_stride * cache.itemsize, entry_stride * cache.itemsize, cache.itemsize))
    for t, s in enumerate(slots):
        if s < 0:
            continue
        view[s // block_size, s % block_size, :] = rows[t]


@pytest.mark.parametrize("shared", [True, False])
def test_raw_bf16_insert_equals_numpy_scatter(orc, shared):
    wl = W.pages_test_insert_workload(cache_dtype=0, shared_slots=shared)
    caches = wl.empty_caches(fill=0xABCD)
    err = orc.insert_grouped(wl.kv_c, wl.k_pe, wl.slot_mapping, wl.slot_layer_stride, caches,
                             None, 0, wl.num_blocks, wl.block_size, wl.block_stride,
                             wl.entry_stride)
    assert err == 0
    for l in range(wl.num_layers):
        ref = np.full_like(caches[l], 0xABCD)
        slots = wl.slot_mapping[0 if shared else l]
        _numpy_scatter(ref, _rows_expected_bf16(wl, l), slots, wl.block_size,
                       wl.block_stride, wl.entry_stride)
        np.testing.assert_array_equal(caches[l], ref)


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("shared", [True, False])
def test_fp8_insert_equals_brute_force_encoder(orc, fmt, shared):
    wl = W.pages_test_insert_workload(cache_dtype=fmt, shared_slots=shared)
    caches = wl.empty_caches(fill=0x5A)
    orc.insert_grouped(wl.kv_c, wl.k_pe, wl.slot_mapping, wl.slot_layer_stride, caches,
                       wl.k_scales, fmt, wl.num_blocks, wl.block_size, wl.block_stride,
                       wl.entry_stride)
    for l in range(wl.num_layers):
        vals = R.bf16_to_f32(_rows_expected_bf16(wl, l))
        q = (vals / np.float32(wl.k_scales[l])).astype(np.float32)
        codes = R.fp8_nearest(q, fmt).reshape(q.shape)
        ref = np.full_like(caches[l], 0x5A)
        _numpy_scatter(ref, codes, wl.slot_mapping[0 if shared else l], wl.block_size,
                       wl.block_stride, wl.entry_stride)
        np.testing.assert_array_equal(caches[l], ref)


def test_grouped_equals_per_layer_and_shared_equals_expanded(orc):
    wl = W.insert_workload(5, 300, 1, num_blocks=16, block_size=32, shared_slots=True,
                           norm=True, rope=True, seed=3)
    table = orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)
    shared = wl.empty_caches()
    orc.insert_grouped(wl.kv_c, wl.k_pe, np.ascontiguousarray(wl.slot_mapping[0]), 0, shared,
                       wl.k_scales, 1, wl.num_blocks, wl.block_size, wl.block_stride,
                       wl.entry_stride, wl.gamma, 1e-6, wl.positions, table)
    expanded = wl.empty_caches()
    orc.insert_grouped(wl.kv_c, wl.k_pe, wl.slot_mapping, wl.num_tokens, expanded, wl.k_scales,
                       1, wl.num_blocks, wl.block_size, wl.block_stride, wl.entry_stride,
                       wl.gamma, 1e-6, wl.positions, table)
    for l in range(5):
        per = wl.empty_caches()[0]
        orc.insert_layer(np.ascontiguousarray(wl.kv_c[l]), np.ascontiguousarray(wl.k_pe[l]),
                         np.ascontiguousarray(wl.slot_mapping[l]), per, 1, wl.num_blocks,
                         wl.block_size, wl.block_stride, wl.entry_stride, wl.k_scales[l],
                         np.ascontiguousarray(wl.gamma[l]), 1e-6, wl.positions, table)
        np.testing.assert_array_equal(shared[l], per)
        np.testing.assert_array_equal(expanded[l], per)


def test_norm_rope_insert_composes_row_functions(orc):
    """A bf16 cache exposes the pre-quantisation values: they are the RMSNorm
    row (torch rms_norm in float64, rounded exactly) and the RoPE row."""
    import torch
    wl = W.insert_workload(2, 24, 0, num_blocks=4, block_size=16, norm=True, rope=True, seed=4)
    table = orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)
    caches = wl.empty_caches()
    orc.insert_grouped(wl.kv_c, wl.k_pe, wl.slot_mapping, 0, caches, None, 0, wl.num_blocks,
                       wl.block_size, wl.block_stride, wl.entry_stride, wl.gamma, 1e-6,
                       wl.positions, table)
    eps = float(np.float32(1e-6))
    for l in range(2):
        view = caches[l].reshape(wl.num_blocks, wl.block_size, ENTRY)
        for t in range(wl.num_tokens):
            s = wl.slot_mapping[l, t]
            row = view[s // wl.block_size, s % wl.block_size]
            x = torch.from_numpy(R.bf16_to_f64(wl.kv_c[l, t]))
            g = torch.from_numpy(R.bf16_to_f64(wl.gamma[l]))
            ref_norm = R.bf16_round_exact(
                torch.nn.functional.rms_norm(x[None], (512,), g, eps)[0].numpy())
            np.testing.assert_array_equal(row[:512], ref_norm)
            pe = R.bf16_to_f64(wl.k_pe[l, t])
            cs = table[wl.positions[t]].astype(np.float64)
            z = (pe[:32] + 1j * pe[32:]) * (cs[:32] + 1j * cs[32:])
            np.testing.assert_array_equal(row[512:544], R.bf16_round_exact(z.real))
            np.testing.assert_array_equal(row[544:], R.bf16_round_exact(z.imag))


def test_out_of_range_slots_and_positions_are_skipped_and_reported(orc):
    wl = W.insert_workload(2, 8, 1, num_blocks=4, block_size=16, norm=True, rope=True, seed=5)
    table = orc.rope_cos_sin_cache(64, 64, W.ROPE_BASE)
    slots = np.array([0, 1, -1, 64, 2, 3, 4, 5], np.int64)  # 64 = capacity: out of range
    pos = np.array([0, 1, 2, 3, 64, 5, -1, 7], np.int64)  # 64, -1: out of table
    caches = wl.empty_caches(fill=0x11)
    err = orc.insert_grouped(wl.kv_c, wl.k_pe, slots, 0, caches, wl.k_scales, 1, 4, 16,
                             wl.block_stride, wl.entry_stride, wl.gamma, 1e-6, pos, table)
    assert err == (orc.ERR_SLOT_OOB | orc.ERR_POS_OOB)
    for l in range(2):
        rows = caches[l].reshape(-1, ENTRY)
        written = {0, 1, 3, 5}  # tokens 0, 1, 5, 7 land in slots 0, 1, 3, 5
        for s in range(64):
            assert (rows[s] != 0x11).any() == (s in written), s


def test_raw_insert_then_gather_round_trip(orc):
    """A bf16 cache round-trips exactly: gathering the inserted slots returns
    the input rows."""
    wl = W.insert_workload(1, 200, 0, num_blocks=8, block_size=64, seed=6)
    cache = wl.empty_caches()[0]
    orc.insert_grouped(wl.kv_c, wl.k_pe, wl.slot_mapping, 0, [cache], None, 0, wl.num_blocks,
                       wl.block_size, wl.block_stride, wl.entry_stride)
    # one "sequence" per token: a 1-token chunk whose position maps to the slot
    slots = wl.slot_mapping[0]
    S = len(slots)
    table = (slots // 64).astype(np.int32)[:, None]
    starts = (slots % 64).astype(np.int32)
    cu = np.arange(S + 1, dtype=np.int32)
    out = np.zeros((S, ENTRY), np.uint16)
    err = orc.context_gather(cache, 0, 8, 64, wl.block_stride, wl.entry_stride, ENTRY, table,
                             cu, starts, out, 0)
    assert err == 0
    np.testing.assert_array_equal(out, _rows_expected_bf16(wl, 0))


@pytest.mark.parametrize("out_dtype", [1, 0])
def test_gather_equals_numpy_fancy_indexing(orc, out_dtype):
    pw = W.pack_workload(num_tokens=2048, chunk=2048, num_blocks=40, block_size=64, seed=7)
    nb, B = pw.num_blocks, pw.block_size
    cache3 = pw.cache.reshape(nb, B, ENTRY)
    # two sequences: context positions [100, 700) of seq 0 and [0, 250) of seq 1
    table = np.stack([pw.block_table[0, :16], pw.block_table[0, 16:32]]).astype(np.int32)
    starts = np.array([100, 0], np.int32)
    cu = np.array([0, 600, 850], np.int32)
    out = np.full((850, ENTRY), 0x77, np.uint8 if out_dtype else np.uint16)
    err = orc.context_gather(pw.cache, 1, nb, B, B * ENTRY, ENTRY, ENTRY, table, cu, starts,
                             out, out_dtype)
    assert err == 0
    ref_rows = []
    for s in range(2):
        p = starts[s] + np.arange(cu[s + 1] - cu[s])
        ref_rows.append(cache3[table[s, p // B], p % B])
    ref = np.concatenate(ref_rows)
    if out_dtype == 0:
        ref = R.fp8_widen_to_bf16(ref, 1).reshape(ref.shape)
    np.testing.assert_array_equal(out, ref)


def test_gather_bad_block_is_skipped_and_reported(orc):
    pw = W.pack_workload(num_tokens=128, chunk=128, num_blocks=4, block_size=64, seed=8)
    table = np.array([[1, 9]], np.int32)  # block 9 does not exist
    out = np.full((128, ENTRY), 0x33, np.uint8)
    err = orc.context_gather(pw.cache, 1, 4, 64, 64 * ENTRY, ENTRY, ENTRY, table,
                             np.array([0, 128], np.int32), np.array([0], np.int32), out, 1)
    assert err == orc.ERR_BLOCK_OOB
    assert (out[64:] == 0x33).all() and (out[:64] != 0x33).any()


def _pack_inputs(T=37, H=3, seed=9, kpe_fp8=False):
    pw = W.pack_workload(num_tokens=T, chunk=T, num_blocks=2, block_size=64, num_heads=H,
                         seed=seed)
    kvb = pw.kv_b_proj[0]  # [T, row_stride]
    ws = pw.cache[: T * ENTRY].reshape(T, ENTRY) if kpe_fp8 else None
    rng = np.random.default_rng(seed)
    kpe_bf16 = R.bf16_round_exact(rng.standard_normal(T * ENTRY)).reshape(T, ENTRY)
    return pw, kvb, (ws if kpe_fp8 else kpe_bf16)


@pytest.mark.parametrize("H", [1, 3, 16])
def test_bf16_pack_is_a_concat_of_the_input_bits(orc, H):
    pw, kvb, ws = _pack_inputs(H=H)
    T, rs = kvb.shape
    key, v = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, ws[:, 512:], ENTRY, 0, T,
                                 H, 128, 64, 128, out_dtype=0)
    heads = kvb[:, : H * 256].reshape(T, H, 256)
    np.testing.assert_array_equal(key[:, :, :128], heads[:, :, :128])
    np.testing.assert_array_equal(key[:, :, 128:], np.broadcast_to(ws[:, None, 512:], (T, H, 64)))
    np.testing.assert_array_equal(v, heads[:, :, 128:])
    if H == 1:  # a single head is a plain row copy of [k_nope | k_pe]
        np.testing.assert_array_equal(key[:, 0], np.concatenate([kvb[:, :128], ws[:, 512:]], 1))


@pytest.mark.parametrize("kpe_fp8", [False, True])
def test_fp8_pack_equals_brute_force_encoder(orc, kpe_fp8):
    pw, kvb, ws = _pack_inputs(H=4, kpe_fp8=kpe_fp8)
    T, rs = kvb.shape
    H, scale = 4, 0.01
    key, v = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, ws[:, 512:], ENTRY,
                                 1 if kpe_fp8 else 0, T, H, 128, 64, 128, out_dtype=1,
                                 out_scale=scale)
    heads = R.bf16_to_f32(kvb[:, : H * 256]).reshape(T, H, 256)
    enc = lambda a: R.fp8_nearest((a / np.float32(scale)).astype(np.float32), 1).reshape(a.shape)
    np.testing.assert_array_equal(key[:, :, :128], enc(heads[:, :, :128]))
    np.testing.assert_array_equal(v, enc(heads[:, :, 128:]))
    if kpe_fp8:  # fp8 k_pe bytes are copied, not rescaled
        np.testing.assert_array_equal(key[:, :, 128:], np.broadcast_to(ws[:, None, 512:], (T, H, 64)))
    else:
        pe = enc(R.bf16_to_f32(ws[:, 512:]))
        np.testing.assert_array_equal(key[:, :, 128:], np.broadcast_to(pe[:, None], (T, H, 64)))


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_fused_pack_equals_stepwise_chain(orc, out_dtype):
    """gather -> cast to the kv_b_proj dtype -> concat -> (fp8) cast, each step
    a separate oracle call, equals the fused pack on the gathered k_pe."""
    pw = W.pack_workload(num_tokens=300, chunk=300, num_blocks=8, block_size=64, seed=10)
    T, H = 300, 16
    cu = np.array([0, T], np.int32)
    ws = np.zeros((T, ENTRY), np.uint8)
    orc.context_gather(pw.cache, 1, 8, 64, 64 * ENTRY, ENTRY, ENTRY, pw.block_table, cu,
                       np.array([0], np.int32), ws, 1)
    kvb = pw.kv_b_proj[0]
    rs = kvb.shape[1]
    # step by step
    latent_bf16 = orc.cast_rows(ws, 1, 0)
    key_bf16 = orc.concat_key(kvb, rs, 256, np.ascontiguousarray(latent_bf16[:, 512:]), 64, T,
                              H, 128, 64)
    v_bf16 = np.ascontiguousarray(kvb[:, : H * 256].reshape(T, H, 256)[:, :, 128:])
    if out_dtype == 0:
        key_ref, v_ref = key_bf16, v_bf16
    else:
        enc = lambda a: orc.fp8_encode((R.bf16_to_f32(a) / np.float32(0.01)).astype(np.float32), 1).reshape(a.shape)
        key_ref, v_ref = enc(key_bf16), enc(v_bf16)
        key_ref[:, :, 128:] = ws[:, None, 512:]  # fp8 k_pe travels as raw bytes
    key, v = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, ws[:, 512:], ENTRY, 1, T,
                                 H, 128, 64, 128, out_dtype=out_dtype, out_scale=0.01)
    np.testing.assert_array_equal(key, key_ref)
    np.testing.assert_array_equal(v, v_ref)
