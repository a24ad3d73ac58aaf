"""The oracle's row loops split over host threads (the multi-core CPU baseline)
give byte-identical results to the single-threaded oracle.

The rows are independent in the pages' definitions: an insert row writes only
the cache row its slot names, and valid slots are distinct within a layer
("PR #55356 [Kimi Perf] Group fp8 mla cache insertion", Source snippets: one
row per (token, layer)); a gather row and a pack token write only their own
output rows ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V
packing", Implementation items 1-2).  So any split of the rows must give the
same bytes, including the rows it leaves untouched and the error bits.
"""
import numpy as np
import pytest

from pack_mla_cache_gb300 import workloads as W

THREADS = [1, 2, 3, 8, 13]


@pytest.mark.parametrize("threads", THREADS)
@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_split_insert_is_byte_identical(orc, threads, shared, fmt):
    wl = W.insert_workload(5, 203, fmt, num_blocks=8, block_size=64, shared_slots=shared,
                           norm=True, rope=True, pad_last=True, seed=11)
    # one out-of-range slot, so the error bits are compared too
    wl.slot_mapping[:, 7] = wl.num_blocks * wl.block_size + 3
    table = orc.rope_cos_sin_cache(W.MAX_POSITION, W.PE_DIM, W.ROPE_BASE)
    fill = 0xABCD if fmt == 0 else 0x5A
    ref, got = wl.empty_caches(fill), wl.empty_caches(fill)
    args = (wl.slot_mapping, wl.slot_layer_stride)
    kw = dict(gamma=wl.gamma, eps=wl.eps, positions=wl.positions, cos_sin_cache=table)
    e1 = orc.insert_grouped(wl.kv_c, wl.k_pe, *args, ref, wl.k_scales, fmt, wl.num_blocks,
                            wl.block_size, wl.block_stride, wl.entry_stride, **kw)
    e2 = orc.insert_grouped_split(threads, wl.kv_c, wl.k_pe, *args, got, wl.k_scales, fmt,
                                  wl.num_blocks, wl.block_size, wl.block_stride,
                                  wl.entry_stride, **kw)
    assert e1 == e2 == orc.ERR_SLOT_OOB
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("threads", THREADS)
@pytest.mark.parametrize("out_dtype", [1, 0])
def test_split_gather_is_byte_identical(orc, threads, out_dtype):
    pw = W.pack_workload(1000, 1000, num_blocks=40, seed=5)
    # three sequences over 1000 rows with a gap of unowned rows (900..999), a
    # sequence starting mid-block and one whose rows run past its block table
    cu = np.array([0, 300, 650, 900], np.int32)
    starts = np.array([17, 0, 380], np.int32)
    bt = np.ascontiguousarray(np.repeat(pw.block_table[:, :8], 3, axis=0))
    bt[2, 4] = 10 ** 6  # bad block id
    odt = np.uint16 if out_dtype == 0 else np.uint8
    ref = np.full((1000, 576), 0x77, odt)
    got = ref.copy()
    args = (pw.cache, 1, pw.num_blocks, 64, 64 * 576, 576, 576, bt, cu, starts)
    e1 = orc.context_gather(*args, ref, out_dtype)
    e2 = orc.context_gather_split(threads, *args, got, out_dtype)
    assert e1 == e2 == orc.ERR_BLOCK_OOB
    np.testing.assert_array_equal(ref, got)


@pytest.mark.parametrize("threads", THREADS)
@pytest.mark.parametrize("out_dtype,kpe_dtype", [(1, 1), (0, 0), (0, 1), (2, 0)])
def test_split_pack_is_byte_identical(orc, threads, out_dtype, kpe_dtype):
    T, H = 157, 5
    pw = W.pack_workload(T, T, num_blocks=4, num_heads=H, seed=9)
    kvb = pw.kv_b_proj[0]
    rs = kvb.shape[1]
    if kpe_dtype == 0:
        kpe = np.ascontiguousarray(kvb[:, H * 256:H * 256 + 64])
    else:
        kpe = np.ascontiguousarray(pw.cache[:T * 576].reshape(T, 576)[:, 512:])
    args = (kvb, rs, 256, kvb[:, 128:], rs, 256, kpe, kpe.shape[1], kpe_dtype, T, H, 128, 64,
            128, out_dtype, 0.01)
    k1, v1 = orc.context_kv_pack(*args)
    k2, v2 = orc.context_kv_pack_split(threads, *args)
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(v1, v2)


def test_host_threads_is_positive(orc):
    assert orc.host_threads() >= 1
