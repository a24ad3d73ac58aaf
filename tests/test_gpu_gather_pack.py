"""GPU parity of the context gather and the K/V pack against the CPU oracle,
through the C ABI -- all bit-exact ("PR #51772 [Attention][MLA] Fuse Kimi-K3
chunked-context K/V packing": the fused loop must equal the generic one
chunk by chunk with atol=0/rtol=0, and the fp8 cast must be bit-identical).

Covers: 32768 context tokens in 4 chunks of 8192 from an fp8 e4m3 cache
(1024 blocks, random block table), raw and bf16-widened gathers, kv_b_proj
output [8192, 4160] bf16 packed to fp8 e4m3 (scale 0.01) and to bf16, head
counts 16 / 3 / 4 (runtime), 0 and ragged token counts, e5m2 output, bf16
k_pe into fp8, no-V packs, several sequences per gather, bad block ids, a
32768-row gather whose warps loop, tables written by kernels just before each
gather, the 16-chunk programmatic-dependent-launch chain, and one
131072-token launch of the grid-capped grid-stride loop (sampled).
"""
import numpy as np
import pytest
import torch

import devutil as D
import refmath as R
from pack_mla_cache_gb300 import ops
from pack_mla_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu
ENTRY = 576


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pack_mla_cache_gb300 import build
    build.build()
    ops.lib()


def dev_cache(pw):
    if pw.cache_dtype == 0:
        return D.dev_bf16(pw.cache)
    return D.dev(pw.cache)


def gpu_gather(pw, cache_t, table, cu, starts, T, out_dtype, err=None):
    out = torch.full((T, ENTRY), 0x3F if out_dtype else 0x3F3F, dtype=torch.int16 if out_dtype == 0 else torch.uint8,
                     device="cuda")
    if out_dtype == 0:
        out = out.view(torch.bfloat16)
    ops.mla_context_gather(cache_t, pw.cache_dtype, pw.num_blocks, pw.block_size,
                           pw.block_size * ENTRY, ENTRY, ENTRY, D.dev(table), D.dev(cu),
                           D.dev(starts), out, out_dtype, err_word=err)
    torch.cuda.synchronize()
    return D.host_u16(out) if out_dtype == 0 else D.host_u8(out)


def oracle_gather(orc, pw, table, cu, starts, T, out_dtype):
    out = np.full((T, ENTRY), 0x3F if out_dtype else 0x3F3F, np.uint8 if out_dtype else np.uint16)
    err = orc.context_gather(pw.cache, pw.cache_dtype, pw.num_blocks, pw.block_size,
                             pw.block_size * ENTRY, ENTRY, ENTRY, table, cu, starts, out, out_dtype)
    return out, err


@pytest.mark.parametrize("out_dtype", [1, 0])
def test_gather_four_chunks_of_8192(orc, out_dtype):
    pw = W.pack_workload(32768, 8192, num_blocks=1024, seed=1)
    cache_t = dev_cache(pw)
    for c in range(4):
        cu = np.array([0, 8192], np.int32)
        st = np.array([c * 8192], np.int32)
        g = gpu_gather(pw, cache_t, pw.block_table, cu, st, 8192, out_dtype)
        r, err = oracle_gather(orc, pw, pw.block_table, cu, st, 8192, out_dtype)
        assert err == 0
        np.testing.assert_array_equal(g, r)


def test_gather_many_sequences_and_bad_blocks(orc):
    pw = W.pack_workload(4096, 4096, num_blocks=128, seed=2)
    cache_t = dev_cache(pw)
    rng = np.random.default_rng(0)
    S = 37
    table = rng.integers(0, 128, size=(S, 8)).astype(np.int32)
    table[5, 1] = 128    # block id out of range
    table[9, 0] = -3
    lens = rng.integers(0, 200, size=S)
    starts = rng.integers(0, 300, size=S).astype(np.int32)  # positions up to 500 < 8 * 64
    # sequence 5 reaches its bad block 1 (positions 10..159), sequence 9 its
    # bad block 0 (positions 0..19)
    lens[5], starts[5] = 150, 10
    lens[9], starts[9] = 20, 0
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1]) + 5  # 5 trailing rows owned by no sequence
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = gpu_gather(pw, cache_t, table, cu, starts, T, 1, err=err)
    r, oerr = oracle_gather(orc, pw, table, cu, starts, T, 1)
    np.testing.assert_array_equal(g, r)
    assert oerr == ops.MLA_ERRBIT_BLOCK_OOB
    assert int(err.item()) == oerr


def test_gather_one_launch_of_32768_rows_with_bad_blocks(orc):
    """One raw gather of 32768 rows: more rows than the capped grid has warps
    (152 SMs x 64), so each warp's first row is looked up before the launch
    wait and its later rows inside the loop.  A bad block id in the table row
    of the first rows and one in that of rows the loop reaches: both skip their
    rows and set the error bit."""
    pw = W.pack_workload(32768, 8192, num_blocks=1024, seed=11)
    table = pw.block_table.copy()
    table[0, 0] = 1024          # rows 0..63: out of range (first lookups)
    table[0, 500] = -1          # rows 32000..32063: negative (looped rows)
    cu = np.array([0, 32768], np.int32)
    st = np.array([0], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = gpu_gather(pw, dev_cache(pw), table, cu, st, 32768, 1, err=err)
    r, oerr = oracle_gather(orc, pw, table, cu, st, 32768, 1)
    assert oerr == ops.MLA_ERRBIT_BLOCK_OOB
    assert int(err.item()) == oerr
    np.testing.assert_array_equal(g, r)


@pytest.mark.parametrize("early", [False, True], ids=["stream_order", "early_tables"])
def test_gather_sees_tables_written_just_before_it(orc, early):
    """With programmatic dependent launch on, tables written by ordinary
    kernels enqueued just before each call on the same stream (they trigger no
    early launch) are the ones the gather reads, both in plain stream order
    (the default) and when the gather reads its tables before waiting on the
    previous grid (mla_set_gather_early_tables)."""
    pw = W.pack_workload(16448, 8192, num_blocks=512, seed=12)  # positions up to 16386
    cache_t = dev_cache(pw)
    src_table = D.dev(pw.block_table)
    table_t = torch.zeros_like(src_table)
    cu_t = torch.zeros(2, dtype=torch.int32, device="cuda")
    st_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = torch.zeros((2, 8192, ENTRY), dtype=torch.uint8, device="cuda")
    prev = ops.mla_set_pdl(True)
    prev_early = ops.mla_set_gather_early_tables(early)
    try:
        for c in range(2):
            table_t.zero_()
            table_t.add_(src_table)
            cu_t.fill_(8192)
            cu_t[0].fill_(0)
            st_t.fill_(c * 8192 + 3)
            ops.mla_context_gather(cache_t, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY,
                                   table_t, cu_t, st_t, outs[c], 1)
            if c == 0:
                # scramble the tables after the first call (kernels again)
                table_t.fill_(-1)
                st_t.fill_(10 ** 6)
        torch.cuda.synchronize()
    finally:
        ops.mla_set_pdl(prev)
        ops.mla_set_gather_early_tables(prev_early)
    for c in range(2):
        cu = np.array([0, 8192], np.int32)
        st = np.array([c * 8192 + 3], np.int32)
        r, err = oracle_gather(orc, pw, pw.block_table, cu, st, 8192, 1)
        assert err == 0
        np.testing.assert_array_equal(D.host_u8(outs[c]), r)


def test_gather_default_order_sees_a_table_written_by_a_pdl_kernel(orc):
    """In the default (plain stream order) the gather reads its block table
    only after the previous grid has completed, even when that grid is a
    library kernel that lets its dependents launch at its start: here a first
    gather (PDL on, early trigger) copies the second gather's block table out of
    a cache row into the table buffer, which held only invalid block ids."""
    pw = W.pack_workload(8192, 8192, num_blocks=256, seed=13)
    cache_t = dev_cache(pw)
    want = pw.block_table[0, :128].astype(np.int32)  # the 128 blocks of 8192 rows
    # a one-block fp8 "cache" whose row 0 holds the table's bytes (576 B row)
    src = np.zeros(64 * ENTRY, np.uint8)
    src[:512] = want.view(np.uint8)
    src_t = D.dev(src)
    one = torch.zeros((1, 144), dtype=torch.int32, device="cuda")  # out: 576 B = 144 int32
    one.fill_(-1)
    cu1 = D.dev(np.array([0, 1], np.int32))
    st1 = D.dev(np.array([0], np.int32))
    bt1 = D.dev(np.zeros((1, 1), np.int32))
    cu = D.dev(np.array([0, 8192], np.int32))
    st = D.dev(np.array([0], np.int32))
    out = torch.zeros((8192, ENTRY), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = ops.mla_set_pdl(True)
    prev_early = ops.mla_set_gather_early_tables(False)
    try:
        for _ in range(3):
            one.fill_(-1)
            ops.mla_context_gather(src_t, 1, 1, 64, 64 * ENTRY, ENTRY, ENTRY, bt1, cu1, st1,
                                   one.view(torch.uint8).view(1, 576), 1)
            ops.mla_context_gather(cache_t, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY,
                                   one[:, :128], cu, st, out, 1, err_word=err)
        torch.cuda.synchronize()
    finally:
        ops.mla_set_pdl(prev)
        ops.mla_set_gather_early_tables(prev_early)
    assert int(err.item()) == 0
    r, oerr = oracle_gather(orc, pw, pw.block_table, np.array([0, 8192], np.int32),
                            np.array([0], np.int32), 8192, 1)
    assert oerr == 0
    np.testing.assert_array_equal(D.host_u8(out), r)


def test_gather_bf16_cache_raw(orc):
    pw = W.pack_workload(3000, 3000, num_blocks=64, cache_dtype=0, seed=3)
    cu = np.array([0, 3000], np.int32)
    st = np.array([0], np.int32)
    g = gpu_gather(pw, dev_cache(pw), pw.block_table, cu, st, 3000, 0)
    r, _ = oracle_gather(orc, pw, pw.block_table, cu, st, 3000, 0)
    np.testing.assert_array_equal(g, r)


@pytest.mark.parametrize("fmt", [1, 2])
def test_gather_widens_every_fp8_code(orc, fmt):
    """A cache row holding every byte value: the widening is exact for all 256
    codes (NaNs become the signed quiet NaN)."""
    pw = W.pack_workload(64, 64, num_blocks=1, cache_dtype=fmt, seed=4)
    pw.cache[:] = (np.arange(pw.cache.size) % 256).astype(np.uint8)
    cu = np.array([0, 64], np.int32)
    st = np.array([0], np.int32)
    g = gpu_gather(pw, dev_cache(pw), pw.block_table, cu, st, 64, 0)
    r, _ = oracle_gather(orc, pw, pw.block_table, cu, st, 64, 0)
    np.testing.assert_array_equal(g, r)


@pytest.mark.parametrize("fmt", [1, 2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("out_dtype", [0, 3], ids=["bf16", "fp16"])
def test_widening_nan_codes_at_every_byte_position(orc, fmt, out_dtype):
    """The widening sends a group of 8 codes (8 bytes) through the hardware
    conversion alone unless the group holds a NaN code.  Here every other
    group of every row holds one NaN code of the format (each sign, each NaN
    pattern) at a byte position that runs through 0..7, between finite codes
    and next to groups without a NaN: every row equals the oracle's."""
    pw = W.pack_workload(64, 64, num_blocks=1, cache_dtype=fmt, seed=4)
    nan_codes = [0x7F, 0xFF] if fmt == 1 else [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    finite = np.array([c for c in range(256) if c not in nan_codes], np.uint8)
    rows = pw.cache.reshape(-1, ENTRY)[:64]
    rows[:] = np.random.default_rng(11).choice(finite, size=rows.shape)
    for r in range(64):
        for g in range(0, ENTRY // 8, 2):
            rows[r, 8 * g + (r + g) % 8] = nan_codes[(7 * r + g) % len(nan_codes)]
    cu, st = np.array([0, 64], np.int32), np.array([0], np.int32)
    out = torch.full((64, ENTRY), 0x1234, dtype=torch.int16, device="cuda")
    out = out.view(torch.bfloat16 if out_dtype == 0 else torch.float16)
    ops.mla_context_gather(dev_cache(pw), fmt, pw.num_blocks, pw.block_size,
                           pw.block_size * ENTRY, ENTRY, ENTRY, D.dev(pw.block_table), D.dev(cu),
                           D.dev(st), out, out_dtype)
    torch.cuda.synchronize()
    ref = np.full((64, ENTRY), 0x1234, np.uint16)
    err = orc.context_gather(pw.cache, fmt, pw.num_blocks, pw.block_size, pw.block_size * ENTRY,
                             ENTRY, ENTRY, pw.block_table, cu, st, ref, out_dtype)
    assert err == 0
    np.testing.assert_array_equal(D.host_u16(out), ref)


# -------------------------------------------------------------------------- pack
def pack_io(kvb, ws, H, out_dtype, kpe_fp8, with_v=True):
    """Device views of a kv_b_proj output [T, >= H*256] and a gather workspace
    [T, 576] (k_pe = columns 512:576), and fresh outputs."""
    T = kvb.shape[0]
    kvb_t = D.dev_bf16(kvb)
    heads = kvb_t[:, : H * 256].view(T, H, 256)
    k_nope, v = heads[:, :, :128], heads[:, :, 128:]
    ws_t = D.dev(ws) if kpe_fp8 else D.dev_bf16(ws)
    k_pe = ws_t[:, 512:]
    odt = torch.bfloat16 if out_dtype == 0 else torch.uint8
    key = torch.zeros((T, H, 192), dtype=odt, device="cuda")
    vout = torch.zeros((T, H, 128), dtype=odt, device="cuda") if with_v else None
    return k_nope, v, k_pe, key, vout


def run_pack(kvb, ws, H, out_dtype, kpe_dtype, scale=0.01, with_v=True):
    k_nope, v, k_pe, key, vout = pack_io(kvb, ws, H, out_dtype, kpe_dtype != 0, with_v)
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda") if out_dtype != 0 else None
    ops.mla_context_kv_pack(k_nope, v, k_pe, key, vout, out_dtype, kpe_dtype=kpe_dtype,
                            out_scale=sc)
    torch.cuda.synchronize()
    conv = D.host_u16 if out_dtype == 0 else D.host_u8
    return conv(key), (conv(vout) if with_v else None)


def oracle_pack(orc, kvb, ws, H, out_dtype, kpe_dtype, scale=0.01, with_v=True):
    T, rs = kvb.shape
    return orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, ws[:, 512:], ENTRY,
                               kpe_dtype, T, H, 128, 64, 128, out_dtype,
                               scale if out_dtype != 0 else 1.0, with_v)


def workspace(orc, pw, T, start, out_dtype):
    ws = np.zeros((T, ENTRY), np.uint8 if out_dtype else np.uint16)
    orc.context_gather(pw.cache, 1, pw.num_blocks, pw.block_size, pw.block_size * ENTRY, ENTRY,
                       ENTRY, pw.block_table, np.array([0, T], np.int32),
                       np.array([start], np.int32), ws, out_dtype)
    return ws


@pytest.mark.parametrize("out_dtype,kpe_dtype", [(1, 1), (0, 0), (0, 1), (1, 0), (2, 0)])
def test_pack_8192_token_chunk(orc, out_dtype, kpe_dtype):
    pw = W.pack_workload(8192, 8192, num_blocks=256, seed=5)
    ws = workspace(orc, pw, 8192, 0, 1 if kpe_dtype else 0)
    kvb = pw.kv_b_proj[0]
    gk, gv = run_pack(kvb, ws, 16, out_dtype, kpe_dtype)
    rk, rv = oracle_pack(orc, kvb, ws, 16, out_dtype, kpe_dtype)
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)


@pytest.mark.parametrize("H", [1, 3, 4, 20])
@pytest.mark.parametrize("T", [1, 77, 1000])
def test_pack_runtime_heads_and_ragged_tokens(orc, H, T):
    pw = W.pack_workload(T, T, num_blocks=16, seed=6, num_heads=H)
    ws = workspace(orc, pw, T, 0, 1)
    kvb = pw.kv_b_proj[0]
    for out_dtype in (1, 0):
        gk, gv = run_pack(kvb, ws, H, out_dtype, 1)
        rk, rv = oracle_pack(orc, kvb, ws, H, out_dtype, 1)
        np.testing.assert_array_equal(gk, rk)
        np.testing.assert_array_equal(gv, rv)


@pytest.mark.parametrize("scale", [0.01, 3.0])
def test_fp8_pack_exhaustive_over_bf16(orc, scale):
    """kv_b_proj output holding all 2^16 bf16 patterns (16 tokens x 16 heads x
    256): the fp8 key and V are bit-exact (zeros, subnormals, overflowing
    quotients, infinities, NaNs)."""
    T, H = 16, 16
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(T, H * 256)
    kvb = np.zeros((T, 4160), np.uint16)
    kvb[:, : H * 256] = pats
    ws = np.random.default_rng(0).integers(0, 126, size=(T, ENTRY)).astype(np.uint8)
    gk, gv = run_pack(kvb, ws, H, 1, 1, scale=scale)
    rk, rv = oracle_pack(orc, kvb, ws, H, 1, 1, scale=scale)
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)


def test_pack_separate_k_nope_and_v_buffers(orc):
    """k_nope and v from two different tensors with their own strides (not
    the interleaved kv_b_proj halves)."""
    T, H = 600, 16
    pw = W.pack_workload(T, T, num_blocks=16, seed=13)
    ws = workspace(orc, pw, T, 0, 1)
    g = torch.Generator().manual_seed(3)
    kn_h = torch.randn((T, H, 160), generator=g).to(torch.bfloat16)   # head stride 160
    v_h = torch.randn((H, T, 128), generator=g).to(torch.bfloat16)    # head-major
    k_nope = kn_h.cuda()[:, :, :128]
    v = v_h.cuda().permute(1, 0, 2)
    key = torch.zeros((T, H, 192), dtype=torch.uint8, device="cuda")
    vo = torch.zeros((T, H, 128), dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    ops.mla_context_kv_pack(k_nope, v, D.dev(ws)[:, 512:], key, vo, 1, kpe_dtype=1, out_scale=sc)
    torch.cuda.synchronize()
    kn_np = kn_h.view(torch.int16).numpy().view(np.uint16)
    v_np = v_h.view(torch.int16).numpy().view(np.uint16)
    rk, rv = orc.context_kv_pack(kn_np.reshape(-1), H * 160, 160, v_np.reshape(-1), 128, T * 128,
                                 ws[:, 512:], ENTRY, 1, T, H, 128, 64, 128, 1, 0.01)
    np.testing.assert_array_equal(D.host_u8(key), rk)
    np.testing.assert_array_equal(D.host_u8(vo), rv)


def test_pack_without_v(orc):
    pw = W.pack_workload(500, 500, num_blocks=8, seed=7)
    ws = workspace(orc, pw, 500, 0, 0)
    gk, gv = run_pack(pw.kv_b_proj[0], ws, 16, 0, 0, with_v=False)
    rk, _ = oracle_pack(orc, pw.kv_b_proj[0], ws, 16, 0, 0, with_v=False)
    assert gv is None
    np.testing.assert_array_equal(gk, rk)


def test_pack_zero_tokens():
    kvb = np.zeros((0, 4160), np.uint16)
    ws = np.zeros((0, ENTRY), np.uint8)
    gk, gv = run_pack(kvb, ws, 16, 1, 1)
    assert gk.size == 0 and gv.size == 0


def test_fused_pack_equals_stepwise_chain_on_gpu(orc):
    """GPU gather -> GPU pack on the gathered fp8 k_pe equals the oracle's
    step-by-step chain gather -> cast -> concat -> cast, for both outputs."""
    pw = W.pack_workload(8192, 8192, num_blocks=256, seed=8)
    cache_t = dev_cache(pw)
    cu = np.array([0, 8192], np.int32)
    st = np.array([0], np.int32)
    ws_g = gpu_gather(pw, cache_t, pw.block_table, cu, st, 8192, 1)
    kvb = pw.kv_b_proj[0]
    T, rs = kvb.shape
    ws_o, _ = oracle_gather(orc, pw, pw.block_table, cu, st, 8192, 1)
    latent = orc.cast_rows(ws_o, 1, 0)
    key_bf16 = orc.concat_key(kvb, rs, 256, np.ascontiguousarray(latent[:, 512:]), 64, T, 16,
                              128, 64)
    v_bf16 = np.ascontiguousarray(kvb[:, :4096].reshape(T, 16, 256)[:, :, 128:])
    # bf16 output from the widened k_pe
    gk, gv = run_pack(kvb, orc.cast_rows(ws_g, 1, 0), 16, 0, 0)
    np.testing.assert_array_equal(gk, key_bf16)
    np.testing.assert_array_equal(gv, v_bf16)
    # fp8 output: k_nope / v cast with the scale, k_pe bytes copied raw
    gk, gv = run_pack(kvb, ws_g, 16, 1, 1)
    enc = lambda a: orc.fp8_encode((R.bf16_to_f32(a) / np.float32(0.01)).astype(np.float32), 1).reshape(a.shape)
    ref_key = enc(key_bf16)
    ref_key[:, :, 128:] = ws_o[:, None, 512:]
    np.testing.assert_array_equal(gk, ref_key)
    np.testing.assert_array_equal(gv, enc(v_bf16))


def test_sixteen_chunk_pdl_chain(orc):
    """16 chunks x 8192 tokens, each a gather into ONE reused workspace then a
    pack, back to back on one stream with programmatic dependent launch: every
    chunk's outputs equal the oracle's (sampled rows), so no kernel read a
    workspace before the previous one finished writing it."""
    pw = W.pack_workload(131072, 8192, num_blocks=2048, seed=9, distinct_chunks=False)
    cache_t = dev_cache(pw)
    table_t = D.dev(pw.block_table)
    kvb = pw.kv_b_proj[0]
    k_nope, v, _, _, _ = pack_io(kvb, np.zeros((8192, ENTRY), np.uint8), 16, 1, True)
    ws = torch.empty((8192, ENTRY), dtype=torch.uint8, device="cuda")
    keys = torch.empty((16, 8192, 16, 192), dtype=torch.uint8, device="cuda")
    vs = torch.empty((16, 8192, 16, 128), dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    cu = D.dev(np.array([0, 8192], np.int32))
    starts = [D.dev(np.array([c * 8192], np.int32)) for c in range(16)]
    ops.mla_set_pdl(True)
    for c in range(16):
        ops.mla_context_gather(cache_t, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY, table_t,
                               cu, starts[c], ws, 1)
        ops.mla_context_kv_pack(k_nope, v, ws[:, 512:], keys[c], vs[c], 1, kpe_dtype=1,
                                out_scale=sc)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    keys_h, vs_h = D.host_u8(keys), D.host_u8(vs)
    for c in range(16):
        ws_o = workspace(orc, pw, 8192, c * 8192, 1)
        rows = np.sort(rng.choice(8192, 256, replace=False))
        sub = np.ascontiguousarray(kvb[rows])
        rk, rv = oracle_pack(orc, sub, np.ascontiguousarray(ws_o[rows]), 16, 1, 1)
        np.testing.assert_array_equal(keys_h[c][rows], rk)
        np.testing.assert_array_equal(vs_h[c][rows], rv)


def test_one_launch_of_131072_tokens_sampled(orc):
    """One 131072-token pack launch (the grid is capped at the resident CTAs,
    so every warp loops over many tokens): 4096 sampled tokens equal the
    oracle and the output is written exactly once (guard bands intact)."""
    T = 131072
    g = torch.Generator().manual_seed(10)
    kvb_t = (torch.randn((T, 4160), generator=g)).to(torch.bfloat16).cuda()
    ws_t = torch.randint(0, 256, (T, ENTRY), generator=g, dtype=torch.int32).to(torch.uint8)
    ws_t[(ws_t & 0x7F) == 0x7F] = 0  # finite codes only
    ws_t = ws_t.cuda()
    heads = kvb_t[:, :4096].view(T, 16, 256)
    key = D.Guarded(T * 16 * 192)
    vo = D.Guarded(T * 16 * 128)
    sc = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:], ws_t[:, 512:],
                            key.t.view(T, 16, 192), vo.t.view(T, 16, 128), 1, kpe_dtype=1,
                            out_scale=sc)
    torch.cuda.synchronize()
    assert key.guards_intact() and vo.guards_intact()
    rows = np.sort(np.random.default_rng(2).choice(T, 4096, replace=False))
    kvb = D.host_u16(kvb_t[rows])
    ws = D.host_u8(ws_t[rows])
    rk, rv = oracle_pack(orc, kvb, ws, 16, 1, 1)
    np.testing.assert_array_equal(key.host().reshape(T, 16, 192)[rows], rk)
    np.testing.assert_array_equal(vo.host().reshape(T, 16, 128)[rows], rv)
