"""GPU parity of the scaled dequantising gather and of the pack that reads
k_pe straight from the paged cache, against the CPU oracle, through the C ABI
-- all bit-exact.

Scaled gather: every fp8 code of both formats at scales that give normal,
subnormal, overflowing and NaN products (zero, infinite and NaN scales too);
four 8192-token chunks at a k_scale drawn like the insert's; 37 sequences with
bad block ids (error word); the kv_c-only 512-column gather into padded rows.

Paged pack ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V
packing", Implementation item 1, with k_pe read from the cache itself): every
cache/output dtype pair on an 8192-token chunk; several sequences with
unaligned starts, bad block ids and unowned tokens (rope slice untouched,
error word); 40 sequences (the binary-search lookup); runtime head counts and
ragged token counts; no-V; zero tokens; the GPU's own gather-then-pack path
gives the same bytes; one 131072-token launch (sampled against the oracle,
whole against the two-kernel path).
"""
import math

import numpy as np
import pytest
import torch

import devutil as D
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
    return D.dev_bf16(pw.cache) if pw.cache_dtype == 0 else D.dev(pw.cache)


def f32(x):
    return torch.tensor([x], dtype=torch.float32, device="cuda")


# ------------------------------------------------------------- scaled gather
def gpu_gather_scaled(pw, cache_t, table, cu, starts, T, scale, *, edim=ENTRY, ors=ENTRY,
                      err=None, fill=0x3F3F):
    out = torch.full((T, ors), fill, dtype=torch.int32, device="cuda").to(torch.int16)
    ops.mla_context_gather_scaled(cache_t, pw.cache_dtype, pw.num_blocks, pw.block_size,
                                  pw.block_size * ENTRY, ENTRY, edim, D.dev(table), D.dev(cu),
                                  D.dev(starts), out.view(torch.bfloat16), f32(scale),
                                  err_word=err)
    torch.cuda.synchronize()
    return D.host_u16(out)


def oracle_gather_scaled(orc, pw, table, cu, starts, T, scale, *, edim=ENTRY, ors=ENTRY,
                         fill=0x3F3F):
    out = np.full((T, ors), fill, np.uint16)
    err = orc.context_gather_scaled(pw.cache, pw.cache_dtype, pw.num_blocks, pw.block_size,
                                    pw.block_size * ENTRY, ENTRY, edim, table, cu, starts, out,
                                    scale)
    return out, err


SCALES = [0.0173, 1.0, 3.7, 123456.7, -0.37, 2.5e-38, 7e-41, 1e-45, 2.0 ** 120, 0.0,
          math.inf, -math.inf, math.nan]


@pytest.mark.parametrize("fmt", [1, 2])
def test_scaled_gather_every_code_every_scale(orc, fmt):
    pw = W.pack_workload(64, 64, num_blocks=1, cache_dtype=fmt, seed=4)
    pw.cache[:] = (np.arange(pw.cache.size) % 256).astype(np.uint8)
    cache_t = dev_cache(pw)
    cu, st = np.array([0, 64], np.int32), np.array([0], np.int32)
    for sc in SCALES:
        g = gpu_gather_scaled(pw, cache_t, pw.block_table, cu, st, 64, sc)
        r, err = oracle_gather_scaled(orc, pw, pw.block_table, cu, st, 64, sc)
        assert err == 0
        np.testing.assert_array_equal(g, r, err_msg=f"scale {sc}")


def test_scaled_gather_four_chunks_of_8192(orc):
    pw = W.pack_workload(32768, 8192, num_blocks=1024, seed=1)
    cache_t = dev_cache(pw)
    scale = float(np.float32(np.random.default_rng(5).uniform(0.005, 0.02)))
    for c in range(4):
        cu, st = np.array([0, 8192], np.int32), np.array([c * 8192], np.int32)
        g = gpu_gather_scaled(pw, cache_t, pw.block_table, cu, st, 8192, scale)
        r, err = oracle_gather_scaled(orc, pw, pw.block_table, cu, st, 8192, scale)
        assert err == 0
        np.testing.assert_array_equal(g, r)


def test_scaled_gather_many_sequences_and_bad_blocks(orc):
    pw = W.pack_workload(4096, 4096, num_blocks=128, seed=2, cache_dtype=2)
    rng = np.random.default_rng(0)
    S = 37
    table = rng.integers(0, 128, size=(S, 8)).astype(np.int32)
    table[5, :], table[9, 0] = 128, -3  # every block id of sequence 5 out of range
    lens = rng.integers(0, 200, size=S)
    lens[5] = max(lens[5], 1)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    starts = rng.integers(0, 300, size=S).astype(np.int32)
    T = int(cu[-1]) + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = gpu_gather_scaled(pw, dev_cache(pw), table, cu, starts, T, 0.011, err=err)
    r, oerr = oracle_gather_scaled(orc, pw, table, cu, starts, T, 0.011)
    np.testing.assert_array_equal(g, r)
    assert int(err.item()) == oerr == ops.MLA_ERRBIT_BLOCK_OOB


def test_scaled_gather_kv_c_columns_into_padded_rows(orc):
    """entry_dim 512 (kv_c only) into rows of stride 640: columns 512.. stay."""
    pw = W.pack_workload(3000, 3000, num_blocks=64, seed=3)
    cu, st = np.array([0, 3000], np.int32), np.array([17], np.int32)
    g = gpu_gather_scaled(pw, dev_cache(pw), pw.block_table, cu, st, 3000, 0.02, edim=512,
                          ors=640)
    r, _ = oracle_gather_scaled(orc, pw, pw.block_table, cu, st, 3000, 0.02, edim=512, ors=640)
    np.testing.assert_array_equal(g, r)
    assert (g[:, 512:] == 0x3F3F).all()


# ---------------------------------------------------------------- paged pack
class PagedCase:
    def __init__(self, cache_dtype, T, H=16, *, seqs=None, seed=11, num_blocks=256):
        ctx = max(T + 512, 4096)
        self.pw = W.pack_workload(ctx, ctx, num_blocks=max(num_blocks, (ctx + 63) // 64),
                                  cache_dtype=cache_dtype, seed=seed, num_heads=H)
        self.T, self.H = T, H
        if seqs is None:  # one sequence starting mid-block
            self.table = self.pw.block_table
            self.cu = np.array([0, T], np.int32)
            self.starts = np.array([37], np.int32)
        else:
            self.table, self.cu, self.starts = seqs
        self.kvb = W.pack_workload(T, T, num_blocks=(T + 63) // 64, num_heads=H,
                                   seed=seed + 1).kv_b_proj[0] \
            if T > 0 else np.zeros((0, H * 256 + 64), np.uint16)
        self.cache_t = dev_cache(self.pw)

    def gpu(self, out_dtype, *, scale=0.01, with_v=True, err=None, key_fill=0x5A):
        T, H = self.T, self.H
        kvb_t = D.dev_bf16(self.kvb)
        heads = kvb_t[:, : H * 256].view(T, H, 256)
        odt = torch.bfloat16 if out_dtype == 0 else torch.uint8
        key = torch.full((T, H, 192), key_fill, dtype=torch.uint8, device="cuda")
        if out_dtype == 0:
            key = torch.full((T, H, 192), key_fill * 0x101, dtype=torch.int32,
                             device="cuda").to(torch.int16).view(torch.bfloat16)
        vout = torch.zeros((T, H, 128), dtype=odt, device="cuda") if with_v else None
        pw = self.pw
        ops.mla_context_kv_pack_paged(
            heads[:, :, :128], heads[:, :, 128:], self.cache_t, pw.cache_dtype, pw.num_blocks,
            pw.block_size, pw.block_size * ENTRY, ENTRY, D.dev(self.table), D.dev(self.cu),
            D.dev(self.starts), key, vout, out_dtype,
            out_scale=f32(scale) if out_dtype else None, err_word=err)
        torch.cuda.synchronize()
        conv = D.host_u16 if out_dtype == 0 else D.host_u8
        return conv(key), (conv(vout) if with_v else None)

    def oracle(self, orc, out_dtype, *, scale=0.01, with_v=True, key_fill=0x5A):
        T, H, pw = self.T, self.H, self.pw
        rs = self.kvb.shape[1]
        odt = np.uint16 if out_dtype == 0 else np.uint8
        init = np.full((T, H, 192), key_fill * 0x101 if out_dtype == 0 else key_fill, odt)
        return orc.context_kv_pack_paged(
            self.kvb, rs, 256, self.kvb[:, 128:], rs, 256, pw.cache, pw.cache_dtype,
            pw.num_blocks, pw.block_size, pw.block_size * ENTRY, ENTRY, 512, self.table, self.cu,
            self.starts, T, H, 128, 64, 128, out_dtype, scale if out_dtype else 1.0, with_v,
            key_init=init)


@pytest.mark.parametrize("cache_dtype,out_dtype", [(1, 1), (1, 0), (2, 2), (2, 0), (0, 0), (0, 1)])
def test_paged_pack_8192_token_chunk(orc, cache_dtype, out_dtype):
    c = PagedCase(cache_dtype, 8192)
    gk, gv = c.gpu(out_dtype)
    rk, rv, err = c.oracle(orc, out_dtype)
    assert err == 0
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)


def _seq_layout(rng, S, nb, T, width=8):
    table = rng.integers(0, nb, size=(S, width)).astype(np.int32)
    lens = rng.multinomial(T - 7, np.ones(S) / S)
    cu = np.concatenate([[3], 3 + np.cumsum(lens)]).astype(np.int32)  # tokens 0-2, T-4.. unowned
    starts = rng.integers(0, 64 * width - lens.max(), size=S).clip(0).astype(np.int32)
    return table, cu, starts


@pytest.mark.parametrize("S", [5, 31, 40])
def test_paged_pack_sequences_bad_blocks_and_unowned_tokens(orc, S):
    rng = np.random.default_rng(S)
    T = 1500
    table, cu, starts = _seq_layout(rng, S, 256, T, width=40)
    table[1, :] = 300        # every block id of sequence 1 out of range
    table[S - 1, 0] = -1
    c = PagedCase(1, T, seqs=(table, cu, starts))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for out_dtype in (1, 0):
        err.zero_()
        gk, gv = c.gpu(out_dtype, err=err)
        rk, rv, oerr = c.oracle(orc, out_dtype)
        np.testing.assert_array_equal(gk, rk)
        np.testing.assert_array_equal(gv, rv)
        assert int(err.item()) == oerr == ops.MLA_ERRBIT_BLOCK_OOB


@pytest.mark.parametrize("H", [1, 3, 20])
@pytest.mark.parametrize("T", [1, 77])
def test_paged_pack_runtime_heads_and_ragged_tokens(orc, H, T):
    c = PagedCase(1, T, H)
    for out_dtype in (1, 0):
        gk, gv = c.gpu(out_dtype)
        rk, rv, _ = c.oracle(orc, out_dtype)
        np.testing.assert_array_equal(gk, rk)
        np.testing.assert_array_equal(gv, rv)


def test_paged_pack_without_v_and_zero_tokens(orc):
    c = PagedCase(0, 500)
    gk, gv = c.gpu(0, with_v=False)
    rk, _, _ = c.oracle(orc, 0, with_v=False)
    assert gv is None
    np.testing.assert_array_equal(gk, rk)
    z = PagedCase(1, 0)
    gk, gv = z.gpu(1)
    assert gk.size == 0 and gv.size == 0


def test_paged_pack_equals_gpu_gather_then_pack():
    """The one-kernel path and the two-kernel path (gather into a workspace,
    pack its k_pe columns) give the same bytes."""
    c = PagedCase(1, 8192, seed=21)
    pw = c.pw
    ws = torch.zeros((8192, ENTRY), dtype=torch.uint8, device="cuda")
    ops.mla_context_gather(c.cache_t, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY,
                           D.dev(c.table), D.dev(c.cu), D.dev(c.starts), ws, 1)
    heads = D.dev_bf16(c.kvb)[:, :4096].view(8192, 16, 256)
    key = torch.full((8192, 16, 192), 0x5A, dtype=torch.uint8, device="cuda")
    vo = torch.zeros((8192, 16, 128), dtype=torch.uint8, device="cuda")
    ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:], ws[:, 512:], key, vo, 1,
                            kpe_dtype=1, out_scale=f32(0.01))
    gk, gv = c.gpu(1)
    np.testing.assert_array_equal(gk, D.host_u8(key))
    np.testing.assert_array_equal(gv, D.host_u8(vo))


def test_paged_pack_one_launch_of_131072_tokens(orc):
    """One 131072-token launch over a 2048-block cache: equal to the
    two-kernel GPU path everywhere and to the oracle on 2048 consecutive
    tokens; outputs written exactly once (guard bands intact)."""
    T = 131072
    pw = W.pack_workload(T, 8192, num_blocks=2048, seed=9, distinct_chunks=False)
    cache_t = dev_cache(pw)
    table_t = D.dev(pw.block_table)
    cu_t, st_t = D.dev(np.array([0, T], np.int32)), D.dev(np.array([0], np.int32))
    g = torch.Generator().manual_seed(12)
    kvb_t = torch.randn((T, 4160), generator=g).to(torch.bfloat16).cuda()
    heads = kvb_t[:, :4096].view(T, 16, 256)
    key = D.Guarded(T * 16 * 192)
    vo = D.Guarded(T * 16 * 128)
    sc = f32(0.01)
    ops.mla_context_kv_pack_paged(heads[:, :, :128], heads[:, :, 128:], cache_t, 1, 2048, 64,
                                  64 * ENTRY, ENTRY, table_t, cu_t, st_t, key.t.view(T, 16, 192),
                                  vo.t.view(T, 16, 128), 1, out_scale=sc)
    ws = torch.empty((T, ENTRY), dtype=torch.uint8, device="cuda")
    ops.mla_context_gather(cache_t, 1, 2048, 64, 64 * ENTRY, ENTRY, ENTRY, table_t, cu_t, st_t,
                           ws, 1)
    key2 = torch.empty((T, 16, 192), dtype=torch.uint8, device="cuda")
    vo2 = torch.empty((T, 16, 128), dtype=torch.uint8, device="cuda")
    ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:], ws[:, 512:], key2, vo2, 1,
                            kpe_dtype=1, out_scale=sc)
    torch.cuda.synchronize()
    assert key.guards_intact() and vo.guards_intact()
    assert torch.equal(key.t.view(T, 16, 192), key2) and torch.equal(vo.t.view(T, 16, 128), vo2)
    t0 = 70001
    kvb = D.host_u16(kvb_t[t0:t0 + 2048])
    rs = kvb.shape[1]
    rk, rv, err = orc.context_kv_pack_paged(
        kvb, rs, 256, kvb[:, 128:], rs, 256, pw.cache, 1, 2048, 64, 64 * ENTRY, ENTRY, 512,
        pw.block_table, np.array([0, 2048], np.int32), np.array([t0], np.int32), 2048, 16, 128,
        64, 128, 1, 0.01)
    assert err == 0
    np.testing.assert_array_equal(key.host().reshape(T, 16, 192)[t0:t0 + 2048], rk)
    np.testing.assert_array_equal(vo.host().reshape(T, 16, 128)[t0:t0 + 2048], rv)
