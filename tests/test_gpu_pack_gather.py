"""GPU parity of the pack launch that also gathers the next chunk
(mla_context_kv_pack_gather) against the CPU oracle, through the C ABI.

The fused call must equal the pack of chunk c followed by the gather of chunk
c + 1 ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing",
Implementation items 1-2: gather, then the fused pack, chunk by chunk; here
the two calls share a launch).  Both halves are bit-exact against the oracle's
context_gather and context_kv_pack: the chunk loop over 32768 context tokens
in 4 chunks of 8192 with two workspaces (fp8 output from a raw fp8 gather, bf16
output from a gather widened to bf16), runtime head counts and ragged token
counts, several sequences with bad block ids in the gathered half, empty
halves, and the overlap check.
"""
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


def oracle_gather(orc, pw, table, cu, starts, T, out_dtype):
    wide = out_dtype in (orc.BF16, orc.F16)
    out = np.full((T, ENTRY), 0x3F3F if wide else 0x3F, np.uint16 if wide else np.uint8)
    err = orc.context_gather(pw.cache, pw.cache_dtype, pw.num_blocks, pw.block_size,
                             pw.block_size * ENTRY, ENTRY, ENTRY, table, cu, starts, out, out_dtype)
    return out, err


def oracle_pack(orc, kvb, ws, H, out_dtype, kpe_dtype, scale):
    T, rs = kvb.shape
    return orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, ws[:, 512:], ENTRY,
                               kpe_dtype, T, H, 128, 64, 128, out_dtype,
                               scale if out_dtype != 0 else 1.0, True)


def host(t, out_dtype):
    return D.host_u16(t) if out_dtype == 0 else D.host_u8(t)


@pytest.mark.parametrize("out_dtype", [1, 0], ids=["fp8_out", "bf16_out"])
def test_chunk_loop_of_four_8192_token_chunks(orc, out_dtype):
    """gather(0); then pack(c) + gather(c + 1) in one call, c = 0..3 (the last
    call gathers nothing); workspaces alternate.  fp8 output packs from a raw
    fp8 gather, bf16 output from a gather widened to bf16."""
    C, NC, H = 8192, 4, 16
    pw = W.pack_workload(C * NC, C, num_blocks=1024, seed=21)
    ws_dt = 1 if out_dtype else 0
    cache_t = D.dev(pw.cache)
    table_t = D.dev(pw.block_table)
    cu = D.dev(np.array([0, C], np.int32))
    starts = [D.dev(np.array([c * C], np.int32)) for c in range(NC)]
    wsd = torch.uint8 if ws_dt else torch.bfloat16
    ws = [torch.zeros((C, ENTRY), dtype=wsd, device="cuda") for _ in range(2)]
    odt = torch.uint8 if out_dtype else torch.bfloat16
    keys = [torch.zeros((C, H, 192), dtype=odt, device="cuda") for _ in range(NC)]
    vs = [torch.zeros((C, H, 128), dtype=odt, device="cuda") for _ in range(NC)]
    kvbs = [D.dev_bf16(b) for b in pw.kv_b_proj]
    sc = torch.tensor([0.01], dtype=torch.float32, device="cuda") if out_dtype else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    empty_cu = D.dev(np.array([0, 0], np.int32))
    gathered = []
    ops.mla_context_gather(cache_t, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY, table_t, cu,
                           starts[0], ws[0], ws_dt)
    for c in range(NC):
        h = kvbs[c][:, :H * 256].view(C, H, 256)
        pack = ops.kv_pack_desc(h[:, :, :128], h[:, :, 128:], ws[c % 2][:, 512:], keys[c], vs[c],
                                out_dtype, kpe_dtype=ws_dt, out_scale=sc)
        nxt = c + 1 < NC
        gdesc = ops.context_gather_desc(cache_t, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY,
                                        table_t, cu if nxt else empty_cu,
                                        starts[c + 1] if nxt else starts[c], ws[(c + 1) % 2],
                                        ws_dt, num_tokens=C if nxt else 0)
        ops.mla_context_kv_pack_gather(pack, gdesc, err_word=err)
        if nxt:  # keep a copy of the gathered workspace before it is overwritten
            gathered.append(ws[(c + 1) % 2].clone())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for c in range(NC):
        rws, rerr = oracle_gather(orc, pw, pw.block_table, np.array([0, C], np.int32),
                                  np.array([c * C], np.int32), C, ws_dt)
        assert rerr == 0
        if c > 0:
            np.testing.assert_array_equal(host(gathered[c - 1], ws_dt), rws)
        rk, rv = oracle_pack(orc, pw.kv_b_proj[c], rws, H, out_dtype, ws_dt, 0.01)
        np.testing.assert_array_equal(host(keys[c], out_dtype), rk)
        np.testing.assert_array_equal(host(vs[c], out_dtype), rv)


@pytest.mark.parametrize("H", [3, 16])
@pytest.mark.parametrize("T", [1, 77, 1000])
def test_ragged_pack_with_many_sequence_gather(orc, H, T):
    """A pack of T tokens and H heads from one workspace, with a gather of 37
    sequences (bad block ids reached, 5 trailing unowned rows) into the other."""
    pw = W.pack_workload(max(T, 64), max(T, 64), num_blocks=128, num_heads=H, seed=22)
    rng = np.random.default_rng(1)
    S = 37
    table = rng.integers(0, 128, size=(S, 8)).astype(np.int32)
    table[5, 1] = 128
    table[9, 0] = -3
    lens = rng.integers(0, 60, size=S)
    starts = rng.integers(0, 300, size=S).astype(np.int32)
    lens[5], starts[5] = 150, 10
    lens[9], starts[9] = 20, 0
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Tg = int(cu[-1]) + 5
    ws_in = np.random.default_rng(2).integers(0, 126, size=(T, ENTRY)).astype(np.uint8)
    kvb = pw.kv_b_proj[0][:T]
    kvb_t = D.dev_bf16(kvb)
    h = kvb_t[:, :H * 256].view(T, H, 256)
    key = torch.zeros((T, H, 192), dtype=torch.uint8, device="cuda")
    vo = torch.zeros((T, H, 128), dtype=torch.uint8, device="cuda")
    out = torch.full((Tg, ENTRY), 0x3F, dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_t = D.dev(ws_in)
    pack = ops.kv_pack_desc(h[:, :, :128], h[:, :, 128:], ws_t[:, 512:], key, vo, 1, kpe_dtype=1,
                            out_scale=sc)
    g = ops.context_gather_desc(D.dev(pw.cache), 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY,
                                D.dev(table), D.dev(cu), D.dev(starts), out, 1)
    ops.mla_context_kv_pack_gather(pack, g, err_word=err)
    torch.cuda.synchronize()
    rg, rerr = oracle_gather(orc, pw, table, cu, starts, Tg, 1)
    assert rerr == ops.MLA_ERRBIT_BLOCK_OOB
    assert int(err.item()) == rerr
    np.testing.assert_array_equal(D.host_u8(out), rg)
    rk, rv = oracle_pack(orc, kvb, ws_in, H, 1, 1, 0.01)
    np.testing.assert_array_equal(D.host_u8(key), rk)
    np.testing.assert_array_equal(D.host_u8(vo), rv)


def test_empty_halves_and_overlap_check(orc):
    """Either half may be empty; a gather writing into the pack's own k_pe
    workspace is rejected before any launch."""
    T, H = 256, 16
    pw = W.pack_workload(T, T, num_blocks=8, seed=23)
    ws_in = np.random.default_rng(3).integers(0, 126, size=(T, ENTRY)).astype(np.uint8)
    ws_t = D.dev(ws_in)
    kvb = pw.kv_b_proj[0]
    h = D.dev_bf16(kvb)[:, :H * 256].view(T, H, 256)
    key = torch.zeros((T, H, 192), dtype=torch.uint8, device="cuda")
    vo = torch.zeros((T, H, 128), dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    out = torch.full((T, ENTRY), 0x3F, dtype=torch.uint8, device="cuda")
    cache_t, table_t = D.dev(pw.cache), D.dev(pw.block_table)
    cu, st = D.dev(np.array([0, T], np.int32)), D.dev(np.array([0], np.int32))
    # overlap: the gather would write the workspace the pack reads k_pe from
    pack = ops.kv_pack_desc(h[:, :, :128], h[:, :, 128:], ws_t[:, 512:], key, vo, 1, kpe_dtype=1,
                            out_scale=sc)
    bad = ops.context_gather_desc(cache_t, 1, 8, 64, 64 * ENTRY, ENTRY, ENTRY, table_t, cu, st,
                                  ws_t, 1)
    with pytest.raises(ops.MlaError, match="overlaps"):
        ops.mla_context_kv_pack_gather(pack, bad)
    assert bool((key == 0).all().item())
    # gather only (pack of 0 tokens)
    empty_pack = ops.kv_pack_desc(h[:0, :, :128], h[:0, :, 128:], ws_t[:0, 512:], key[:0], vo[:0],
                                  1, kpe_dtype=1, out_scale=sc)
    g = ops.context_gather_desc(cache_t, 1, 8, 64, 64 * ENTRY, ENTRY, ENTRY, table_t, cu, st, out,
                                1)
    ops.mla_context_kv_pack_gather(empty_pack, g)
    torch.cuda.synchronize()
    rg, _ = oracle_gather(orc, pw, pw.block_table, np.array([0, T], np.int32),
                          np.array([0], np.int32), T, 1)
    np.testing.assert_array_equal(D.host_u8(out), rg)
    # pack only (gather of 0 rows)
    g0 = ops.context_gather_desc(cache_t, 1, 8, 64, 64 * ENTRY, ENTRY, ENTRY, table_t, cu, st,
                                 out, 1, num_tokens=0)
    ops.mla_context_kv_pack_gather(pack, g0)
    torch.cuda.synchronize()
    rk, rv = oracle_pack(orc, kvb, ws_in, H, 1, 1, 0.01)
    np.testing.assert_array_equal(D.host_u8(key), rk)
    np.testing.assert_array_equal(D.host_u8(vo), rv)


@pytest.mark.parametrize("cfmt", [1, 2], ids=["e4m3", "e5m2"])
def test_fp16_chunk_launch_with_widening_gather(orc, cfmt):
    """fp16 kv_b_proj output: the chunk launch packs chunk 0 into an fp16 key
    and V from a workspace widened to fp16, and gathers chunk 1 from an fp8
    cache (e4m3 or e5m2) widened to fp16 into the other workspace."""
    C, H = 2048, 16
    pw = W.pack_workload(2 * C, C, num_blocks=128, cache_dtype=cfmt, seed=24 + cfmt)
    g = torch.Generator().manual_seed(cfmt)
    kvb = torch.randn((C, 4160), generator=g).to(torch.float16)
    kvb_np = kvb.view(torch.int16).numpy().view(np.uint16)
    cache_t, table_t = D.dev(pw.cache), D.dev(pw.block_table)
    cu = D.dev(np.array([0, C], np.int32))
    st0, st1 = D.dev(np.array([0], np.int32)), D.dev(np.array([C], np.int32))
    ws = [torch.zeros((C, ENTRY), dtype=torch.float16, device="cuda") for _ in range(2)]
    ops.mla_context_gather(cache_t, cfmt, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY, table_t, cu,
                           st0, ws[0], ops.MLA_FP16)
    h = kvb.cuda()[:, :H * 256].view(C, H, 256)
    key = torch.zeros((C, H, 192), dtype=torch.float16, device="cuda")
    vo = torch.zeros((C, H, 128), dtype=torch.float16, device="cuda")
    pack = ops.kv_pack_desc(h[:, :, :128], h[:, :, 128:], ws[0][:, 512:], key, vo, ops.MLA_FP16,
                            kpe_dtype=ops.MLA_FP16)
    gd = ops.context_gather_desc(cache_t, cfmt, pw.num_blocks, 64, 64 * ENTRY, ENTRY, ENTRY,
                                 table_t, cu, st1, ws[1], ops.MLA_FP16)
    ops.mla_context_kv_pack_gather(pack, gd)
    torch.cuda.synchronize()
    for c in range(2):
        r, err = oracle_gather(orc, pw, pw.block_table, np.array([0, C], np.int32),
                               np.array([c * C], np.int32), C, orc.F16)
        assert err == 0
        np.testing.assert_array_equal(D.host_u16(ws[c]), r)
    r0, _ = oracle_gather(orc, pw, pw.block_table, np.array([0, C], np.int32),
                          np.array([0], np.int32), C, orc.F16)
    rk, rv = orc.context_kv_pack(kvb_np, 4160, 256, kvb_np[:, 128:], 4160, 256, r0[:, 512:], ENTRY,
                                 orc.F16, C, H, 128, 64, 128, orc.F16, 1.0, True,
                                 in_dtype=orc.F16)
    np.testing.assert_array_equal(D.host_u16(key), rk)
    np.testing.assert_array_equal(D.host_u16(vo), rv)
