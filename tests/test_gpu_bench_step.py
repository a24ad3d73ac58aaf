"""The benchmark's own step, in the launch configuration bench.py times, against
the oracle.

bench.Workload builds the step's device buffers from the seeded generators: a
5-layer fp8 e4m3 insert of 65536 tokens with RMSNorm + RoPE into caches of
2048 blocks x 64 ("PR #55356 [Kimi Perf] Group fp8 mla cache insertion"), and
131072 context tokens packed in 16 chunks of 8192, 16 heads, fp8 key and V,
gathered from an fp8 paged cache ("PR #51772 [Attention][MLA] Fuse Kimi-K3
chunked-context K/V packing", Implementation items 1-2), with the gather's
early-table switch on.  step_pipelined() runs one step: the insert, the gather
of chunk 0 and 16 chunk launches (pack of chunk c + gather of chunk c + 1 into
the other workspace).  The oracle recomputes samples one by one: 2048 tokens
of the insert in all 5 layers (within the insert's fp8 tolerance: at most one
fp8 code apart, from the order of the RMSNorm sum), and 512 tokens of every
chunk's key and V (bit-exact); cache rows that no slot names stay zero and
both error words stay 0.
"""
import numpy as np
import pytest
import torch

import bench
import devutil as D
from pack_mla_cache_gb300 import ops
from pack_mla_cache_gb300 import workloads as W
from test_gpu_insert import assert_within_tolerance, oracle_insert

pytestmark = pytest.mark.gpu
ENTRY = bench.ENTRY


@pytest.fixture(scope="module")
def stepped():
    from pack_mla_cache_gb300 import build
    build.build()
    ops.lib()
    prev = ops.mla_set_gather_early_tables(False)
    w = bench.Workload(seed=1000)
    w.pipelined_setup()
    w.step_pipelined()
    torch.cuda.synchronize()
    yield w
    ops.mla_set_gather_early_tables(prev)


def test_error_words_are_clear(stepped):
    assert stepped.err.cpu().tolist() == [0, 0]


def test_insert_sampled_against_oracle(orc, stepped):
    w = stepped
    wl = w.wl
    L, T = bench.L_LAYERS, bench.T_INSERT
    sample = np.sort(np.random.default_rng(5).choice(T, 2048, replace=False))
    sub = W.InsertWorkload(L, 2048, 1, bench.NB_INSERT, bench.BS,
                           np.ascontiguousarray(wl.kv_c[:, sample]),
                           np.ascontiguousarray(wl.k_pe[:, sample]),
                           np.ascontiguousarray(wl.slot_mapping[:, sample]), True, wl.k_scales,
                           wl.gamma, np.ascontiguousarray(wl.positions[sample]), eps=wl.eps)
    ref, err = oracle_insert(orc, sub, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE))
    assert err == 0
    slots = wl.slot_mapping[0]
    for l in range(L):
        g = D.host_u8(w.caches[l]).reshape(-1, ENTRY)
        r = ref[l].reshape(-1, ENTRY)
        s = slots[sample]
        assert_within_tolerance([g[s].ravel()], [r[s].ravel()], 1)
        written = np.zeros(g.shape[0], bool)
        written[slots] = True
        assert (g[~written] == 0).all()


def test_every_chunk_sampled_against_oracle(orc, stepped):
    w = stepped
    pw = w.pw
    C, H = bench.CHUNK, bench.HEADS
    rng = np.random.default_rng(6)
    keys = D.host_u8(w.key_all).reshape(pw.num_chunks, C, H, 192)
    vs = D.host_u8(w.vout_all).reshape(pw.num_chunks, C, H, 128)
    cu = np.array([0, C], np.int32)
    for c in range(pw.num_chunks):
        ws = np.full((C, ENTRY), 0x3F, np.uint8)
        gerr = orc.context_gather(pw.cache, pw.cache_dtype, pw.num_blocks, pw.block_size,
                                  pw.block_size * ENTRY, ENTRY, ENTRY, pw.block_table, cu,
                                  np.array([c * C], np.int32), ws, 1)
        assert gerr == 0
        rows = np.sort(rng.choice(C, 512, replace=False))
        kvb = np.ascontiguousarray(pw.kv_b_proj[c][rows])
        rs = kvb.shape[1]
        wsr = np.ascontiguousarray(ws[rows])
        rk, rv = orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, wsr[:, 512:], ENTRY, 1,
                                     512, H, 128, 64, 128, 1, bench.OUT_SCALE, True)
        np.testing.assert_array_equal(keys[c][rows], rk, err_msg=f"key, chunk {c}")
        np.testing.assert_array_equal(vs[c][rows], rv, err_msg=f"V, chunk {c}")
