"""GPU parity of the standalone grouped RMSNorm + RoPE against the CPU oracle,
through the C ABI ("PR #50585 [K3 Perf] Optimize k3 dspark fused kv",
_precompute_fused_context_kv).

The tolerance is the insert's for RMSNorm + RoPE: within 1 bf16 ulp of the
oracle (which rounds the exact result once), on a small fraction of the
elements.  The kernel shares the insert's arithmetic, so its rows are also
bit-identical to those a bf16 grouped insert writes; without a norm or a
rotation the result is the exact layout change.  Cases: the [T, L, 576]
projection read in place and written layer-major (T 4096 and a ragged 4099,
L 5 and 3), norm only, rotation only, out-of-table positions, 0 and 1 tokens,
and the 65536-token x 5-layer size (sampled).  Every output sits between guard
bands.
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


@pytest.fixture(scope="module")
def tables(orc):
    return D.gpu_rope_table(), orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)


def dspark_input(wl):
    """The [T, L, 576] projection output holding the workload's rows."""
    kv = np.empty((wl.num_tokens, wl.num_layers, ENTRY), np.uint16)
    kv[:, :, :512] = wl.kv_c.transpose(1, 0, 2)
    kv[:, :, 512:] = wl.k_pe.transpose(1, 0, 2)
    return kv


def gpu_norm_rope(wl, kv, cos_sin, *, norm=True, rope=True, positions=None, err=None):
    """Run on the [T, L, 576] input; returns layer-major (kv_c [L,T,512],
    k_pe [L,T,64]) as uint16 and whether the guard bands held."""
    T, L = wl.num_tokens, wl.num_layers
    kv_t = D.dev_bf16(kv)
    oc = D.Guarded(L * T * 512 * 2)
    op = D.Guarded(L * T * 64 * 2)
    oc.t.fill_(0x11)  # payloads only: the guard bands keep their canary
    op.t.fill_(0x22)
    oc_v = oc.t.view(torch.bfloat16).view(L, T, 512)
    op_v = op.t.view(torch.bfloat16).view(L, T, 64)
    pos = positions if positions is not None else wl.positions
    ops.mla_norm_rope_grouped(
        kv_t[:, :, :512], kv_t[:, :, 512:], oc_v.transpose(0, 1), op_v.transpose(0, 1),
        gamma=D.dev_bf16(wl.gamma) if norm else None, eps=wl.eps,
        positions=D.dev(pos) if rope else None, cos_sin_cache=cos_sin if rope else None,
        err_word=err)
    torch.cuda.synchronize()
    return (D.host_u16(oc_v), D.host_u16(op_v), oc.guards_intact() and op.guards_intact())


def oracle_norm_rope(orc, wl, kv, table, *, norm=True, rope=True, positions=None):
    T, L = wl.num_tokens, wl.num_layers
    flat = kv.reshape(-1)
    oc = np.full((L, T, 512), 0x1111, np.uint16)
    op = np.full((L, T, 64), 0x2222, np.uint16)
    pos = positions if positions is not None else wl.positions
    return orc.norm_rope_grouped(flat, L * ENTRY, ENTRY, flat[512:], L * ENTRY, ENTRY, T, L,
                                 gamma=wl.gamma if norm else None, eps=wl.eps,
                                 positions=pos if rope else None,
                                 cos_sin_cache=table if rope else None, out_c=oc, oc_ts=512,
                                 oc_ls=T * 512, out_p=op, op_ts=64, op_ls=T * 64)


def within_one_ulp(g, r, frac):
    d = R.ulp_diff_bf16(g.ravel(), r.ravel())
    assert d.max() <= 1, d.max()
    assert (d != 0).mean() <= frac, (d != 0).mean()


@pytest.mark.parametrize("L,T", [(5, 4096), (3, 4099)])
def test_dspark_layout_within_one_ulp(orc, tables, L, T):
    wl = W.insert_workload(L, T, 0, num_blocks=(T + 63) // 64, norm=True, rope=True, seed=50 + L)
    kv = dspark_input(wl)
    gc, gp, guards = gpu_norm_rope(wl, kv, tables[0])
    rc, rp, err = oracle_norm_rope(orc, wl, kv, tables[1])
    assert guards and err == 0
    within_one_ulp(gc, rc, 2e-3)
    within_one_ulp(gp, rp, 2e-3)


@pytest.mark.parametrize("T", [1024, 2048, 28000])
def test_rows_equal_the_bf16_insert(tables, T):
    """The same rows through a bf16 grouped insert (identity slots) and
    through the standalone kernel are bit-identical, in every pairing of
    layouts: 1024 tokens x 5 layers (one row per warp in both), 2048 (four
    rows per warp in the insert, two here), 28000 (the insert's bulk-copy
    ring, two rows per warp, against one row per warp here)."""
    L = 5
    wl = W.insert_workload(L, T, 0, num_blocks=(T + 63) // 64, norm=True, rope=True, seed=60)
    wl.slot_mapping = np.ascontiguousarray(np.tile(np.arange(T, dtype=np.int64), (L, 1)))
    wl.shared_slots = False
    caches, guards, _ = D.gpu_insert(wl, cos_sin=tables[0], slot_shared_1d=False)
    gc, gp, g2 = gpu_norm_rope(wl, dspark_input(wl), tables[0])
    assert guards and g2
    for l in range(L):
        rows = caches[l].reshape(-1, ENTRY)[:T]
        np.testing.assert_array_equal(gc[l], rows[:, :512])
        np.testing.assert_array_equal(gp[l], rows[:, 512:])


def test_without_norm_and_rope_is_the_exact_layout_change(tables):
    wl = W.insert_workload(5, 1000, 0, num_blocks=16, seed=61)
    kv = dspark_input(wl)
    gc, gp, guards = gpu_norm_rope(wl, kv, tables[0], norm=False, rope=False)
    assert guards
    np.testing.assert_array_equal(gc, kv[:, :, :512].transpose(1, 0, 2))
    np.testing.assert_array_equal(gp, kv[:, :, 512:].transpose(1, 0, 2))


@pytest.mark.parametrize("norm,rope", [(True, False), (False, True)])
def test_norm_only_and_rotation_only(orc, tables, norm, rope):
    wl = W.insert_workload(5, 777, 0, num_blocks=16, norm=True, rope=True, seed=62)
    kv = dspark_input(wl)
    gc, gp, guards = gpu_norm_rope(wl, kv, tables[0], norm=norm, rope=rope)
    rc, rp, _ = oracle_norm_rope(orc, wl, kv, tables[1], norm=norm, rope=rope)
    assert guards
    within_one_ulp(gc, rc, 2e-3)
    within_one_ulp(gp, rp, 2e-3)
    if not norm:
        np.testing.assert_array_equal(gc, rc)
    if not rope:
        np.testing.assert_array_equal(gp, rp)


def test_out_of_table_positions_skip_rows(orc, tables):
    wl = W.insert_workload(3, 300, 0, num_blocks=8, norm=True, rope=True, seed=63)
    pos = wl.positions.copy()
    pos[[0, 17, 299]] = [-1, W.MAX_POSITION, 1 << 40]
    kv = dspark_input(wl)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc, gp, guards = gpu_norm_rope(wl, kv, tables[0], positions=pos, err=err)
    rc, rp, oerr = oracle_norm_rope(orc, wl, kv, tables[1], positions=pos)
    assert guards and int(err.item()) == oerr == ops.MLA_ERRBIT_POS_OOB
    for t in (0, 17, 299):
        assert (gc[:, t] == 0x1111).all() and (gp[:, t] == 0x2222).all()
    within_one_ulp(gc, rc, 2e-3)
    within_one_ulp(gp, rp, 2e-3)


@pytest.mark.parametrize("T", [0, 1])
def test_tiny_token_counts(orc, tables, T):
    wl = W.insert_workload(5, T, 0, num_blocks=1, norm=True, rope=True, seed=64)
    kv = dspark_input(wl)
    gc, gp, guards = gpu_norm_rope(wl, kv, tables[0])
    rc, rp, _ = oracle_norm_rope(orc, wl, kv, tables[1])
    assert guards and gc.size == rc.size == 5 * T * 512
    if T:
        within_one_ulp(gc, rc, 1.0)
        within_one_ulp(gp, rp, 1.0)


def test_65536_tokens_by_5_layers_sampled(orc, tables):
    L, T = 5, 65536
    wl = W.insert_workload(L, T, 0, num_blocks=T // 64, norm=True, rope=True, seed=65)
    kv = dspark_input(wl)
    gc, gp, guards = gpu_norm_rope(wl, kv, tables[0])
    assert guards
    rows = np.sort(np.random.default_rng(3).choice(T, 2048, replace=False))
    sub = W.InsertWorkload(L, 2048, 0, 32, 64, np.ascontiguousarray(wl.kv_c[:, rows]),
                           np.ascontiguousarray(wl.k_pe[:, rows]), wl.slot_mapping[:, :2048],
                           True, None, wl.gamma, np.ascontiguousarray(wl.positions[rows]))
    rc, rp, err = oracle_norm_rope(orc, sub, np.ascontiguousarray(kv[rows]), tables[1])
    assert err == 0
    within_one_ulp(gc[:, rows], rc, 2e-3)
    within_one_ulp(gp[:, rows], rp, 2e-3)
