"""Pins for the oracle's standalone grouped RMSNorm + RoPE ("PR #50585 [K3
Perf] Optimize k3 dspark fused kv", Implementation item 3 and Source snippets:
_precompute_fused_context_kv on the [num_ctx, L, 576] projection output).

* It equals the bf16 grouped insert (itself pinned) with an identity slot
  mapping: cache row t of layer l is [normed kv_c | rotated k_pe].
* Read in place from the token-major [T, L, 576] projection output and
  written layer-major, every row is torch's float64 rms_norm with layer l's
  weight row and the complex-multiplication form of the neox rotation, each
  rounded once to bf16 by exact rational comparison.
* Without gamma and positions it is the plain layout change
  (permute(1, 0, 2).contiguous()) that numpy's transpose gives.
* Rows with a position outside the table are skipped in every layer.
"""
import numpy as np
import torch

import refmath as R
from pack_mla_cache_gb300 import workloads as W

ENTRY = 576


def _dspark_input(wl):
    """The [T, L, 576] projection output holding the workload's rows."""
    L, T = wl.num_layers, wl.num_tokens
    kv = np.empty((T, L, ENTRY), np.uint16)
    kv[:, :, :512] = wl.kv_c.transpose(1, 0, 2)
    kv[:, :, 512:] = wl.k_pe.transpose(1, 0, 2)
    return kv


def test_equals_bf16_insert_with_identity_slots(orc):
    wl = W.insert_workload(3, 40, 0, num_blocks=1, block_size=64, norm=True, rope=True, seed=31)
    table = orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)
    L, T = 3, 40
    ident = np.tile(np.arange(T, dtype=np.int64), (L, 1))
    caches = [np.zeros(64 * ENTRY, np.uint16) for _ in range(L)]
    assert orc.insert_grouped(wl.kv_c, wl.k_pe, ident, T, caches, None, 0, 1, 64, 64 * ENTRY,
                              ENTRY, wl.gamma, 1e-6, wl.positions, table) == 0
    oc, op, err = orc.norm_rope_grouped(wl.kv_c, 512, T * 512, wl.k_pe, 64, T * 64, T, L,
                                        gamma=wl.gamma, positions=wl.positions,
                                        cos_sin_cache=table)
    assert err == 0
    for l in range(L):
        rows = caches[l].reshape(64, ENTRY)[:T]
        np.testing.assert_array_equal(oc[l], rows[:, :512])
        np.testing.assert_array_equal(op[l], rows[:, 512:])


def test_dspark_layout_rows_are_rms_norm_and_rotation(orc):
    wl = W.insert_workload(5, 12, 0, num_blocks=1, block_size=64, norm=True, rope=True, seed=32)
    table = orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)
    L, T = 5, 12
    kv = _dspark_input(wl)
    flat = kv.reshape(-1)
    oc, op, err = orc.norm_rope_grouped(flat, L * ENTRY, ENTRY, flat[512:], L * ENTRY, ENTRY, T,
                                        L, gamma=wl.gamma, positions=wl.positions,
                                        cos_sin_cache=table)
    assert err == 0
    eps = float(np.float32(1e-6))
    for l in range(L):
        x = torch.from_numpy(R.bf16_to_f64(kv[:, l, :512]))
        g = torch.from_numpy(R.bf16_to_f64(wl.gamma[l]))
        ref = torch.nn.functional.rms_norm(x, (512,), g, eps).numpy()
        np.testing.assert_array_equal(oc[l], R.bf16_round_exact(ref).reshape(T, 512))
        pe = R.bf16_to_f64(kv[:, l, 512:])
        cs = table[wl.positions].astype(np.float64)
        z = (pe[:, :32] + 1j * pe[:, 32:]) * (cs[:, :32] + 1j * cs[:, 32:])
        np.testing.assert_array_equal(op[l, :, :32], R.bf16_round_exact(z.real).reshape(T, 32))
        np.testing.assert_array_equal(op[l, :, 32:], R.bf16_round_exact(z.imag).reshape(T, 32))


def test_without_norm_and_rope_is_the_layout_change(orc):
    wl = W.insert_workload(4, 33, 0, num_blocks=1, block_size=64, seed=33)
    kv = _dspark_input(wl)
    flat = kv.reshape(-1)
    oc, op, err = orc.norm_rope_grouped(flat, 4 * ENTRY, ENTRY, flat[512:], 4 * ENTRY, ENTRY, 33,
                                        4)
    assert err == 0
    np.testing.assert_array_equal(oc, np.ascontiguousarray(kv[:, :, :512].transpose(1, 0, 2)))
    np.testing.assert_array_equal(op, np.ascontiguousarray(kv[:, :, 512:].transpose(1, 0, 2)))


def test_out_of_table_positions_skip_the_row_in_every_layer(orc):
    wl = W.insert_workload(2, 6, 0, num_blocks=1, block_size=64, norm=True, rope=True, seed=34)
    table = orc.rope_cos_sin_cache(64, 64, W.ROPE_BASE)
    pos = np.array([0, 64, 5, -1, 63, 7], np.int64)
    oc0 = np.full((2, 6, 512), 0x1111, np.uint16)
    op0 = np.full((2, 6, 64), 0x2222, np.uint16)
    oc, op, err = orc.norm_rope_grouped(wl.kv_c, 512, 6 * 512, wl.k_pe, 64, 6 * 64, 6, 2,
                                        gamma=wl.gamma, positions=pos, cos_sin_cache=table,
                                        out_c=oc0, oc_ts=512, oc_ls=6 * 512, out_p=op0, op_ts=64,
                                        op_ls=6 * 64)
    assert err == orc.ERR_POS_OOB
    for t in range(6):
        skipped = t in (1, 3)
        assert (oc[:, t] == 0x1111).all() == skipped
        assert (op[:, t] == 0x2222).all() == skipped
