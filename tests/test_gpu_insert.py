"""GPU parity of the grouped insert against the CPU oracle, through the C ABI.

Bit-exact for the raw bf16 copy and the raw fp8 conversion ("PR #55356 [Kimi
Perf] Group fp8 mla cache insertion": grouped == per-layer, rtol=0 atol=0);
for RMSNorm + RoPE a stated tolerance: within 1 bf16 ulp before
quantisation (observed through a bf16 cache) and within 1 fp8 ulp on at most
1e-4 of the elements after.  Every case also checks the guard bands around
each cache and that rows no slot names are untouched.
"""
import dataclasses

import numpy as np
import pytest
import torch

import devutil as D
import refmath as R
from pack_mla_cache_gb300 import ops
from pack_mla_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FP8_MISMATCH_MAX = 1e-4  # fraction of elements allowed 1 fp8 ulp off (norm+rope)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pack_mla_cache_gb300 import build
    build.build()
    ops.lib()


def oracle_insert(orc, wl, table=None, fill=0):
    caches = wl.empty_caches(fill=fill)
    slots = np.ascontiguousarray(wl.slot_mapping[0]) if wl.shared_slots else wl.slot_mapping
    err = orc.insert_grouped(wl.kv_c, wl.k_pe, slots, wl.slot_layer_stride, caches,
                             wl.k_scales, wl.cache_dtype, wl.num_blocks, wl.block_size,
                             wl.block_stride, wl.entry_stride, wl.gamma, wl.eps, wl.positions,
                             table)
    return caches, err


def assert_exact(gpu, ref):
    for l, (g, r) in enumerate(zip(gpu, ref)):
        bad = np.nonzero(g != r)[0]
        assert bad.size == 0, (l, bad[:10], g[bad[:10]], r[bad[:10]])


def assert_within_tolerance(gpu, ref, cache_dtype):
    total, off = 0, 0
    for g, r in zip(gpu, ref):
        d = R.ulp_diff_bf16(g, r) if cache_dtype == 0 else R.ulp_diff_fp8(g, r)
        assert d.max() <= 1, d.max()
        total += g.size
        off += int((d != 0).sum())
    if cache_dtype != 0:
        assert off <= FP8_MISMATCH_MAX * total, (off, total)
    return off, total


# ---------------------------------------------------------------- raw inserts
def test_single_layer_bf16_exact_copy(orc):
    """64 tokens into a bf16 cache of 16 blocks x 64, slots from a random
    permutation of 1024: the cache rows are the input bits."""
    wl = W.insert_workload(1, 64, 0, num_blocks=16, block_size=64, seed=1)
    gpu, guards, _ = D.gpu_insert(wl, fill=0x5A)
    ref, err = oracle_insert(orc, wl, fill=0x5A5A)
    assert guards and err == 0
    assert_exact(gpu, ref)


@pytest.mark.parametrize("dtype", [0, 1, 2])
@pytest.mark.parametrize("shared", [True, False])
def test_pages_grouped_test_shape(orc, dtype, shared):
    """5 layers, block_size 16, 8 blocks, 42 tokens, k_scale linspace(0.05,
    0.25), last slot -1, shared (aliased) or per-layer mappings."""
    wl = W.pages_test_insert_workload(dtype, shared)
    gpu, guards, _ = D.gpu_insert(wl, slot_shared_1d=False)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_small_decode_batch_fp8_e4m3(orc, T):
    wl = W.insert_workload(5, T, 1, num_blocks=64, block_size=64, seed=2 + T)
    gpu, guards, _ = D.gpu_insert(wl)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


@pytest.mark.parametrize("dtype", [1, 2])
@pytest.mark.parametrize("scale", [1.0, 0.005, 0.0123, 0.02, 0.25, 3.0])
def test_fp8_conversion_exhaustive_over_bf16(orc, dtype, scale):
    """kv_c holds all 2^16 bf16 patterns (incl. NaN, inf, subnormals): the
    cache must equal the oracle's RNE-saturating conversion bit for bit."""
    wl = W.insert_workload(1, 128, dtype, num_blocks=2, block_size=64, seed=9)
    wl.kv_c = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(1, 128, 512)
    wl.k_pe = np.ascontiguousarray(wl.kv_c[:, :, :64][:, ::-1])
    wl.k_scales = np.array([scale], np.float32)
    gpu, guards, _ = D.gpu_insert(wl)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


@pytest.mark.parametrize("dtype", [1, 2])
def test_fp8_conversion_exhaustive_through_every_shape(orc, bulk, dtype):
    """All 2^16 bf16 patterns tiled over 4096 tokens (the bulk-copy shape when
    forced, else the row-per-warp shape): bit-exact, including zeros of both
    signs, subnormals, values whose quotient overflows, infinities and NaNs."""
    wl = W.insert_workload(1, 4096, dtype, num_blocks=64, block_size=64, seed=16)
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    wl.kv_c = np.tile(pats, 32).reshape(1, 4096, 512)
    wl.k_pe = np.ascontiguousarray(np.tile(pats[::-1], 4).reshape(1, 4096, 64))
    wl.k_scales = np.array([0.0123], np.float32)
    gpu, guards, _ = D.gpu_insert(wl)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


def test_ragged_non_power_of_two_blocks_and_large_rows(orc):
    """11111 tokens x 3 layers with per-layer mappings (33333 rows: not a
    multiple of any tile, more rows than the capped grid has warps, so warps
    loop), block_size 48 (the division path instead of the shift)."""
    wl = W.insert_workload(3, 11111, 1, num_blocks=300, block_size=48, shared_slots=False,
                           seed=11)
    gpu, guards, _ = D.gpu_insert(wl)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


@pytest.mark.parametrize("T", [257, 1000])
def test_dspark_projection_layout_input(orc, T):
    """kv_c / k_pe read straight from a [T, L, 576] projection output (no
    permute().contiguous()), as strided views (the row-per-warp shape, the only
    one that takes these strides)."""
    wl = W.insert_workload(5, T, 1, num_blocks=16, block_size=64, seed=12, norm=True, rope=True)
    T, L = wl.num_tokens, wl.num_layers
    proj = np.concatenate([wl.kv_c, wl.k_pe], axis=2).transpose(1, 0, 2).copy()  # [T, L, 576]
    pt = D.dev_bf16(proj)
    kv_c = pt[:, :, :512].permute(1, 0, 2)
    k_pe = pt[:, :, 512:].permute(1, 0, 2)
    gpu, guards, _ = D.gpu_insert(wl, kv_c=kv_c, k_pe=k_pe, cos_sin=D.gpu_rope_table())
    ref, _ = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE))
    assert guards
    assert_within_tolerance(gpu, ref, 1)


@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_ragged_tail_and_padding(orc, bulk, dtype):
    """4099 tokens x 3 layers with a shared mapping (a partial last run of
    tokens in the bulk-copy shape) and some -1 padding slots."""
    wl = W.insert_workload(3, 4099, dtype, num_blocks=80, block_size=64, norm=True, rope=True,
                           seed=14)
    wl.slot_mapping[:, ::97] = -1
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.gpu_rope_table(), fill=0x3C)
    ref, _ = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE),
                           fill=0x3C3C if dtype == 0 else 0x3C)
    assert guards
    assert_within_tolerance(gpu, ref, dtype)


def test_raw_fp8_insert_large_exact(orc, bulk):
    """No norm / RoPE, 8192 tokens x 5 layers: the raw fp8 conversion through
    every launch shape is bit-exact."""
    wl = W.insert_workload(5, 8192, 1, num_blocks=256, block_size=64, seed=15)
    gpu, guards, _ = D.gpu_insert(wl)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


def test_maximum_layer_count(orc, bulk):
    """128 layers (the most one call takes) x 64 tokens with a mapping per
    layer: 8192 rows, so the bulk-copy shape runs over items of every layer
    index; bit-exact raw fp8 with a different k_scale per layer."""
    wl = W.insert_workload(128, 64, 1, num_blocks=2, block_size=64, shared_slots=False, seed=17)
    gpu, guards, _ = D.gpu_insert(wl)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


def test_odd_layer_count_with_norm_rope_and_per_layer_slots(orc, bulk):
    """37 layers x 300 tokens (item index -> (run, layer) with a layer count
    that divides nothing), RMSNorm + RoPE into a bf16 cache, a mapping per
    layer: within 1 bf16 ulp."""
    wl = W.insert_workload(37, 300, 0, num_blocks=5, block_size=64, shared_slots=False,
                           norm=True, rope=True, seed=18)
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.gpu_rope_table())
    ref, _ = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE))
    assert guards
    assert_within_tolerance(gpu, ref, 0)


def test_out_of_range_data_is_skipped_and_reported(orc):
    wl = W.insert_workload(2, 8, 1, num_blocks=4, block_size=16, norm=True, rope=True, seed=5)
    wl.slot_mapping = np.array([[0, 1, -1, 64, 2, 3, 4, 5]] * 2, np.int64)
    wl.positions = np.array([0, 1, 2, 3, 64, 5, -1, 7], np.int64)
    table_g = D.gpu_rope_table(64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=table_g, fill=0x11, err=err)
    ref, oerr = oracle_insert(orc, wl, orc.rope_cos_sin_cache(64, 64, W.ROPE_BASE), fill=0x11)
    assert guards
    assert int(err.item()) == oerr == (ops.MLA_ERRBIT_SLOT_OOB | ops.MLA_ERRBIT_POS_OOB)
    for g, r in zip(gpu, ref):
        written = (r.reshape(-1, 576) != 0x11).any(1)
        np.testing.assert_array_equal((g.reshape(-1, 576) != 0x11).any(1), written)
        assert_within_tolerance([g], [r], 1)


def test_misaligned_cache_pointer_is_skipped_and_reported():
    wl = W.insert_workload(2, 4, 1, num_blocks=1, block_size=16, seed=6)
    good = D.Guarded(16 * 576 + 64)
    good.t.fill_(0x22)
    bad_ptr = good.ptr() + 8
    ptrs = torch.tensor([good.ptr(), bad_ptr], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.mla_cache_insert_grouped(D.dev_bf16(wl.kv_c), D.dev_bf16(wl.k_pe),
                                 D.dev(np.ascontiguousarray(wl.slot_mapping[0])), ptrs,
                                 D.dev(wl.k_scales), 1, 1, 16, 16 * 576, 576, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ops.MLA_ERRBIT_MISALIGNED
    assert good.guards_intact()


def test_zero_tokens_launches_nothing():
    wl = W.insert_workload(5, 0, 1, num_blocks=1, block_size=64, seed=0)
    gpu, guards, _ = D.gpu_insert(wl, fill=0x33)
    assert guards and all((g == 0x33).all() for g in gpu)


def test_host_pointer_for_scales_is_rejected():
    wl = W.insert_workload(5, 4, 1, num_blocks=1, block_size=64, seed=0)
    c = D.Guarded(64 * 576)
    ptrs = torch.tensor([c.ptr()] * 5, dtype=torch.int64, device="cuda")
    host_scales = torch.ones(5, dtype=torch.float32)
    with pytest.raises(ops.MlaError, match="same CUDA device"):
        ops.mla_cache_insert_grouped(D.dev_bf16(wl.kv_c), D.dev_bf16(wl.k_pe),
                                     D.dev(np.ascontiguousarray(wl.slot_mapping[0])), ptrs,
                                     host_scales, 1, 1, 64, 64 * 576, 576)


def test_host_pointer_for_kv_c_is_rejected():
    wl = W.insert_workload(5, 4, 1, num_blocks=1, block_size=64, seed=0)
    c = D.Guarded(64 * 576)
    ptrs = torch.tensor([c.ptr()] * 5, dtype=torch.int64, device="cuda")
    host_kv_c = torch.zeros((5, 4, 512), dtype=torch.bfloat16)
    with pytest.raises(ops.MlaError, match="kv_c must be device memory"):
        ops.mla_cache_insert_grouped(host_kv_c, D.dev_bf16(wl.k_pe),
                                     D.dev(np.ascontiguousarray(wl.slot_mapping[0])), ptrs,
                                     D.dev(wl.k_scales), 1, 1, 64, 64 * 576, 576)
    assert c.guards_intact() and bool((c.t == D.CANARY).all().item())


def test_pointer_checks_off_runs_the_same_insert(orc):
    """With the per-call device-pointer checks switched off (device pointers
    only), the insert writes exactly what it writes with them on."""
    wl = W.insert_workload(5, 8, 1, num_blocks=4, block_size=64, seed=3)
    prev = ops.mla_set_pointer_checks(False)
    try:
        gpu, guards, _ = D.gpu_insert(wl)
    finally:
        ops.mla_set_pointer_checks(prev)
    ref, _ = oracle_insert(orc, wl)
    assert guards
    assert_exact(gpu, ref)


def test_null_layer_cache_pointer_skips_that_layer(orc, bulk):
    """A null entry in kv_cache_ptrs: that layer's rows are skipped with
    MLA_ERRBIT_MISALIGNED (no write near address 0); the other layers are
    exact.  8192 tokens x 5 layers so the bulk-copy shape runs when forced."""
    wl = W.insert_workload(5, 8192, 1, num_blocks=256, block_size=64, seed=4)
    nbytes = wl.num_blocks * wl.block_size * W.ENTRY
    caches = [D.Guarded(nbytes) for _ in range(5)]
    for c in caches:
        c.t.fill_(0x44)
    ptrs = torch.tensor([c.ptr() for c in caches], dtype=torch.int64, device="cuda")
    ptrs[2] = 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.mla_cache_insert_grouped(D.dev_bf16(wl.kv_c), D.dev_bf16(wl.k_pe),
                                 D.dev(np.ascontiguousarray(wl.slot_mapping[0])), ptrs,
                                 D.dev(wl.k_scales), 1, wl.num_blocks, 64, 64 * 576, 576,
                                 err_word=err)
    torch.cuda.synchronize()
    ref, oerr = oracle_insert(orc, wl, fill=0x44)
    assert oerr == 0
    assert int(err.item()) == ops.MLA_ERRBIT_MISALIGNED
    for l, c in enumerate(caches):
        assert c.guards_intact()
        h = c.host()
        if l == 2:
            assert (h == 0x44).all()
        else:
            np.testing.assert_array_equal(h, ref[l])


def test_bulk_ring_timeout_path_returns_and_reports(orc):
    """The bulk-copy ring's bounded waits: with a 1 ms limit and the producer
    of the first CTA issuing no copies for its local item 3 (a testing hook),
    the consumer waiting for that item runs out of time.  The call returns,
    MLA_ERRBIT_TIMEOUT is set, every row is either the oracle's or untouched
    (the skipped item's rows untouched), the guard bands hold, and the next
    call with the default limit is exact.  No fault is involved: only a wait
    that gives up."""
    wl = W.insert_workload(5, 512, 1, num_blocks=16, block_size=64, seed=5)
    ref, _ = oracle_insert(orc, wl, fill=0x3C)
    prev = ops.mla_set_bulk_copy(2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        ops.mla_test_insert_timeout(1_000_000, 3)
        gpu, guards, _ = D.gpu_insert(wl, fill=0x3C, err=err)
    finally:
        ops.mla_test_insert_timeout()
    try:
        assert guards
        assert int(err.item()) & ops.MLA_ERRBIT_TIMEOUT
        # item 3 of CTA 0 is global item G * 3 (G CTAs; items are (4-token run, layer))
        items = (512 // 4) * 5
        G = min(ops_grid_ctas(), -(-items // 23))
        j = G * 3
        run, layer = j // 5, j % 5
        slots = wl.slot_mapping[0]
        written = 0
        for l in range(5):
            g = gpu[l].reshape(-1, 576)
            r = ref[l].reshape(-1, 576)
            unnamed = np.ones(g.shape[0], bool)
            unnamed[slots] = False
            assert (g[unnamed] == 0x3C).all()
            for t in range(512):
                row = g[slots[t]]
                untouched = bool((row == 0x3C).all())
                if l == layer and run * 4 <= t < run * 4 + 4:
                    assert untouched, ("the skipped item's row was written", l, t)
                elif not untouched:  # rows after the timeout may be dropped
                    np.testing.assert_array_equal(row, r[slots[t]])
                    written += 1
        assert written > 0
        gpu2, guards2, _ = D.gpu_insert(wl, fill=0x3C)
        assert guards2
        assert_exact(gpu2, ref)
    finally:
        ops.mla_set_bulk_copy(prev)


def ops_grid_ctas():
    """CTAs of the bulk-copy ring that can be resident: one per SM."""
    return torch.cuda.get_device_properties(0).multi_processor_count


# ------------------------------------------------------------ norm + rope inserts
@pytest.mark.parametrize("dtype", [1, 2])
@pytest.mark.parametrize("shared", [True, False])
def test_norm_rope_4096_tokens(orc, bulk, dtype, shared):
    """RMSNorm (eps 1e-6, gamma ~ N(1, 0.1)) + neox RoPE (positions in
    [0, 32768)), 4096 tokens x 5 layers into 512-block caches; each side uses
    its own cos/sin table."""
    wl = W.insert_workload(5, 4096, dtype, num_blocks=512, block_size=64, shared_slots=shared,
                           norm=True, rope=True, seed=20 + dtype)
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.gpu_rope_table())
    ref, _ = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE))
    assert guards
    assert_within_tolerance(gpu, ref, dtype)


def test_norm_rope_bf16_cache_within_one_ulp(orc, bulk):
    """A bf16 cache exposes the pre-quantisation values: within 1 bf16 ulp."""
    wl = W.insert_workload(5, 4096, 0, num_blocks=512, block_size=64, norm=True, rope=True,
                           seed=30)
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.gpu_rope_table())
    ref, _ = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE))
    assert guards
    off, total = assert_within_tolerance(gpu, ref, 0)
    assert off <= 2e-3 * total, (off, total)


def test_rotation_arithmetic_on_a_shared_random_table(orc):
    """Both sides read the same seeded random cos/sin values: isolates the
    rotation arithmetic from the table construction."""
    wl = W.insert_workload(5, 2048, 0, num_blocks=256, block_size=64, norm=False, rope=True,
                           seed=31)
    g = torch.Generator().manual_seed(7)
    table = (torch.rand((W.MAX_POSITION, 64), generator=g) * 2 - 1).numpy().astype(np.float32)
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.dev(table))
    ref, _ = oracle_insert(orc, wl, table)
    assert guards
    off, total = assert_within_tolerance(gpu, ref, 0)
    assert off <= 1e-3 * total


def test_rope_table_matches_oracle(orc):
    """Both tables evaluate the angle in double precision, but the device's and
    the host library's pow() may differ in the last double bit, which moves an
    angle of up to ~3.3e4 rad by up to ~2e-11.  So each entry is within one fp32
    ulp of the oracle's, or within 2^-35 absolute (near the zeros of cos/sin)."""
    t = D.gpu_rope_table().cpu().numpy()
    r = orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)
    diff = np.abs(t.astype(np.float64) - r.astype(np.float64))
    bound = np.maximum(np.spacing(np.abs(r)).astype(np.float64), 2.0 ** -35)
    assert (diff <= bound).all(), diff[diff > bound][:10]
    assert (t != r).mean() < 1e-3


@pytest.mark.parametrize("dtype", [0, 1])
def test_every_layout_gives_the_same_bits(dtype):
    """RMSNorm + RoPE rows are computed one, two or four per warp in the row
    shape (by call size) or by the bulk-copy ring, with one summation tree for
    the sum of squares.  The same 2048 tokens x 5 layers as one call (10240
    rows: four rows per warp), as calls of 1600 + 448 tokens (8000 rows: two
    rows per warp; 2240: one), as two calls of 1024 tokens (one row per warp),
    and through the bulk-copy shape give the same caches bit for bit (a bf16
    cache shows the normalised values themselves)."""
    wl = W.insert_workload(5, 2048, dtype, num_blocks=256, block_size=64, norm=True, rope=True,
                           seed=41)
    table = D.gpu_rope_table()

    def part(t0, t1):
        return W.InsertWorkload(5, t1 - t0, dtype, 256, 64,
                                np.ascontiguousarray(wl.kv_c[:, t0:t1]),
                                np.ascontiguousarray(wl.k_pe[:, t0:t1]),
                                np.ascontiguousarray(wl.slot_mapping[:, t0:t1]),
                                True, wl.k_scales, wl.gamma,
                                np.ascontiguousarray(wl.positions[t0:t1]))

    one, g1, _ = D.gpu_insert(wl, cos_sin=table, fill=0x11)
    results, guards = [], [g1]
    for cuts in ((0, 1600, 2048), (0, 1024, 2048)):
        caches = None
        for t0, t1 in zip(cuts[:-1], cuts[1:]):
            out, g, caches = D.gpu_insert(part(t0, t1), cos_sin=table, fill=0x11, caches=caches)
            guards.append(g)
        results.append(out)
    prev = ops.mla_set_bulk_copy(2)
    try:
        ring, g3, _ = D.gpu_insert(wl, cos_sin=table, fill=0x11)
    finally:
        ops.mla_set_bulk_copy(prev)
    assert all(guards) and g3
    for out in results:
        assert_exact(out, one)
    assert_exact(ring, one)


@pytest.mark.parametrize("early", [False, True], ids=["stream_order", "early_tables"])
@pytest.mark.parametrize("dtype,norm,rope,shared", [(1, True, True, True), (2, True, True, False),
                                                    (0, True, True, True), (1, True, False, True),
                                                    (1, False, True, False)])
def test_four_rows_per_warp_against_oracle(orc, dtype, norm, rope, shared, early):
    """2400 tokens x 5 layers (12000 rows): more than one round of the
    two-rows-per-warp row shape, one round of four rows per warp, so the
    quarter-warp kernel runs; against the oracle with RMSNorm and / or RoPE,
    bf16 / e4m3 / e5m2 caches, shared and per-layer mappings, with an
    out-of-range slot, a padding slot and an out-of-table position mixed in."""
    wl = W.insert_workload(5, 2400, dtype, num_blocks=256, block_size=64, shared_slots=shared,
                           norm=norm, rope=rope, seed=50 + dtype)
    wl.slot_mapping = wl.slot_mapping.copy()
    wl.slot_mapping[:, 17] = -1
    wl.slot_mapping[:, 1000] = 256 * 64 + 5  # beyond the cache
    if rope:
        wl.positions = wl.positions.copy()
        wl.positions[2222] = W.MAX_POSITION
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = ops.mla_set_insert_early_tables(early)
    try:
        gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.gpu_rope_table() if rope else None, fill=0x19,
                                      err=err)
    finally:
        ops.mla_set_insert_early_tables(prev)
    ref, oerr = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE)
                              if rope else None, fill=0x1919 if dtype == 0 else 0x19)
    assert guards
    assert int(err.item()) == oerr
    assert oerr & ops.MLA_ERRBIT_SLOT_OOB
    assert_within_tolerance(gpu, ref, dtype)


@pytest.mark.parametrize("T", [1600, 2048], ids=["two_rows_per_warp", "four_rows_per_warp"])
@pytest.mark.parametrize("dtype", [1, 2])
def test_trimmed_row_shape_gives_the_same_bits(orc, dtype, T):
    """With early tables the row shape's two-rows-per-warp RMSNorm form works
    on negated rows and skips the special-value test for layers whose gamma
    bound allows it; it must give the bits of the plain form in every case:
    5 layers whose scales take the fast division without the test (two
    normal scales), the fast division with the test (a scale so small that
    normalised values can overflow the quotient), and the guarded division (a
    subnormal scale and a huge one), 1600 tokens x 5 layers (two rows per
    warp) and 2048 (four rows per warp), the rows a warp instruction serves in
    different layers, with inf / NaN rows mixed in."""
    wl = W.insert_workload(5, T, dtype, num_blocks=256, block_size=64, norm=True, rope=True,
                           seed=47)
    wl.k_scales = np.array([0.0123, 3.0, 1e-36, 1e-39, 1e38], np.float32)
    kv = wl.kv_c.copy()
    kv[2, 7, 5] = 0x7F80   # +inf in one row
    kv[3, 9, 100] = 0x7FC0  # NaN in another
    wl.kv_c = kv
    table = D.gpu_rope_table()
    prev = ops.mla_set_insert_early_tables(False)
    try:
        plain, g1, _ = D.gpu_insert(wl, cos_sin=table, fill=0x21)
        ops.mla_set_insert_early_tables(True)
        trimmed, g2, _ = D.gpu_insert(wl, cos_sin=table, fill=0x21)
    finally:
        ops.mla_set_insert_early_tables(prev)
    assert g1 and g2
    assert_exact(trimmed, plain)
    ref, _ = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE),
                           fill=0x21)
    assert_within_tolerance(plain, ref, dtype)


def _insert_with_tables(wl, kv_c, k_pe, slots, ptr_t, sc_t, gamma, pos, table, err):
    ops.mla_cache_insert_grouped(kv_c, k_pe, slots, ptr_t, sc_t, wl.cache_dtype, wl.num_blocks,
                                 wl.block_size, wl.block_stride, wl.entry_stride, gamma=gamma,
                                 eps=wl.eps, positions=pos, cos_sin_cache=table, err_word=err)


@pytest.mark.parametrize("shape", [0, 2], ids=["rows", "ring"])
def test_layer_tables_written_just_before_each_call(orc, shape):
    """With programmatic dependent launch on, per-layer cache pointers, scales
    and gamma written by ordinary kernels enqueued just before each call (they
    trigger no early launch) are the ones the insert uses, in plain stream
    order (the default) and when the per-layer table is built before the wait
    on the previous grid (mla_set_insert_early_tables), in the row shape and in
    the bulk-copy shape: two back-to-back calls of 4096 tokens x 5 layers
    (e4m3, RMSNorm + RoPE) through ONE pointer array, ONE scale array and ONE
    gamma array into two sets of caches with two sets of scales and gamma.
    Both modes give the same bits, and each set equals the oracle with its own
    scales and gamma."""
    wl = W.insert_workload(5, 4096, 1, num_blocks=128, block_size=64, norm=True, rope=True,
                           seed=43)
    scales = [wl.k_scales, (wl.k_scales * 2.5).astype(np.float32)]
    gammas = [wl.gamma, np.ascontiguousarray(wl.gamma[::-1])]
    table = D.gpu_rope_table()
    kv_c, k_pe = D.dev_bf16(wl.kv_c), D.dev_bf16(wl.k_pe)
    slots = D.dev(np.ascontiguousarray(wl.slot_mapping[0]))
    pos = D.dev(wl.positions)
    src_g = [D.dev_bf16(g) for g in gammas]
    gamma = torch.zeros_like(src_g[0])
    nbytes = wl.num_blocks * wl.block_size * W.ENTRY
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    results = {}
    prev = ops.mla_set_pdl(True)
    prev_early = ops.mla_set_insert_early_tables(False)
    prev_bulk = ops.mla_set_bulk_copy(shape)
    try:
        for early in (False, True):
            ops.mla_set_insert_early_tables(early)
            sets = [[D.Guarded(nbytes) for _ in range(5)] for _ in range(2)]
            for cs in sets:
                for c in cs:
                    c.t.fill_(0x33)
            src_ptrs = [torch.tensor([c.ptr() for c in cs], dtype=torch.int64, device="cuda")
                        for cs in sets]
            src_sc = [D.dev(sc) for sc in scales]
            ptr_t = torch.zeros(5, dtype=torch.int64, device="cuda")
            sc_t = torch.zeros(5, dtype=torch.float32, device="cuda")
            for k in range(2):
                ptr_t.copy_(src_ptrs[k])
                sc_t.copy_(src_sc[k])
                gamma.copy_(src_g[k])
                _insert_with_tables(wl, kv_c, k_pe, slots, ptr_t, sc_t, gamma, pos, table, err)
                if k == 0:  # scramble the arrays after the first call (kernels again)
                    ptr_t.zero_()
                    sc_t.fill_(-1.0)
                    gamma.fill_(0.0)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert all(c.guards_intact() for cs in sets for c in cs)
            results[early] = [[c.host() for c in cs] for cs in sets]
    finally:
        ops.mla_set_pdl(prev)
        ops.mla_set_insert_early_tables(prev_early)
        ops.mla_set_bulk_copy(prev_bulk)
    for k in range(2):
        assert_exact(results[True][k], results[False][k])
        ref, rerr = oracle_insert(orc, dataclasses.replace(wl, k_scales=scales[k], gamma=gammas[k]),
                                  orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE),
                                  fill=0x33)
        assert rerr == 0
        assert_within_tolerance(results[False][k], ref, 1)


@pytest.mark.parametrize("shape", [0, 2], ids=["rows", "ring"])
def test_default_order_sees_layer_tables_written_by_a_pdl_kernel(orc, shape):
    """In the default (plain stream order) the insert reads kv_cache_ptrs and
    kv_scales only after the previous grid has completed, even when that grid
    is a library kernel that lets its dependents launch at its start: here a
    context gather (PDL on, early trigger) copies the five cache pointers and
    scales out of a one-row fp8 "cache" into the buffer the insert then reads
    them from, which held null pointers and zero scales before each copy (a
    null cache pointer would make the insert skip the row and report
    MLA_ERRBIT_MISALIGNED)."""
    wl = W.insert_workload(5, 4096, 1, num_blocks=128, block_size=64, norm=True, rope=True,
                           seed=44)
    nbytes = wl.num_blocks * wl.block_size * W.ENTRY
    caches = [D.Guarded(nbytes) for _ in range(5)]
    for c in caches:
        c.t.fill_(0x33)
    row = np.zeros(64 * W.ENTRY, np.uint8)  # one block of 64 rows; row 0 holds the tables
    row[:40] = np.array([c.ptr() for c in caches], np.int64).view(np.uint8)
    row[64:84] = wl.k_scales.astype(np.float32).view(np.uint8)
    src_t = D.dev(row)
    tab = torch.zeros((1, W.ENTRY), dtype=torch.uint8, device="cuda")
    cu1 = D.dev(np.array([0, 1], np.int32))
    st1 = D.dev(np.array([0], np.int32))
    bt1 = D.dev(np.zeros((1, 1), np.int32))
    table = D.gpu_rope_table()
    kv_c, k_pe = D.dev_bf16(wl.kv_c), D.dev_bf16(wl.k_pe)
    slots = D.dev(np.ascontiguousarray(wl.slot_mapping[0]))
    gamma, pos = D.dev_bf16(wl.gamma), D.dev(wl.positions)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = ops.mla_set_pdl(True)
    prev_early = ops.mla_set_insert_early_tables(False)
    prev_bulk = ops.mla_set_bulk_copy(shape)
    try:
        for _ in range(3):
            tab.zero_()
            ops.mla_context_gather(src_t, 1, 1, 64, 64 * W.ENTRY, W.ENTRY, W.ENTRY, bt1, cu1, st1,
                                   tab, 1)
            _insert_with_tables(wl, kv_c, k_pe, slots, tab[0, :40].view(torch.int64),
                                tab[0, 64:84].view(torch.float32), gamma, pos, table, err)
        torch.cuda.synchronize()
    finally:
        ops.mla_set_pdl(prev)
        ops.mla_set_insert_early_tables(prev_early)
        ops.mla_set_bulk_copy(prev_bulk)
    assert int(err.item()) == 0
    assert all(c.guards_intact() for c in caches)
    ref, rerr = oracle_insert(orc, wl, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE),
                              fill=0x33)
    assert rerr == 0
    assert_within_tolerance([c.host() for c in caches], ref, 1)


# ----------------------------------------------------- full size, as benchmarked
def test_large_insert_65536_tokens_sampled(orc, bulk):
    """65536 tokens x 5 layers, e4m3, RMSNorm + RoPE, caches of 2048 blocks x
    64, one shared mapping -- the benchmarked launch.  The oracle recomputes
    2048 sampled tokens; every row no slot names must stay untouched."""
    wl = W.insert_workload(5, 65536, 1, num_blocks=2048, block_size=64, norm=True, rope=True,
                           seed=40, slot_pool=131072)
    gpu, guards, _ = D.gpu_insert(wl, cos_sin=D.gpu_rope_table(), fill=0x7A)
    assert guards
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(65536, 2048, replace=False))
    sub = W.InsertWorkload(5, 2048, 1, 2048, 64, np.ascontiguousarray(wl.kv_c[:, sample]),
                           np.ascontiguousarray(wl.k_pe[:, sample]),
                           np.ascontiguousarray(wl.slot_mapping[:, sample]), True, wl.k_scales,
                           wl.gamma, np.ascontiguousarray(wl.positions[sample]))
    ref, _ = oracle_insert(orc, sub, orc.rope_cos_sin_cache(W.MAX_POSITION, 64, W.ROPE_BASE),
                           fill=0x7A)
    slots = wl.slot_mapping[0]
    for l in range(5):
        g = gpu[l].reshape(-1, 576)
        r = ref[l].reshape(-1, 576)
        s = slots[sample]
        assert_within_tolerance([g[s].ravel()], [r[s].ravel()], 1)
        written = np.zeros(g.shape[0], bool)
        written[slots] = True
        assert (g[~written] == 0x7A).all()
