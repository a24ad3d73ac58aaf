"""GPU parity of the chunked-context path with fp16 inputs against the CPU
oracle, through the C ABI -- bit-exact ("PR #51772 [Attention][MLA] Fuse
Kimi-K3 chunked-context K/V packing", Review: the fused kernel is tested with
bf16 and fp16 inputs and fp8 must match bit for bit).

Covers: an 8192-token fp16 kv_b_proj output packed to fp16 (fp16 k_pe, and fp8
k_pe widened) and to fp8 e4m3 / e5m2; runtime head counts with ragged token
counts; all 2^16 fp16 bit patterns through the fp8 pack at ordinary scales and
at a scale so small that every value takes the guarded division; the gather's
exact widening of every fp8 code into fp16 rows and of 8192-row chunks; the
paged pack with fp16 inputs.
"""
import numpy as np
import pytest
import torch

import devutil as D
from pack_mla_cache_gb300 import ops
from pack_mla_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu
ENTRY = 576
F16 = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pack_mla_cache_gb300 import build
    build.build()
    ops.lib()


def dev_f16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()


def f16_rows(T, cols, seed, scale=4.0):
    rng = np.random.default_rng(seed)
    return np.ascontiguousarray(
        (rng.standard_normal((T, cols)) * scale).astype(np.float16).view(np.uint16))


def run_pack(kvb, kpe, kpe_dtype, H, out_dtype, scale):
    T = kvb.shape[0]
    heads = dev_f16(kvb)[:, : H * 256].view(T, H, 256)
    k_pe = dev_f16(kpe) if kpe_dtype == F16 else D.dev(kpe)
    odt = torch.float16 if out_dtype == F16 else torch.uint8
    key = torch.zeros((T, H, 192), dtype=odt, device="cuda")
    vo = torch.zeros((T, H, 128), dtype=odt, device="cuda")
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda") if out_dtype != F16 else None
    ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:], k_pe, key, vo, out_dtype,
                            kpe_dtype=kpe_dtype, out_scale=sc)
    torch.cuda.synchronize()
    conv = D.host_u16 if out_dtype == F16 else D.host_u8
    return conv(key), conv(vo)


def oracle_pack(orc, kvb, kpe, kpe_dtype, H, out_dtype, scale):
    T, rs = kvb.shape
    return orc.context_kv_pack(kvb, rs, 256, kvb[:, 128:], rs, 256, kpe, kpe.shape[1], kpe_dtype,
                               T, H, 128, 64, 128, out_dtype,
                               scale if out_dtype != F16 else 1.0, True, in_dtype=F16)


@pytest.mark.parametrize("out_dtype,kpe_dtype", [(F16, F16), (F16, 1), (F16, 2), (1, F16),
                                                 (1, 1), (2, F16), (2, 2)])
def test_fp16_pack_8192_tokens(orc, out_dtype, kpe_dtype):
    T, H = 8192, 16
    kvb = f16_rows(T, 4160, 1)
    if kpe_dtype == F16:
        kpe = f16_rows(T, 64, 2)
    else:
        kpe = np.random.default_rng(3).integers(0, 256, size=(T, 64)).astype(np.uint8)
    gk, gv = run_pack(kvb, kpe, kpe_dtype, H, out_dtype, 0.01)
    rk, rv = oracle_pack(orc, kvb, kpe, kpe_dtype, H, out_dtype, 0.01)
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)


@pytest.mark.parametrize("H", [1, 3, 20])
@pytest.mark.parametrize("T", [1, 77])
def test_fp16_pack_runtime_heads(orc, H, T):
    kvb = f16_rows(T, H * 256 + 64, 4 + H)
    kpe = np.random.default_rng(5).integers(0, 126, size=(T, 64)).astype(np.uint8)
    for out_dtype in (F16, 1):
        gk, gv = run_pack(kvb, kpe, 1, H, out_dtype, 0.05)
        rk, rv = oracle_pack(orc, kvb, kpe, 1, H, out_dtype, 0.05)
        np.testing.assert_array_equal(gk, rk)
        np.testing.assert_array_equal(gv, rv)


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("scale", [0.01, 3.0, 1e-35])
def test_fp16_to_fp8_exhaustive(orc, fmt, scale):
    """All 2^16 fp16 patterns (16 tokens x 16 heads x 256): zeros, subnormals,
    overflowing quotients, infinities and NaNs.  At scale 1e-35 the reciprocal
    exceeds 2^111, so every nonzero value takes the guarded division."""
    T, H = 16, 16
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(T, H * 256)
    kvb = np.zeros((T, 4160), np.uint16)
    kvb[:, : H * 256] = pats
    kpe = pats[:, :64].copy()
    gk, gv = run_pack(kvb, kpe, F16, H, fmt, scale)
    rk, rv = oracle_pack(orc, kvb, kpe, F16, H, fmt, scale)
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)


def gpu_gather_f16(pw, table, cu, st, T):
    out = torch.full((T, ENTRY), 0x1234, dtype=torch.int16, device="cuda").view(torch.float16)
    ops.mla_context_gather(dev_cache(pw), pw.cache_dtype, pw.num_blocks, pw.block_size,
                           pw.block_size * ENTRY, ENTRY, ENTRY, D.dev(table), D.dev(cu), D.dev(st),
                           out, F16)
    torch.cuda.synchronize()
    return D.host_u16(out)


def dev_cache(pw):
    return D.dev(pw.cache)


def oracle_gather_f16(orc, pw, table, cu, st, T):
    out = np.full((T, ENTRY), 0x1234, np.uint16)
    err = orc.context_gather(pw.cache, pw.cache_dtype, pw.num_blocks, pw.block_size,
                             pw.block_size * ENTRY, ENTRY, ENTRY, table, cu, st, out, F16)
    assert err == 0
    return out


@pytest.mark.parametrize("fmt", [1, 2])
def test_gather_widens_every_code_into_fp16(orc, fmt):
    pw = W.pack_workload(64, 64, num_blocks=1, cache_dtype=fmt, seed=4)
    pw.cache[:] = (np.arange(pw.cache.size) % 256).astype(np.uint8)
    cu, st = np.array([0, 64], np.int32), np.array([0], np.int32)
    np.testing.assert_array_equal(gpu_gather_f16(pw, pw.block_table, cu, st, 64),
                                  oracle_gather_f16(orc, pw, pw.block_table, cu, st, 64))


def test_gather_fp16_rows_8192(orc):
    pw = W.pack_workload(16448, 8192, num_blocks=512, seed=6, cache_dtype=2)
    for c in range(2):
        cu, st = np.array([0, 8192], np.int32), np.array([c * 8192 + 5], np.int32)
        np.testing.assert_array_equal(gpu_gather_f16(pw, pw.block_table, cu, st, 8192),
                                      oracle_gather_f16(orc, pw, pw.block_table, cu, st, 8192))


@pytest.mark.parametrize("out_dtype", [F16, 1])
def test_paged_pack_fp16_inputs(orc, out_dtype):
    T, H = 3000, 16
    pw = W.pack_workload(4096, 4096, num_blocks=128, seed=7)
    kvb = f16_rows(T, 4160, 8)
    cu, st = np.array([0, T], np.int32), np.array([21], np.int32)
    heads = dev_f16(kvb)[:, :4096].view(T, H, 256)
    odt = torch.float16 if out_dtype == F16 else torch.uint8
    key = torch.zeros((T, H, 192), dtype=odt, device="cuda")
    vo = torch.zeros((T, H, 128), dtype=odt, device="cuda")
    sc = torch.tensor([0.02], dtype=torch.float32, device="cuda") if out_dtype != F16 else None
    ops.mla_context_kv_pack_paged(heads[:, :, :128], heads[:, :, 128:], D.dev(pw.cache), 1,
                                  pw.num_blocks, 64, 64 * ENTRY, ENTRY, D.dev(pw.block_table),
                                  D.dev(cu), D.dev(st), key, vo, out_dtype, out_scale=sc)
    torch.cuda.synchronize()
    rs = kvb.shape[1]
    rk, rv, err = orc.context_kv_pack_paged(
        kvb, rs, 256, kvb[:, 128:], rs, 256, pw.cache, 1, pw.num_blocks, 64, 64 * ENTRY, ENTRY,
        512, pw.block_table, cu, st, T, H, 128, 64, 128, out_dtype,
        0.02 if out_dtype != F16 else 1.0, in_dtype=F16)
    assert err == 0
    conv = D.host_u16 if out_dtype == F16 else D.host_u8
    np.testing.assert_array_equal(conv(key), rk)
    np.testing.assert_array_equal(conv(vo), rv)
