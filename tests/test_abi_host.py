"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* the library builds, loads, and exports every entry point include/mla_cache.h
  declares;
* the vLLM cache-dtype strings map as the grouped insert's host whitelist does
  ("PR #55356 [Kimi Perf] Group fp8 mla cache insertion", Source snippets:
  "auto"/"bfloat16", "fp8"/"fp8_e4m3", "fp8_e5m2");
* every argument check rejects its case with the documented status before any
  CUDA call (fake, never-dereferenced addresses are used), including the
  pages' "FP8 ... requires kv_scales" and "BF16 ... does not use kv_scales";
* a call that passes validation on a machine without a GPU fails with
  MLA_ERR_CUDA instead of crashing.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from pack_mla_cache_gb300 import build as B
from pack_mla_cache_gb300 import ops

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "mla_cache.h")
A = 0x7F0000000000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def L():
    B.build()
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_expected_entry_points():
    assert declared_functions() == sorted(ops.SIGNATURES)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mla_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(L, name)


def test_version_and_dtype_strings(L):
    assert "sm_103a" in ops.mla_version()
    m = {"auto": 0, "bfloat16": 0, "fp8": 1, "fp8_e4m3": 1, "fp8_e5m2": 2}
    for s, code in m.items():
        assert ops.mla_dtype_from_string(s) == code
    for s in ("fp16", "fp8_ds_mla", "", "FP8"):
        assert ops.mla_dtype_from_string(s) == -1


def test_pdl_and_bulk_copy_toggles(L):
    prev = ops.mla_set_pdl(False)
    assert ops.mla_set_pdl(True) is False
    ops.mla_set_pdl(prev)
    prev = ops.mla_set_bulk_copy(0)
    assert ops.mla_set_bulk_copy(2) == 0
    assert ops.mla_set_bulk_copy(7) == 2      # out of range sets the default
    assert ops.mla_set_bulk_copy(prev) == 1


def test_pointer_check_early_table_and_timeout_hook_toggles(L):
    prev = ops.mla_set_pointer_checks(False)
    assert ops.mla_set_pointer_checks(True) is False
    ops.mla_set_pointer_checks(prev)
    assert prev is True  # checked by default
    prev = ops.mla_set_gather_early_tables(True)
    assert prev is False  # plain stream order by default
    assert ops.mla_set_gather_early_tables(False) is True
    prev = ops.mla_set_insert_early_tables(True)
    assert prev is False  # plain stream order by default
    assert ops.mla_set_insert_early_tables(False) is True
    assert L.mla_test_insert_timeout(1000, 5) == 0
    assert L.mla_test_insert_timeout(0, -1) == 0  # defaults back


def insert(L, **kw):
    args = dict(kv_c=A, kvc_ts=512, kvc_ls=512 * 8, k_pe=A + 4096, kpe_ts=64, kpe_ls=64 * 8,
                T=8, nl=5, R=512, P=64, slots=A + 8192, sls=0, ptrs=A + 16384, scales=A + 32768,
                dtype=1, nb=64, bs=64, bstride=64 * 576, estride=576, nr=None, err=None)
    args.update(kw)
    return L.mla_cache_insert_grouped(
        args["kv_c"], args["kvc_ts"], args["kvc_ls"], args["k_pe"], args["kpe_ts"],
        args["kpe_ls"], args["T"], args["nl"], args["R"], args["P"], args["slots"], args["sls"],
        args["ptrs"], args["scales"], args["dtype"], args["nb"], args["bs"], args["bstride"],
        args["estride"], args["nr"], args["err"], None)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(T=-1), ops.MLA_ERR_INVALID_ARG, "num_tokens"),
    (dict(nl=0), ops.MLA_ERR_INVALID_ARG, "num_layers"),
    (dict(dtype=7), ops.MLA_ERR_INVALID_ARG, "cache_dtype"),
    (dict(dtype=3), ops.MLA_ERR_INVALID_ARG, "cache_dtype"),  # no fp16 caches in the insert
    (dict(R=256), ops.MLA_ERR_UNSUPPORTED, "kv_lora_rank"),
    (dict(P=32), ops.MLA_ERR_UNSUPPORTED, "pe_dim"),
    (dict(scales=None), ops.MLA_ERR_INVALID_ARG, "FP8 grouped cache insert requires kv_scales"),
    (dict(dtype=0, bstride=64 * 576), ops.MLA_ERR_INVALID_ARG, "BF16 grouped cache insert does not use kv_scales"),
    (dict(kv_c=None), ops.MLA_ERR_INVALID_ARG, "non-null"),
    (dict(slots=None), ops.MLA_ERR_INVALID_ARG, "non-null"),
    (dict(ptrs=None), ops.MLA_ERR_INVALID_ARG, "non-null"),
    (dict(sls=-1), ops.MLA_ERR_INVALID_ARG, "slot_layer_stride"),
    (dict(bs=0), ops.MLA_ERR_INVALID_ARG, "block_size"),
    (dict(estride=500), ops.MLA_ERR_INVALID_ARG, "entry_stride"),
    (dict(bstride=576), ops.MLA_ERR_INVALID_ARG, "block_stride"),
    (dict(kv_c=A + 8), ops.MLA_ERR_MISALIGNED, "kv_c"),
    (dict(kvc_ts=500), ops.MLA_ERR_MISALIGNED, "kv_c"),
    (dict(k_pe=A + 2), ops.MLA_ERR_MISALIGNED, "k_pe"),
    (dict(kpe_ls=100), ops.MLA_ERR_MISALIGNED, "k_pe"),
    (dict(estride=580, bstride=64 * 580), ops.MLA_ERR_MISALIGNED, "entry_stride"),
    (dict(slots=A + 4), ops.MLA_ERR_MISALIGNED, "8-byte"),
    (dict(err=A + 2), ops.MLA_ERR_MISALIGNED, "err_word"),
])
def test_insert_argument_checks(L, kw, status, msg):
    assert insert(L, **kw) == status
    assert msg in ops.mla_last_error()


def test_insert_norm_rope_checks(L):
    nr = ops.NormRope(A + 8, 512, 1e-6, None, None, 0)
    assert insert(L, nr=ctypes.byref(nr)) == ops.MLA_ERR_MISALIGNED
    nr = ops.NormRope(A, 512, -1.0, None, None, 0)
    assert insert(L, nr=ctypes.byref(nr)) == ops.MLA_ERR_INVALID_ARG
    nr = ops.NormRope(None, 0, 1e-6, A, None, 0)
    assert insert(L, nr=ctypes.byref(nr)) == ops.MLA_ERR_INVALID_ARG
    assert "cos_sin_cache" in ops.mla_last_error()
    nr = ops.NormRope(None, 0, 1e-6, A, A + 4, 32768)
    assert insert(L, nr=ctypes.byref(nr)) == ops.MLA_ERR_MISALIGNED


def test_zero_tokens_is_a_no_op_without_cuda(L):
    assert insert(L, T=0) == ops.MLA_OK
    assert L.mla_context_kv_pack(A, 4160, 256, A, 4160, 256, 0, A, 576, 1, 0, 16, 128, 64, 128,
                                 A, A, 1, None, None, None) == ops.MLA_OK


def test_validated_call_without_gpu_reports_cuda_error(L):
    if torch.cuda.is_available():
        pytest.skip("this check is for machines without a GPU")
    assert insert(L) == ops.MLA_ERR_CUDA
    assert "cudaPointerGetAttributes" in ops.mla_last_error()
    assert "kv_c" in ops.mla_last_error()  # the first pointer checked


def test_pointer_checks_off_skips_the_runtime_queries_without_gpu(L):
    """With the checks off nothing asks the runtime about the pointers; on a
    machine without a GPU the call then fails at the launch.  (Never run with
    these fake addresses where a GPU could dereference them.)"""
    if torch.cuda.is_available():
        pytest.skip("this check is for machines without a GPU")
    prev = ops.mla_set_pointer_checks(False)
    try:
        assert insert(L) == ops.MLA_ERR_CUDA
        assert "cudaPointerGetAttributes" not in ops.mla_last_error()
    finally:
        ops.mla_set_pointer_checks(prev)


def gather(L, **kw):
    a = dict(cache=A, cdt=1, nb=1024, bs=64, bstride=64 * 576, estride=576, edim=576, bt=A,
             bts=512, cu=A + 4096, st=A + 8192, S=1, T=8192, out=A + 65536, ors=576, odt=1,
             err=None)
    a.update(kw)
    return L.mla_context_gather(a["cache"], a["cdt"], a["nb"], a["bs"], a["bstride"],
                                a["estride"], a["edim"], a["bt"], a["bts"], a["cu"], a["st"],
                                a["S"], a["T"], a["out"], a["ors"], a["odt"], a["err"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), ops.MLA_ERR_INVALID_ARG),
    (dict(S=0), ops.MLA_ERR_INVALID_ARG),
    (dict(cdt=0, odt=1), ops.MLA_ERR_UNSUPPORTED),
    (dict(cdt=1, odt=2), ops.MLA_ERR_UNSUPPORTED),
    (dict(cdt=0, odt=3), ops.MLA_ERR_UNSUPPORTED),     # bf16 rows are not widened to fp16
    (dict(cdt=3, odt=0), ops.MLA_ERR_UNSUPPORTED),
    (dict(bt=None), ops.MLA_ERR_INVALID_ARG),
    (dict(edim=600), ops.MLA_ERR_INVALID_ARG),
    (dict(edim=570, estride=576), ops.MLA_ERR_MISALIGNED),
    (dict(ors=500), ops.MLA_ERR_INVALID_ARG),
    (dict(out=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(cache=A + 4), ops.MLA_ERR_MISALIGNED),
    (dict(bts=0), ops.MLA_ERR_INVALID_ARG),
    (dict(cdt=0, odt=0, edim=1024, estride=1024, bstride=64 * 1024, ors=1024), ops.MLA_ERR_UNSUPPORTED),
])
def test_gather_argument_checks(L, kw, status):
    assert gather(L, **kw) == status


def gather_scaled(L, **kw):
    a = dict(cache=A, cdt=1, nb=1024, bs=64, bstride=64 * 576, estride=576, edim=576, bt=A,
             bts=512, cu=A + 4096, st=A + 8192, S=1, T=8192, out=A + 65536, ors=576,
             scale=A + 128, err=None)
    a.update(kw)
    return L.mla_context_gather_scaled(a["cache"], a["cdt"], a["nb"], a["bs"], a["bstride"],
                                       a["estride"], a["edim"], a["bt"], a["bts"], a["cu"],
                                       a["st"], a["S"], a["T"], a["out"], a["ors"], a["scale"],
                                       a["err"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), ops.MLA_ERR_INVALID_ARG),
    (dict(cdt=0), ops.MLA_ERR_UNSUPPORTED),      # a bf16 cache has nothing to dequantise
    (dict(cdt=3), ops.MLA_ERR_UNSUPPORTED),
    (dict(cdt=7), ops.MLA_ERR_INVALID_ARG),
    (dict(scale=None), ops.MLA_ERR_INVALID_ARG),
    (dict(scale=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(S=0), ops.MLA_ERR_INVALID_ARG),
    (dict(out=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(ors=572), ops.MLA_ERR_INVALID_ARG),
    (dict(ors=580), ops.MLA_ERR_MISALIGNED),     # 1160-byte bf16 rows
    (dict(bstride=63 * 576), ops.MLA_ERR_INVALID_ARG),
    (dict(edim=2048, estride=2048, bstride=64 * 2048, ors=2048), ops.MLA_ERR_UNSUPPORTED),
    (dict(cu=A + 2), ops.MLA_ERR_MISALIGNED),
])
def test_gather_scaled_argument_checks(L, kw, status):
    assert gather_scaled(L, **kw) == status


def test_gather_scaled_zero_tokens_is_ok_without_pointers(L):
    assert gather_scaled(L, T=0, cache=None, bt=None, cu=None, st=None, out=None) == ops.MLA_OK


def pack_paged(L, **kw):
    a = dict(kn=A, kts=4160, khs=256, v=A + 256, vts=4160, vhs=256, idt=0, cache=A + (3 << 30),
             cdt=1,
             nb=1024, bs=64, bstride=64 * 576, estride=576, roff=512, bt=A + 4096, bts=512,
             cu=A + 8192, st=A + 12288, S=1, T=8192, H=16, N=128, R=64, V=128,
             key=A + (1 << 30), vout=A + (2 << 30), odt=1, scale=None, err=None)
    a.update(kw)
    return L.mla_context_kv_pack_paged(
        a["kn"], a["kts"], a["khs"], a["v"], a["vts"], a["vhs"], a["idt"], a["cache"], a["cdt"],
        a["nb"],
        a["bs"], a["bstride"], a["estride"], a["roff"], a["bt"], a["bts"], a["cu"], a["st"],
        a["S"], a["T"], a["H"], a["N"], a["R"], a["V"], a["key"], a["vout"], a["odt"],
        a["scale"], a["err"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), ops.MLA_ERR_INVALID_ARG),
    (dict(H=0), ops.MLA_ERR_INVALID_ARG),
    (dict(S=0), ops.MLA_ERR_INVALID_ARG),
    (dict(R=32), ops.MLA_ERR_UNSUPPORTED),
    (dict(cdt=2, odt=1), ops.MLA_ERR_UNSUPPORTED),  # fp8 k_pe bytes of another format
    (dict(cdt=5), ops.MLA_ERR_INVALID_ARG),
    (dict(odt=0, scale=A), ops.MLA_ERR_INVALID_ARG),
    (dict(roff=520), ops.MLA_ERR_INVALID_ARG),      # 520 + 64 > entry_stride
    (dict(roff=-8), ops.MLA_ERR_INVALID_ARG),
    (dict(roff=508), ops.MLA_ERR_MISALIGNED),       # fp8 k_pe must start on 8 bytes
    (dict(cdt=0, odt=0, roff=508, bstride=64 * 576), ops.MLA_ERR_MISALIGNED),
    (dict(cache=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(estride=580, bstride=64 * 580), ops.MLA_ERR_MISALIGNED),
    (dict(bstride=63 * 576 + 575), ops.MLA_ERR_INVALID_ARG),
    (dict(bts=0), ops.MLA_ERR_INVALID_ARG),
    (dict(nb=0), ops.MLA_ERR_INVALID_ARG),
    (dict(bt=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(kn=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(key=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(err=A + 1), ops.MLA_ERR_MISALIGNED),
    (dict(cache=None), ops.MLA_ERR_INVALID_ARG),
    (dict(bt=None), ops.MLA_ERR_INVALID_ARG),
    (dict(kn=None), ops.MLA_ERR_INVALID_ARG),
    (dict(idt=3, cdt=0, odt=1), ops.MLA_ERR_UNSUPPORTED),  # bf16 cache rows, fp16 k_nope
])
def test_pack_paged_argument_checks(L, kw, status):
    assert pack_paged(L, **kw) == status


def test_pack_paged_zero_tokens_is_ok_without_pointers(L):
    assert pack_paged(L, T=0, kn=None, v=None, cache=None, bt=None, cu=None, st=None, key=None,
                      vout=None) == ops.MLA_OK


def test_paged_calls_that_pass_validation_need_a_gpu(L):
    if torch.cuda.is_available():
        pytest.skip("this check is for machines without a GPU")
    assert pack_paged(L) == ops.MLA_ERR_CUDA
    assert gather_scaled(L) == ops.MLA_ERR_CUDA


def norm_rope(L, nr=None, **kw):
    a = dict(kvc=A, kts=5 * 576, kls=576, kpe=A + 1024, pts=5 * 576, pls=576, T=4096, Ly=5,
             R=512, P=64, oc=A + (1 << 30), octs=512, ocls=4096 * 512, op=A + (2 << 30),
             opts=64, opls=4096 * 64, err=None)
    a.update(kw)
    return L.mla_norm_rope_grouped(a["kvc"], a["kts"], a["kls"], a["kpe"], a["pts"], a["pls"],
                                   a["T"], a["Ly"], a["R"], a["P"],
                                   ctypes.byref(nr) if nr is not None else None, a["oc"],
                                   a["octs"], a["ocls"], a["op"], a["opts"], a["opls"], a["err"],
                                   None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), ops.MLA_ERR_INVALID_ARG),
    (dict(Ly=0), ops.MLA_ERR_INVALID_ARG),
    (dict(R=256), ops.MLA_ERR_UNSUPPORTED),
    (dict(P=32), ops.MLA_ERR_UNSUPPORTED),
    (dict(kvc=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(kls=580), ops.MLA_ERR_MISALIGNED),
    (dict(kpe=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(oc=A + 4), ops.MLA_ERR_MISALIGNED),
    (dict(octs=500), ops.MLA_ERR_MISALIGNED),
    (dict(op=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(opls=4), ops.MLA_ERR_MISALIGNED),
    (dict(err=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(T=1 << 30, Ly=8), ops.MLA_ERR_UNSUPPORTED),
    (dict(kvc=None), ops.MLA_ERR_INVALID_ARG),
    (dict(op=None), ops.MLA_ERR_INVALID_ARG),
])
def test_norm_rope_argument_checks(L, kw, status):
    assert norm_rope(L, **kw) == status


def test_norm_rope_description_checks(L):
    bad_gamma = ops.NormRope(A + 2, 512, 1e-6, None, None, 0)
    assert norm_rope(L, bad_gamma) == ops.MLA_ERR_MISALIGNED
    bad_eps = ops.NormRope(A, 512, -1.0, None, None, 0)
    assert norm_rope(L, bad_eps) == ops.MLA_ERR_INVALID_ARG
    no_table = ops.NormRope(None, 0, 0.0, A, None, 32768)
    assert norm_rope(L, no_table) == ops.MLA_ERR_INVALID_ARG
    bad_pos = ops.NormRope(None, 0, 0.0, A + 4, A, 32768)
    assert norm_rope(L, bad_pos) == ops.MLA_ERR_MISALIGNED
    assert norm_rope(L, T=0, kvc=None, kpe=None, oc=None, op=None) == ops.MLA_OK
    if not torch.cuda.is_available():
        assert norm_rope(L) == ops.MLA_ERR_CUDA  # valid; the launch needs a GPU
        ok = ops.NormRope(A, 512, 1e-6, A + 64, A + 128, 32768)
        assert norm_rope(L, ok) == ops.MLA_ERR_CUDA


def pack(L, **kw):
    a = dict(kn=A, kts=4160, khs=256, v=A + 256, vts=4160, vhs=256, idt=0, kpe=A + 1024,
             kpets=576, kdt=1, T=8192, H=16, N=128, R=64, V=128, key=A + (1 << 30),
             vout=A + (2 << 30), odt=1, scale=None, err=None)
    a.update(kw)
    return L.mla_context_kv_pack(a["kn"], a["kts"], a["khs"], a["v"], a["vts"], a["vhs"],
                                 a["idt"], a["kpe"], a["kpets"], a["kdt"], a["T"], a["H"], a["N"],
                                 a["R"],
                                 a["V"], a["key"], a["vout"], a["odt"], a["scale"], a["err"],
                                 None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), ops.MLA_ERR_INVALID_ARG),
    (dict(H=0), ops.MLA_ERR_INVALID_ARG),
    (dict(N=64), ops.MLA_ERR_UNSUPPORTED),
    (dict(V=64), ops.MLA_ERR_UNSUPPORTED),
    (dict(kdt=2, odt=1), ops.MLA_ERR_UNSUPPORTED),
    (dict(odt=0, kdt=0, scale=A), ops.MLA_ERR_INVALID_ARG),
    (dict(kn=None), ops.MLA_ERR_INVALID_ARG),
    (dict(kn=A + 2), ops.MLA_ERR_MISALIGNED),
    (dict(khs=100), ops.MLA_ERR_MISALIGNED),
    (dict(v=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(kpe=A + 4), ops.MLA_ERR_MISALIGNED),
    (dict(kdt=0, kpe=A + 8, odt=0), ops.MLA_ERR_MISALIGNED),
    (dict(key=A + 8), ops.MLA_ERR_MISALIGNED),
    (dict(odt=9), ops.MLA_ERR_INVALID_ARG),
    (dict(err=A + 1), ops.MLA_ERR_MISALIGNED),
    (dict(idt=1), ops.MLA_ERR_UNSUPPORTED),            # k_nope / v must be 16-bit
    (dict(idt=7), ops.MLA_ERR_INVALID_ARG),
    (dict(idt=3, odt=0, kdt=0), ops.MLA_ERR_UNSUPPORTED),  # fp16 input, bf16 output
    (dict(idt=3, odt=1, kdt=0), ops.MLA_ERR_UNSUPPORTED),  # bf16 k_pe with fp16 k_nope
    (dict(idt=0, odt=3, kdt=1), ops.MLA_ERR_UNSUPPORTED),  # fp16 output of bf16 input
    (dict(idt=3, odt=3, kdt=3, scale=A), ops.MLA_ERR_INVALID_ARG),
    (dict(T=1 << 30, H=20), ops.MLA_ERR_UNSUPPORTED),  # 5 * 2^30 work items
])
def test_pack_argument_checks(L, kw, status):
    assert pack(L, **kw) == status


def test_rope_table_argument_checks(L):
    assert L.mla_rope_cos_sin_cache(None, 10, 64, 1e4, None) == ops.MLA_ERR_INVALID_ARG
    assert L.mla_rope_cos_sin_cache(A, 10, 63, 1e4, None) == ops.MLA_ERR_INVALID_ARG
    assert L.mla_rope_cos_sin_cache(A, 0, 64, 1e4, None) == ops.MLA_ERR_INVALID_ARG
    assert L.mla_rope_cos_sin_cache(A, 10, 64, 0.5, None) == ops.MLA_ERR_INVALID_ARG
    assert L.mla_rope_cos_sin_cache(A + 4, 10, 64, 1e4, None) == ops.MLA_ERR_MISALIGNED


def test_error_message_is_thread_local(L):
    import threading
    insert(L, T=-1)
    seen = []
    t = threading.Thread(target=lambda: seen.append(ops.mla_last_error()))
    t.start()
    t.join()
    assert seen == [""]
    assert "num_tokens" in ops.mla_last_error()


# ------------------------------------------------ pack + next gather, one launch
def fused_descs(**kw):
    """Descriptors of an fp8 pack (8192 tokens, 16 heads, k_pe from workspace
    A) and a raw fp8 gather of 8192 rows into workspace B (fake addresses)."""
    ws_a, ws_b = A + (1 << 30), A + (1 << 31)
    p = dict(k_nope=A, kn_token_stride=4160, kn_head_stride=256, v=A + 256, v_token_stride=4160,
             v_head_stride=256, in_dtype=0, k_pe=ws_a + 1024, kpe_token_stride=576, kpe_dtype=1,
             num_tokens=8192, num_heads=16, nope_dim=128, rope_dim=64, v_dim=128,
             key_out=A + (1 << 32), v_out=A + (1 << 33), out_dtype=1, out_scale=A + 64)
    g = dict(kv_cache=A + (1 << 34), cache_dtype=1, num_blocks=1024, block_size=64,
             block_stride=64 * 576, entry_stride=576, entry_dim=576, block_table=A + 4096,
             block_table_stride=512, cu_chunk_lens=A + 8192, chunk_starts=A + 12288, num_seqs=1,
             num_tokens=8192, out=ws_b, out_row_stride=576, out_dtype=1)
    for k, v in kw.items():  # g_<name>: the gather's field of that name
        if k.startswith("g_"):
            g[k[2:]] = v
        else:
            (p if k in p else g)[k] = v
    return ops.KvPack(**p), ops.ContextGather(**g)


def fused(L, **kw):
    import ctypes
    pk, gk = fused_descs(**kw)
    return L.mla_context_kv_pack_gather(ctypes.byref(pk), ctypes.byref(gk), None, None)


def test_fused_pack_gather_argument_checks(L):
    import ctypes
    pk, gk = fused_descs()
    assert L.mla_context_kv_pack_gather(None, ctypes.byref(gk), None, None) == \
        ops.MLA_ERR_INVALID_ARG
    assert L.mla_context_kv_pack_gather(ctypes.byref(pk), None, None, None) == \
        ops.MLA_ERR_INVALID_ARG
    # the gather must write its cache's type or the pack's input type
    assert fused(L, out_dtype=0, in_dtype=3, kn_token_stride=4160) == ops.MLA_ERR_UNSUPPORTED
    # the pack half keeps its own rules (bad head count), the gather half its own
    assert fused(L, num_heads=0) == ops.MLA_ERR_INVALID_ARG
    assert fused(L, num_seqs=0) == ops.MLA_ERR_INVALID_ARG
    # both halves empty: nothing to do, no CUDA call
    assert fused(L, num_tokens=0, g_num_tokens=0) == ops.MLA_OK


@pytest.mark.parametrize("target", ["k_pe", "k_nope", "key_out", "v_out"])
def test_fused_pack_gather_rejects_overlap_before_any_cuda_call(L, target):
    """The gather's output must not overlap any buffer of the pack; the check
    runs before any CUDA call, so it is the error even without a GPU."""
    pk, _ = fused_descs()
    addr = getattr(pk, target) + 64
    assert fused(L, out=addr) == ops.MLA_ERR_INVALID_ARG
    assert "overlaps" in ops.mla_last_error()


def test_fused_pack_gather_without_gpu_reports_cuda_error(L):
    if torch.cuda.is_available():
        pytest.skip("this check is for machines without a GPU")
    assert fused(L) == ops.MLA_ERR_CUDA
    assert "cudaPointerGetAttributes" in ops.mla_last_error()
