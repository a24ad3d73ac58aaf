"""CPU oracle for the MLA latent-KV data-movement path (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import it.  The product
library (``pack_mla_cache_gb300``) never imports, links or calls anything here,
and this package imports nothing from the product.

The arithmetic lives in ``mla_oracle.c`` (plain single-threaded C, fp64 where a
rounded result is produced, compiled with ``-ffp-contract=off``).  This module
only compiles it with gcc and marshals numpy arrays through ctypes.

Passages followed (page title, section):
  * "PR #55356 [Kimi Perf] Group fp8 mla cache insertion" -- Implementation
    items 2-3 and Source snippets (concat_and_cache_mla_grouped_kernel, the host
    validation, test_concat_and_cache_mla_grouped): ``insert_layer``,
    ``insert_grouped``, the fp8 conversion.
  * "PR #50585 [K3 Perf] Optimize k3 dspark fused kv" -- Source snippets
    (_precompute_fused_context_kv): ``rms_norm_row``, ``rope_neox_row``,
    ``rope_cos_sin_cache``.
  * "PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing" --
    Implementation items 1, 2, 5 and Source snippets (fused_mla_kv_concat,
    fused_mla_kv_concat_quant_fp8): ``context_gather``, ``cast_rows``,
    ``concat_key``, ``context_kv_pack``.
  * OCP 8-bit Floating Point Specification (OFP8) rev. 1.0: the e4m3fn and
    e5m2 encodings behind ``fp8_from_f32`` / ``fp8_to_f64``; IEEE 754 binary16
    behind ``f16_from_f64`` / ``f16_to_f64`` (the pack's fp16 inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, FP8_E4M3, FP8_E5M2, F16 = 0, 1, 2, 3
ERR_SLOT_OOB, ERR_BLOCK_OOB, ERR_POS_OOB = 1, 2, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_SPLIT_SRC = os.path.join(_HERE, "mla_oracle_split.c")
_HDR = os.path.join(_HERE, "mla_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (idempotent; rebuilds when the source is newer)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SPLIT_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, "-pthread", _SRC, _SPLIT_SRC, "-o", tmp,
                               "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i32, i64, u32, f32, f64, vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                           ctypes.c_float, ctypes.c_double, ctypes.c_void_p)
            sig = {
                "orc_bf16_from_f64": (ctypes.c_uint16, [f64]),
                "orc_bf16_from_f32": (ctypes.c_uint16, [f32]),
                "orc_bf16_to_f64": (f64, [ctypes.c_uint16]),
                "orc_fp8_from_f32": (ctypes.c_uint8, [f32, ctypes.c_int]),
                "orc_fp8_to_f64": (f64, [ctypes.c_uint8, ctypes.c_int]),
                "orc_bf16_from_fp8": (ctypes.c_uint16, [ctypes.c_uint8, ctypes.c_int]),
                "orc_f16_from_f64": (ctypes.c_uint16, [f64]),
                "orc_f16_to_f64": (f64, [ctypes.c_uint16]),
                "orc_f16_from_fp8": (ctypes.c_uint16, [ctypes.c_uint8, ctypes.c_int]),
                "orc_fp8_encode_f32_array": (None, [vp, i64, ctypes.c_int, vp]),
                "orc_fp8_decode_array": (None, [vp, i64, ctypes.c_int, vp]),
                "orc_bf16_from_f64_array": (None, [vp, i64, vp]),
                "orc_bf16_from_f32_array": (None, [vp, i64, vp]),
                "orc_rope_cos_sin_cache": (None, [i64, i32, f64, vp]),
                "orc_rms_norm_row": (None, [vp, vp, i32, f32, vp]),
                "orc_rope_neox_row": (None, [vp, vp, i32, vp]),
                "orc_insert_layer": (u32, [vp, i64, vp, i64, i32, i32, i32, vp, vp, i32, i64,
                                           i32, i64, i64, f32, vp, f32, vp, vp, i64]),
                "orc_insert_grouped": (u32, [vp, i64, i64, vp, i64, i64, i32, i32, i32, i32,
                                             vp, i64, vp, vp, i32, i64, i32, i64, i64, vp,
                                             i64, f32, vp, vp, i64]),
                "orc_context_gather": (u32, [vp, i32, i64, i32, i64, i64, i32, vp, i64, vp,
                                             vp, i32, i32, vp, i64, i32]),
                "orc_cast_rows": (None, [vp, i32, i64, i64, i64, vp, i32, i64]),
                "orc_concat_key": (None, [vp, i64, i64, vp, i64, i32, i32, i32, i32, vp]),
                "orc_context_kv_pack": (None, [vp, i64, i64, vp, i64, i64, vp, i64, i32, i32,
                                              i32, i32, i32, i32, vp, vp, i32, f32, i32]),
                "orc_norm_rope_grouped": (u32, [vp, i64, i64, vp, i64, i64, i32, i32, i32, i32,
                                                vp, i64, f32, vp, vp, i64, vp, i64, i64, vp, i64,
                                                i64]),
                "orc_bf16_from_fp8_scaled": (ctypes.c_uint16, [ctypes.c_uint8, ctypes.c_int, f32]),
                "orc_context_gather_scaled": (u32, [vp, i32, i64, i32, i64, i64, i32, vp, i64, vp,
                                                    vp, i32, i32, vp, i64, f32]),
                "orc_context_kv_pack_paged": (u32, [vp, i64, i64, vp, i64, i64, vp, i32, i64, i32,
                                                    i64, i64, i32, vp, i64, vp, vp, i32, i32, i32,
                                                    i32, i32, i32, vp, vp, i32, f32, i32]),
                "orc_split_insert_grouped": (u32, [i32, vp, i64, i64, vp, i64, i64, i32, i32, i32,
                                                   i32, vp, i64, vp, vp, i32, i64, i32, i64, i64,
                                                   vp, i64, f32, vp, vp, i64]),
                "orc_split_context_gather": (u32, [i32, vp, i32, i64, i32, i64, i64, i32, vp, i64,
                                                   vp, vp, i32, i32, vp, i64, i32]),
                "orc_split_context_kv_pack": (None, [i32, vp, i64, i64, vp, i64, i64, vp, i64, i32,
                                                     i32, i32, i32, i32, i32, vp, vp, i32, f32,
                                                     i32]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _chk(a, dtype):
    assert isinstance(a, np.ndarray) and a.dtype == dtype, (a.dtype if isinstance(a, np.ndarray) else type(a), dtype)
    assert a.flags["C_CONTIGUOUS"]
    return a


# ---------------------------------------------------------------- scalar codecs
def bf16_from_f64(x: float) -> int:
    return lib().orc_bf16_from_f64(float(x))


def bf16_to_f64(b: int) -> float:
    return lib().orc_bf16_to_f64(int(b))


def fp8_from_f32(x: float, fmt: int) -> int:
    return lib().orc_fp8_from_f32(float(x), fmt)


def fp8_to_f64(c: int, fmt: int) -> float:
    return lib().orc_fp8_to_f64(int(c), fmt)


def bf16_from_fp8(c: int, fmt: int) -> int:
    return lib().orc_bf16_from_fp8(int(c), fmt)


def f16_from_f64(x: float) -> int:
    return lib().orc_f16_from_f64(float(x))


def f16_to_f64(h: int) -> float:
    return lib().orc_f16_to_f64(int(h))


def f16_from_fp8(c: int, fmt: int) -> int:
    return lib().orc_f16_from_fp8(int(c), fmt)


# ----------------------------------------------------------------- array codecs
def fp8_encode(x: np.ndarray, fmt: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_fp8_encode_f32_array(_p(x), x.size, fmt, _p(out))
    return out


def fp8_decode(c: np.ndarray, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_fp8_decode_array(_p(c), c.size, fmt, _p(out))
    return out


def bf16_from_f64_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_f64_array(_p(x), x.size, _p(out))
    return out


def bf16_from_f32_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_f32_array(_p(x), x.size, _p(out))
    return out


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (a bf16 is the top half of an fp32)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# -------------------------------------------------------------- RMSNorm / RoPE
def rope_cos_sin_cache(max_position: int, rot_dim: int, base: float) -> np.ndarray:
    out = np.empty((max_position, rot_dim), np.float32)
    lib().orc_rope_cos_sin_cache(max_position, rot_dim, float(base), _p(out))
    return out


def rms_norm_row(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    x, gamma = _chk(x, np.uint16), _chk(gamma, np.uint16)
    y = np.empty_like(x)
    lib().orc_rms_norm_row(_p(x), _p(gamma), x.size, eps, _p(y))
    return y


def rope_neox_row(x: np.ndarray, cos_sin_row: np.ndarray) -> np.ndarray:
    x, cs = _chk(x, np.uint16), _chk(cos_sin_row, np.float32)
    y = np.empty_like(x)
    lib().orc_rope_neox_row(_p(x), _p(cs), x.size, _p(y))
    return y


# ------------------------------------------------------------------------ insert
def insert_layer(kv_c, k_pe, slot_mapping, cache, cache_dtype, num_blocks, block_size,
                 block_stride, entry_stride, k_scale=1.0, gamma=None, eps=1e-6,
                 positions=None, cos_sin_cache=None):
    """One layer's insert into ``cache`` (a flat numpy buffer, modified in place).

    kv_c [T, R] and k_pe [T, P] are uint16 bf16 bits (row-major, any row stride
    via a 2-D C-contiguous view of the rows); returns the error bits."""
    _chk(kv_c, np.uint16), _chk(k_pe, np.uint16), _chk(slot_mapping, np.int64)
    assert cache.flags["C_CONTIGUOUS"]
    T, R = kv_c.shape
    P = k_pe.shape[1]
    if positions is not None:
        _chk(positions, np.int64), _chk(cos_sin_cache, np.float32)
    return lib().orc_insert_layer(
        _p(kv_c), R, _p(k_pe), P, T, R, P, _p(slot_mapping), _p(cache), cache_dtype,
        num_blocks, block_size, block_stride, entry_stride, float(k_scale),
        _p(gamma), float(eps), _p(positions), _p(cos_sin_cache),
        0 if cos_sin_cache is None else cos_sin_cache.shape[0])


def insert_grouped(kv_c, k_pe, slot_mapping, slot_layer_stride, caches, k_scales, cache_dtype,
                   num_blocks, block_size, block_stride, entry_stride, gamma=None, eps=1e-6,
                   positions=None, cos_sin_cache=None):
    """Grouped insert: kv_c [L, T, R], k_pe [L, T, P] (uint16 bf16 bits, contiguous),
    slot_mapping int64 holding layer l's mapping at l * slot_layer_stride, caches a
    list of L flat numpy buffers (modified in place).  Returns the error bits."""
    _chk(kv_c, np.uint16), _chk(k_pe, np.uint16), _chk(slot_mapping, np.int64)
    L, T, R = kv_c.shape
    P = k_pe.shape[2]
    ptrs = (ctypes.c_void_p * L)(*[c.ctypes.data for c in caches])
    for c in caches:
        assert c.flags["C_CONTIGUOUS"]
    if k_scales is not None:
        k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
    if gamma is not None:
        _chk(gamma, np.uint16)
    if positions is not None:
        _chk(positions, np.int64), _chk(cos_sin_cache, np.float32)
    return lib().orc_insert_grouped(
        _p(kv_c), R, T * R, _p(k_pe), P, T * P, T, L, R, P, _p(slot_mapping), slot_layer_stride,
        ctypes.cast(ptrs, ctypes.c_void_p), _p(k_scales), cache_dtype, num_blocks, block_size,
        block_stride, entry_stride, _p(gamma), 0 if gamma is None else gamma.shape[-1],
        float(eps), _p(positions), _p(cos_sin_cache),
        0 if cos_sin_cache is None else cos_sin_cache.shape[0])


# ------------------------------------------------------------------ gather/cast
def context_gather(cache, cache_dtype, num_blocks, block_size, block_stride, entry_stride,
                   entry_dim, block_table, cu_chunk_lens, chunk_starts, out, out_dtype):
    """Gather into ``out`` (2-D, C-contiguous, modified in place); returns error bits."""
    _chk(block_table, np.int32), _chk(cu_chunk_lens, np.int32), _chk(chunk_starts, np.int32)
    assert out.flags["C_CONTIGUOUS"] and cache.flags["C_CONTIGUOUS"]
    S = chunk_starts.shape[0]
    return lib().orc_context_gather(
        _p(cache), cache_dtype, num_blocks, block_size, block_stride, entry_stride, entry_dim,
        _p(block_table), block_table.shape[1], _p(cu_chunk_lens), _p(chunk_starts), S,
        out.shape[0], _p(out), out.shape[1], out_dtype)


def cast_rows(src, src_dtype, dst_dtype):
    rows, cols = src.shape
    out = np.empty((rows, cols), np.uint16 if dst_dtype in (BF16, F16) else np.uint8)
    lib().orc_cast_rows(_p(np.ascontiguousarray(src)), src_dtype, cols, rows, cols, _p(out),
                        dst_dtype, cols)
    return out


# ------------------------------------------------------------------------- pack
def concat_key(k_nope_rows, kn_token_stride, kn_head_stride, k_pe_rows, kpe_token_stride,
               T, H, nope, rope):
    """bf16 key concat over flat uint16 buffers addressed by element strides."""
    key = np.empty((T, H, nope + rope), np.uint16)
    lib().orc_concat_key(_p(k_nope_rows), kn_token_stride, kn_head_stride, _p(k_pe_rows),
                         kpe_token_stride, T, H, nope, rope, _p(key))
    return key


def context_kv_pack(k_nope_buf, kn_token_stride, kn_head_stride, v_buf, v_token_stride,
                    v_head_stride, k_pe_buf, kpe_token_stride, kpe_dtype, T, H, nope, rope,
                    v_dim, out_dtype, out_scale=1.0, with_v=True, in_dtype=BF16):
    """Fused pack over flat buffers addressed by element strides.

    ``k_nope_buf`` / ``v_buf`` are flat uint16 arrays positioned at the first
    element (numpy views are fine: their data pointer is used).  Returns
    (key [T, H, nope+rope], v [T, H, v_dim] or None) in the output format."""
    odt = np.uint16 if out_dtype in (BF16, F16) else np.uint8
    key = np.empty((T, H, nope + rope), odt)
    vout = np.empty((T, H, v_dim), odt) if with_v else None
    lib().orc_context_kv_pack(_p(k_nope_buf), kn_token_stride, kn_head_stride, _p(v_buf),
                              v_token_stride, v_head_stride, _p(k_pe_buf), kpe_token_stride,
                              kpe_dtype, T, H, nope, rope, v_dim, _p(key), _p(vout),
                              out_dtype, float(out_scale), in_dtype)
    return key, vout


# -------------------------------------------------------------- next steps
def bf16_from_fp8_scaled(c: int, fmt: int, scale: float) -> int:
    return lib().orc_bf16_from_fp8_scaled(int(c), fmt, float(scale))


def context_gather_scaled(cache, cache_dtype, num_blocks, block_size, block_stride, entry_stride,
                          entry_dim, block_table, cu_chunk_lens, chunk_starts, out, dequant_scale):
    """Gather with the scaled fp8 -> bf16 widening into ``out`` (uint16 2-D, in place)."""
    _chk(block_table, np.int32), _chk(cu_chunk_lens, np.int32), _chk(chunk_starts, np.int32)
    _chk(out, np.uint16)
    return lib().orc_context_gather_scaled(
        _p(cache), cache_dtype, num_blocks, block_size, block_stride, entry_stride, entry_dim,
        _p(block_table), block_table.shape[1], _p(cu_chunk_lens), _p(chunk_starts),
        chunk_starts.shape[0], out.shape[0], _p(out), out.shape[1], float(dequant_scale))


def context_kv_pack_paged(k_nope_buf, kn_token_stride, kn_head_stride, v_buf, v_token_stride,
                          v_head_stride, cache, cache_dtype, num_blocks, block_size, block_stride,
                          entry_stride, rope_offset, block_table, cu_chunk_lens, chunk_starts, T,
                          H, nope, rope, v_dim, out_dtype, out_scale=1.0, with_v=True,
                          key_init=None, v_init=None, in_dtype=BF16):
    """Pack with k_pe from the paged cache.  Returns (key, v, error bits); key
    starts as ``key_init`` (rope slices of tokens without a row stay as given)."""
    odt = np.uint16 if out_dtype in (BF16, F16) else np.uint8
    key = (np.array(key_init, dtype=odt, copy=True) if key_init is not None
           else np.zeros((T, H, nope + rope), odt))
    vout = (np.array(v_init, dtype=odt, copy=True) if v_init is not None
            else np.zeros((T, H, v_dim), odt)) if with_v else None
    err = lib().orc_context_kv_pack_paged(
        _p(k_nope_buf), kn_token_stride, kn_head_stride, _p(v_buf), v_token_stride, v_head_stride,
        _p(cache), cache_dtype, num_blocks, block_size, block_stride, entry_stride, rope_offset,
        _p(block_table), block_table.shape[1], _p(cu_chunk_lens), _p(chunk_starts),
        chunk_starts.shape[0], T, H, nope, rope, v_dim, _p(key), _p(vout), out_dtype,
        float(out_scale), in_dtype)
    return key, vout, err


def norm_rope_grouped(kv_c_buf, kvc_ts, kvc_ls, k_pe_buf, kpe_ts, kpe_ls, T, L, R=512, P=64,
                      gamma=None, gamma_ls=512, eps=1e-6, positions=None, cos_sin_cache=None,
                      out_c=None, oc_ts=None, oc_ls=None, out_p=None, op_ts=None, op_ls=None):
    """Grouped RMSNorm + RoPE into layer-major outputs (default [L, T, R] and
    [L, T, P]; pass ``out_c`` / ``out_p`` with strides for other layouts).
    Returns (kv_c_out, k_pe_out, error bits)."""
    if out_c is None:
        out_c, oc_ts, oc_ls = np.zeros((L, T, R), np.uint16), R, T * R
    if out_p is None:
        out_p, op_ts, op_ls = np.zeros((L, T, P), np.uint16), P, T * P
    if gamma is not None:
        _chk(gamma, np.uint16)
    if positions is not None:
        _chk(positions, np.int64), _chk(cos_sin_cache, np.float32)
    err = lib().orc_norm_rope_grouped(
        _p(kv_c_buf), kvc_ts, kvc_ls, _p(k_pe_buf), kpe_ts, kpe_ls, T, L, R, P, _p(gamma),
        gamma_ls, float(eps), _p(positions), _p(cos_sin_cache),
        0 if cos_sin_cache is None else cos_sin_cache.shape[0], _p(out_c), oc_ts, oc_ls,
        _p(out_p), op_ts, op_ls)
    return out_c, out_p, err


# ------------------------------------------------------- split over host threads
def host_threads() -> int:
    """Host cores this process may run on (the multi-core baseline's thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # not Linux
        return os.cpu_count() or 1


def insert_grouped_split(threads, kv_c, k_pe, slot_mapping, slot_layer_stride, caches, k_scales,
                         cache_dtype, num_blocks, block_size, block_stride, entry_stride,
                         gamma=None, eps=1e-6, positions=None, cos_sin_cache=None):
    """``insert_grouped`` with its tokens split over ``threads`` host threads (the
    unchanged single-threaded oracle per token range; byte-identical result)."""
    _chk(kv_c, np.uint16), _chk(k_pe, np.uint16), _chk(slot_mapping, np.int64)
    L, T, R = kv_c.shape
    P = k_pe.shape[2]
    ptrs = (ctypes.c_void_p * L)(*[c.ctypes.data for c in caches])
    for c in caches:
        assert c.flags["C_CONTIGUOUS"]
    if k_scales is not None:
        k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
    if gamma is not None:
        _chk(gamma, np.uint16)
    if positions is not None:
        _chk(positions, np.int64), _chk(cos_sin_cache, np.float32)
    return lib().orc_split_insert_grouped(
        int(threads), _p(kv_c), R, T * R, _p(k_pe), P, T * P, T, L, R, P, _p(slot_mapping),
        slot_layer_stride, ctypes.cast(ptrs, ctypes.c_void_p), _p(k_scales), cache_dtype,
        num_blocks, block_size, block_stride, entry_stride, _p(gamma),
        0 if gamma is None else gamma.shape[-1], float(eps), _p(positions), _p(cos_sin_cache),
        0 if cos_sin_cache is None else cos_sin_cache.shape[0])


def context_gather_split(threads, cache, cache_dtype, num_blocks, block_size, block_stride,
                         entry_stride, entry_dim, block_table, cu_chunk_lens, chunk_starts, out,
                         out_dtype):
    """``context_gather`` with its output rows split over ``threads`` host threads."""
    _chk(block_table, np.int32), _chk(cu_chunk_lens, np.int32), _chk(chunk_starts, np.int32)
    assert out.flags["C_CONTIGUOUS"] and cache.flags["C_CONTIGUOUS"]
    S = chunk_starts.shape[0]
    return lib().orc_split_context_gather(
        int(threads), _p(cache), cache_dtype, num_blocks, block_size, block_stride, entry_stride,
        entry_dim, _p(block_table), block_table.shape[1], _p(cu_chunk_lens), _p(chunk_starts), S,
        out.shape[0], _p(out), out.shape[1], out_dtype)


def context_kv_pack_split(threads, k_nope_buf, kn_token_stride, kn_head_stride, v_buf,
                          v_token_stride, v_head_stride, k_pe_buf, kpe_token_stride, kpe_dtype, T,
                          H, nope, rope, v_dim, out_dtype, out_scale=1.0, with_v=True,
                          in_dtype=BF16):
    """``context_kv_pack`` with its tokens split over ``threads`` host threads."""
    odt = np.uint16 if out_dtype in (BF16, F16) else np.uint8
    key = np.empty((T, H, nope + rope), odt)
    vout = np.empty((T, H, v_dim), odt) if with_v else None
    lib().orc_split_context_kv_pack(int(threads), _p(k_nope_buf), kn_token_stride,
                                    kn_head_stride, _p(v_buf), v_token_stride, v_head_stride,
                                    _p(k_pe_buf), kpe_token_stride, kpe_dtype, T, H, nope, rope,
                                    v_dim, _p(key), _p(vout), out_dtype, float(out_scale),
                                    in_dtype)
    return key, vout
