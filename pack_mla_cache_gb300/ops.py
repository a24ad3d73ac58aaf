"""Thin Python binding of libmla_cache (include/mla_cache.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Each function has the name of the C entry point it calls, takes
torch tensors (device memory) and forwards their data pointers, element
strides and the current CUDA stream.  A failing call raises ``MlaError`` with
the library's status and message.  There is no fallback: if the library is
not built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

MLA_BF16, MLA_FP8_E4M3, MLA_FP8_E5M2, MLA_FP16 = 0, 1, 2, 3
MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_MISALIGNED, MLA_ERR_CUDA = range(5)
MLA_ERRBIT_SLOT_OOB, MLA_ERRBIT_BLOCK_OOB, MLA_ERRBIT_POS_OOB, MLA_ERRBIT_MISALIGNED = 1, 2, 4, 8
MLA_ERRBIT_TIMEOUT = 16

_TORCH_DTYPE = {MLA_BF16: torch.bfloat16, MLA_FP8_E4M3: torch.float8_e4m3fn,
                MLA_FP8_E5M2: torch.float8_e5m2, MLA_FP16: torch.float16}


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[mla status {status}] {message}")
        self.status = status


class KvPack(ctypes.Structure):
    _fields_ = [("k_nope", ctypes.c_void_p), ("kn_token_stride", ctypes.c_int64),
                ("kn_head_stride", ctypes.c_int64), ("v", ctypes.c_void_p),
                ("v_token_stride", ctypes.c_int64), ("v_head_stride", ctypes.c_int64),
                ("in_dtype", ctypes.c_int), ("k_pe", ctypes.c_void_p),
                ("kpe_token_stride", ctypes.c_int64), ("kpe_dtype", ctypes.c_int),
                ("num_tokens", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("nope_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("v_dim", ctypes.c_int32), ("key_out", ctypes.c_void_p),
                ("v_out", ctypes.c_void_p), ("out_dtype", ctypes.c_int),
                ("out_scale", ctypes.c_void_p)]


class ContextGather(ctypes.Structure):
    _fields_ = [("kv_cache", ctypes.c_void_p), ("cache_dtype", ctypes.c_int),
                ("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("block_stride", ctypes.c_int64), ("entry_stride", ctypes.c_int64),
                ("entry_dim", ctypes.c_int32), ("block_table", ctypes.c_void_p),
                ("block_table_stride", ctypes.c_int64), ("cu_chunk_lens", ctypes.c_void_p),
                ("chunk_starts", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
                ("num_tokens", ctypes.c_int32), ("out", ctypes.c_void_p),
                ("out_row_stride", ctypes.c_int64), ("out_dtype", ctypes.c_int)]


class NormRope(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_void_p), ("gamma_layer_stride", ctypes.c_int64),
                ("eps", ctypes.c_float), ("positions", ctypes.c_void_p),
                ("cos_sin_cache", ctypes.c_void_p), ("max_position", ctypes.c_int64)]


_lib = None

# C signatures of every entry point declared in include/mla_cache.h
_i32, _i64, _u32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p
SIGNATURES = {
    "mla_dtype_from_string": (ctypes.c_int, [ctypes.c_char_p]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_version": (ctypes.c_char_p, []),
    "mla_set_pdl": (ctypes.c_int, [ctypes.c_int]),
    "mla_set_bulk_copy": (ctypes.c_int, [ctypes.c_int]),
    "mla_set_pointer_checks": (ctypes.c_int, [ctypes.c_int]),
    "mla_set_gather_early_tables": (ctypes.c_int, [ctypes.c_int]),
    "mla_set_insert_early_tables": (ctypes.c_int, [ctypes.c_int]),
    "mla_test_insert_timeout": (ctypes.c_int, [ctypes.c_uint64, _i64]),
    "mla_cache_insert_grouped": (ctypes.c_int, [
        _vp, _i64, _i64, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp, _i64, _vp, _vp,
        ctypes.c_int, _i64, _i32, _i64, _i64, ctypes.POINTER(NormRope), _vp, _vp]),
    "mla_context_gather": (ctypes.c_int, [
        _vp, ctypes.c_int, _i64, _i32, _i64, _i64, _i32, _vp, _i64, _vp, _vp, _i32, _i32, _vp,
        _i64, ctypes.c_int, _vp, _vp]),
    "mla_context_kv_pack": (ctypes.c_int, [
        _vp, _i64, _i64, _vp, _i64, _i64, ctypes.c_int, _vp, _i64, ctypes.c_int, _i32, _i32, _i32,
        _i32, _i32, _vp, _vp, ctypes.c_int, _vp, _vp, _vp]),
    "mla_context_gather_scaled": (ctypes.c_int, [
        _vp, ctypes.c_int, _i64, _i32, _i64, _i64, _i32, _vp, _i64, _vp, _vp, _i32, _i32, _vp,
        _i64, _vp, _vp, _vp]),
    "mla_context_kv_pack_paged": (ctypes.c_int, [
        _vp, _i64, _i64, _vp, _i64, _i64, ctypes.c_int, _vp, ctypes.c_int, _i64, _i32, _i64, _i64,
        _i64, _vp,
        _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, ctypes.c_int, _vp, _vp,
        _vp]),
    "mla_norm_rope_grouped": (ctypes.c_int, [
        _vp, _i64, _i64, _vp, _i64, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(NormRope), _vp,
        _i64, _i64, _vp, _i64, _i64, _vp, _vp]),
    "mla_rope_cos_sin_cache": (ctypes.c_int, [_vp, _i64, _i32, ctypes.c_double, _vp]),
    "mla_context_kv_pack_gather": (ctypes.c_int, [ctypes.POINTER(KvPack),
                                                  ctypes.POINTER(ContextGather), _vp, _vp]),
}


def lib() -> ctypes.CDLL:
    """Load libmla_cache.so (built in-tree by pack_mla_cache_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libmla_cache.so is not built ({LIB_PATH} missing): run "
                "pack_mla_cache_gb300.build.build() first; there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != MLA_OK:
        raise MlaError(status, lib().mla_last_error().decode())


def dtype_code(d) -> int:
    if isinstance(d, int):
        return d
    if isinstance(d, torch.dtype):
        for k, v in _TORCH_DTYPE.items():
            if v == d:
                return k
        raise ValueError(f"unsupported dtype {d}")
    code = lib().mla_dtype_from_string(str(d).encode())
    if code < 0:
        raise MlaError(MLA_ERR_INVALID_ARG, f"unknown kv cache dtype string {d!r}")
    return code


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def mla_dtype_from_string(s: str) -> int:
    return lib().mla_dtype_from_string(s.encode())


def mla_last_error() -> str:
    return lib().mla_last_error().decode()


def mla_version() -> str:
    return lib().mla_version().decode()


def mla_set_pdl(enable: bool) -> bool:
    return bool(lib().mla_set_pdl(1 if enable else 0))


def mla_set_bulk_copy(mode: int) -> int:
    """0 never, 1 large calls (default), 2 every call whose layout qualifies;
    returns the previous mode."""
    return int(lib().mla_set_bulk_copy(int(mode)))


def mla_set_pointer_checks(enable: bool) -> bool:
    """Switch the per-call device-pointer checks on (default) or off; returns
    the previous setting."""
    return bool(lib().mla_set_pointer_checks(1 if enable else 0))


def mla_set_gather_early_tables(enable: bool) -> bool:
    """Let the context gathers read their tables before the programmatic
    launch wait (the tables must be complete before each call is enqueued);
    returns the previous setting."""
    return bool(lib().mla_set_gather_early_tables(1 if enable else 0))


def mla_set_insert_early_tables(enable: bool) -> bool:
    """Let the grouped insert read kv_cache_ptrs and kv_scales before the
    programmatic launch wait (both must be complete before each call is
    enqueued); returns the previous setting."""
    return bool(lib().mla_set_insert_early_tables(1 if enable else 0))


def mla_test_insert_timeout(wait_limit_ns: int = 0, skip_item: int = -1) -> None:
    """Testing hook of the insert's bulk-copy pipeline (see the C header);
    ``mla_test_insert_timeout()`` restores the defaults."""
    lib().mla_test_insert_timeout(int(wait_limit_ns), int(skip_item))


def mla_cache_insert_grouped(kv_c, k_pe, slot_mapping, kv_cache_ptrs, kv_scales, cache_dtype,
                             num_blocks, block_size, block_stride, entry_stride, *,
                             slot_layer_stride=None, gamma=None, eps=1e-6, positions=None,
                             cos_sin_cache=None, err_word=None, stream=None):
    """kv_c [L, T, R] and k_pe [L, T, P] bf16 views (any strides, unit last
    stride); slot_mapping int64 [L, T] or [T] (shared); kv_cache_ptrs int64 [L];
    kv_scales fp32 [L] or None."""
    L, T, R = kv_c.shape
    P = k_pe.shape[2]
    if slot_layer_stride is None:
        slot_layer_stride = 0 if slot_mapping.dim() == 1 else slot_mapping.stride(0)
    nr = None
    if gamma is not None or positions is not None:
        nr = NormRope(_ptr(gamma), 0 if gamma is None else gamma.stride(0), float(eps),
                      _ptr(positions), _ptr(cos_sin_cache),
                      0 if cos_sin_cache is None else cos_sin_cache.shape[0])
    _check(lib().mla_cache_insert_grouped(
        _ptr(kv_c), kv_c.stride(1), kv_c.stride(0), _ptr(k_pe), k_pe.stride(1), k_pe.stride(0),
        T, L, R, P, _ptr(slot_mapping), slot_layer_stride, _ptr(kv_cache_ptrs), _ptr(kv_scales),
        dtype_code(cache_dtype), num_blocks, block_size, block_stride, entry_stride,
        ctypes.byref(nr) if nr is not None else None, _ptr(err_word), _stream(stream)))


def mla_norm_rope_grouped(kv_c, k_pe, kv_c_out, k_pe_out, *, gamma=None, eps=1e-6,
                          positions=None, cos_sin_cache=None, err_word=None, stream=None):
    """Every tensor is a bf16 view indexed [token, layer, i] (any strides, unit
    last stride): kv_c / kv_c_out [T, L, 512], k_pe / k_pe_out [T, L, 64].  For
    layer-major outputs pass e.g. ``out.transpose(0, 1)`` of an [L, T, .] tensor."""
    T, L, R = kv_c.shape
    P = k_pe.shape[2]
    nr = None
    if gamma is not None or positions is not None:
        nr = NormRope(_ptr(gamma), 0 if gamma is None else gamma.stride(0), float(eps),
                      _ptr(positions), _ptr(cos_sin_cache),
                      0 if cos_sin_cache is None else cos_sin_cache.shape[0])
    _check(lib().mla_norm_rope_grouped(
        _ptr(kv_c), kv_c.stride(0), kv_c.stride(1), _ptr(k_pe), k_pe.stride(0), k_pe.stride(1),
        T, L, R, P, ctypes.byref(nr) if nr is not None else None, _ptr(kv_c_out),
        kv_c_out.stride(0), kv_c_out.stride(1), _ptr(k_pe_out), k_pe_out.stride(0),
        k_pe_out.stride(1), _ptr(err_word), _stream(stream)))


def mla_context_gather(kv_cache, cache_dtype, num_blocks, block_size, block_stride,
                       entry_stride, entry_dim, block_table, cu_chunk_lens, chunk_starts, out,
                       out_dtype, *, num_tokens=None, err_word=None, stream=None):
    """kv_cache: the cache base (any tensor over its bytes); block_table int32
    [S, W]; out [num_tokens, >= entry_dim] with unit last stride."""
    S = chunk_starts.shape[0]
    n = out.shape[0] if num_tokens is None else num_tokens
    _check(lib().mla_context_gather(
        _ptr(kv_cache), dtype_code(cache_dtype), num_blocks, block_size, block_stride,
        entry_stride, entry_dim, _ptr(block_table), _bt_stride(block_table), _ptr(cu_chunk_lens),
        _ptr(chunk_starts), S, n, _ptr(out), out.stride(0), dtype_code(out_dtype),
        _ptr(err_word), _stream(stream)))


def _bt_stride(block_table):
    # row width of the table: its row stride (a one-row table's stride is not
    # meaningful, so its width is used)
    return block_table.stride(0) if block_table.size(0) > 1 else block_table.size(1)


def mla_context_gather_scaled(kv_cache, cache_dtype, num_blocks, block_size, block_stride,
                              entry_stride, entry_dim, block_table, cu_chunk_lens, chunk_starts,
                              out, k_scale, *, num_tokens=None, err_word=None, stream=None):
    """The gather with the fp8 -> bf16 widening times ``k_scale`` (device fp32
    scalar tensor); out is bf16 [num_tokens, >= entry_dim]."""
    S = chunk_starts.shape[0]
    n = out.shape[0] if num_tokens is None else num_tokens
    _check(lib().mla_context_gather_scaled(
        _ptr(kv_cache), dtype_code(cache_dtype), num_blocks, block_size, block_stride,
        entry_stride, entry_dim, _ptr(block_table), _bt_stride(block_table),
        _ptr(cu_chunk_lens), _ptr(chunk_starts), S, n, _ptr(out), out.stride(0), _ptr(k_scale),
        _ptr(err_word), _stream(stream)))


def mla_context_kv_pack_paged(k_nope, v, kv_cache, cache_dtype, num_blocks, block_size,
                              block_stride, entry_stride, block_table, cu_chunk_lens,
                              chunk_starts, key_out, v_out, out_dtype, *, rope_offset=512,
                              rope_dim=64, out_scale=None, in_dtype=None, err_word=None,
                              stream=None):
    """The pack with each token's k_pe read from its paged cache row at
    ``rope_offset``; k_nope / v [T, H, 128] bf16 views (strided)."""
    T, H, N = k_nope.shape
    _check(lib().mla_context_kv_pack_paged(
        _ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(v), v.stride(0), v.stride(1),
        dtype_code(in_dtype if in_dtype is not None else k_nope.dtype), _ptr(kv_cache),
        dtype_code(cache_dtype), num_blocks, block_size, block_stride,
        entry_stride, rope_offset, _ptr(block_table), _bt_stride(block_table),
        _ptr(cu_chunk_lens), _ptr(chunk_starts), chunk_starts.shape[0], T, H, N, rope_dim,
        v.shape[2], _ptr(key_out), _ptr(v_out), dtype_code(out_dtype), _ptr(out_scale),
        _ptr(err_word), _stream(stream)))


def mla_context_kv_pack(k_nope, v, k_pe, key_out, v_out, out_dtype, *, kpe_dtype=None,
                        out_scale=None, in_dtype=None, err_word=None, stream=None):
    """k_nope / v: [T, H, 128] bf16 or fp16 views (strided; their dtype is the
    input type unless ``in_dtype`` is given); k_pe [T, 64] (the input type or
    fp8, strided rows); key_out [T, H, 192] and v_out [T, H, 128] (or None)."""
    T, H, N = k_nope.shape
    kd = dtype_code(kpe_dtype if kpe_dtype is not None else k_pe.dtype)
    _check(lib().mla_context_kv_pack(
        _ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(v), v.stride(0), v.stride(1),
        dtype_code(in_dtype if in_dtype is not None else k_nope.dtype), _ptr(k_pe),
        k_pe.stride(0), kd, T, H, N, k_pe.shape[-1], v.shape[2], _ptr(key_out),
        _ptr(v_out), dtype_code(out_dtype), _ptr(out_scale), _ptr(err_word), _stream(stream)))


def mla_rope_cos_sin_cache(out, base=10000.0, *, stream=None):
    """Fill out (fp32 [max_position, rot_dim]) with the rotary cos/sin table."""
    _check(lib().mla_rope_cos_sin_cache(_ptr(out), out.shape[0], out.shape[1], float(base),
                                        _stream(stream)))


def kv_pack_desc(k_nope, v, k_pe, key_out, v_out, out_dtype, *, kpe_dtype=None, out_scale=None,
                 in_dtype=None) -> KvPack:
    """The arguments of ``mla_context_kv_pack`` as the C struct."""
    T, H, N = k_nope.shape
    return KvPack(_ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(v), v.stride(0),
                  v.stride(1), dtype_code(in_dtype if in_dtype is not None else k_nope.dtype),
                  _ptr(k_pe), k_pe.stride(0),
                  dtype_code(kpe_dtype if kpe_dtype is not None else k_pe.dtype), T, H, N,
                  k_pe.shape[-1], v.shape[2], _ptr(key_out), _ptr(v_out), dtype_code(out_dtype),
                  _ptr(out_scale))


def context_gather_desc(kv_cache, cache_dtype, num_blocks, block_size, block_stride,
                        entry_stride, entry_dim, block_table, cu_chunk_lens, chunk_starts, out,
                        out_dtype, *, num_tokens=None) -> ContextGather:
    """The arguments of ``mla_context_gather`` as the C struct."""
    n = out.shape[0] if num_tokens is None else num_tokens
    return ContextGather(_ptr(kv_cache), dtype_code(cache_dtype), num_blocks, block_size,
                         block_stride, entry_stride, entry_dim, _ptr(block_table),
                         _bt_stride(block_table), _ptr(cu_chunk_lens), _ptr(chunk_starts),
                         chunk_starts.shape[0], n, _ptr(out), out.stride(0),
                         dtype_code(out_dtype))


def mla_context_kv_pack_gather(pack: KvPack, next_gather: ContextGather, *, err_word=None,
                               stream=None):
    """One launch: the pack described by ``pack`` (``kv_pack_desc``) and the
    gather described by ``next_gather`` (``context_gather_desc``); the gather
    must write a workspace the pack does not use."""
    _check(lib().mla_context_kv_pack_gather(ctypes.byref(pack), ctypes.byref(next_gather),
                                            _ptr(err_word), _stream(stream)))
