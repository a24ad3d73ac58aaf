"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no normalisation, rotation, fp8 conversion, gather or
pack), so the CPU oracle and the CUDA path can both be fed from it.  Everything
is generated on the CPU with ``torch.Generator`` (one fixed seed per workload,
tensors drawn in a fixed order) and returned as numpy arrays of raw bits:
bf16 tensors as ``uint16``, fp8 caches as ``uint8``.

Workloads (the shapes of the grouped insert in "PR #55356 [Kimi Perf] Group fp8
mla cache insertion" -- five DSpark draft layers, kv_lora_rank 512, rope dim 64
-- and of the chunked-context pack in "PR #51772 [Attention][MLA] Fuse Kimi-K3
chunked-context K/V packing" -- 16 heads of 128 k_nope + 128 v, chunks of 8192
context tokens):

* ``insert_workload``: kv_c [L, T, 512] and k_pe [L, T, 64] ~ N(0, 1) in bf16,
  distinct random slots (one shared mapping or one per layer, optionally with a
  trailing -1 padding slot), per-layer k_scale ~ U[0.005, 0.02], RMSNorm weight
  ~ N(1, 0.1) in bf16, positions ~ U[0, 32768).
* ``pack_workload``: a paged fp8 e4m3 (or bf16) latent cache holding the
  context in randomly chosen blocks (the block table), filled with N(0, 1)
  values cast by torch, and per chunk a kv_b_proj output [T, 4160] bf16 ~ N(0, 1)
  of which 16 x (128 + 128) columns are used (64 columns of row padding).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

KV_LORA_RANK = 512
PE_DIM = 64
ENTRY = KV_LORA_RANK + PE_DIM
ROPE_BASE = 10000.0
MAX_POSITION = 32768


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _bf16_normal(g, shape, mean=0.0, std=1.0) -> np.ndarray:
    x = torch.randn(shape, generator=g, dtype=torch.float32) * std + mean
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@dataclass
class InsertWorkload:
    num_layers: int
    num_tokens: int
    cache_dtype: int  # 0 bf16, 1 e4m3, 2 e5m2
    num_blocks: int
    block_size: int
    kv_c: np.ndarray  # uint16 [L, T, 512]
    k_pe: np.ndarray  # uint16 [L, T, 64]
    slot_mapping: np.ndarray  # int64 [L, T] (row 0 only used when shared)
    shared_slots: bool
    k_scales: np.ndarray | None  # float32 [L] (None for a bf16 cache)
    gamma: np.ndarray | None  # uint16 [L, 512]
    positions: np.ndarray | None  # int64 [T]
    eps: float = 1e-6
    extras: dict = field(default_factory=dict)

    @property
    def slot_layer_stride(self) -> int:
        return 0 if self.shared_slots else self.num_tokens

    @property
    def elt_size(self) -> int:
        return 2 if self.cache_dtype == 0 else 1

    @property
    def block_stride(self) -> int:  # elements
        return self.block_size * ENTRY

    @property
    def entry_stride(self) -> int:  # elements
        return ENTRY

    def empty_caches(self, fill: int = 0) -> list[np.ndarray]:
        dt = np.uint16 if self.cache_dtype == 0 else np.uint8
        return [np.full(self.num_blocks * self.block_size * ENTRY, fill, dt)
                for _ in range(self.num_layers)]


def insert_workload(num_layers: int, num_tokens: int, cache_dtype: int, num_blocks: int,
                    block_size: int = 64, shared_slots: bool = True, norm: bool = False,
                    rope: bool = False, pad_last: bool = False, seed: int = 0,
                    scale_range=(0.005, 0.02), slot_pool: int | None = None,
                    kv_std: float = 1.0) -> InsertWorkload:
    """Seeded grouped-insert inputs.  Slots are the first T entries of a random
    permutation of ``slot_pool`` (default: every slot of the cache), drawn once
    (shared) or once per layer."""
    g = _gen(seed)
    L, T = num_layers, num_tokens
    kv_c = _bf16_normal(g, (L, T, KV_LORA_RANK), std=kv_std)
    k_pe = _bf16_normal(g, (L, T, PE_DIM), std=kv_std)
    pool = slot_pool if slot_pool is not None else num_blocks * block_size
    assert T <= pool
    rows = 1 if shared_slots else L
    slots = torch.stack([torch.randperm(pool, generator=g)[:T] for _ in range(rows)])
    if shared_slots:
        slots = slots.expand(L, T)
    slots = slots.contiguous().numpy().astype(np.int64)
    if pad_last and T > 0:
        slots[:, -1] = -1
    k_scales = None
    if cache_dtype != 0:
        lo, hi = scale_range
        k_scales = (torch.rand(L, generator=g, dtype=torch.float32) * (hi - lo) + lo).numpy()
    gamma = _bf16_normal(g, (L, KV_LORA_RANK), mean=1.0, std=0.1) if norm else None
    positions = (torch.randint(0, MAX_POSITION, (T,), generator=g, dtype=torch.int64).numpy()
                 if rope else None)
    return InsertWorkload(L, T, cache_dtype, num_blocks, block_size, kv_c, k_pe, slots,
                          shared_slots, k_scales, gamma, positions)


def pages_test_insert_workload(cache_dtype: int, shared_slots: bool, seed: int = 0) -> InsertWorkload:
    """The shape of test_concat_and_cache_mla_grouped ("PR #55356", its test
    snippet): 5 layers, block_size 16, 8 blocks, 42 tokens, k_scale =
    linspace(0.05, 0.25, 5), per-layer random slots with the last one set to -1."""
    wl = insert_workload(5, 42, cache_dtype, num_blocks=8, block_size=16,
                         shared_slots=shared_slots, pad_last=True, seed=seed)
    if cache_dtype != 0:
        wl.k_scales = np.linspace(0.05, 0.25, 5, dtype=np.float32)
    return wl


@dataclass
class PackWorkload:
    num_tokens: int  # context tokens in total
    chunk: int  # tokens per chunk
    num_heads: int
    nope: int
    v_dim: int
    row_stride: int  # kv_b_proj output row stride (elements)
    cache_dtype: int
    num_blocks: int
    block_size: int
    cache: np.ndarray  # flat uint8 (fp8) or uint16 (bf16) [num_blocks * block_size * 576]
    block_table: np.ndarray  # int32 [1, max_blocks]
    kv_b_proj: list  # per chunk uint16 [chunk, row_stride]
    out_scale: float = 0.01

    @property
    def num_chunks(self) -> int:
        return (self.num_tokens + self.chunk - 1) // self.chunk

    def chunk_range(self, c: int) -> tuple[int, int]:
        s = c * self.chunk
        return s, min(self.chunk, self.num_tokens - s)


def pack_workload(num_tokens: int, chunk: int, num_blocks: int, block_size: int = 64,
                  num_heads: int = 16, nope: int = 128, v_dim: int = 128,
                  row_stride: int | None = None, cache_dtype: int = 1, seed: int = 0,
                  distinct_chunks: bool = True) -> PackWorkload:
    """Seeded chunked-context inputs: one sequence of ``num_tokens`` context
    tokens held in ``ceil(num_tokens / block_size)`` random blocks of a paged
    cache, and a kv_b_proj output per chunk (one shared buffer when
    ``distinct_chunks`` is False)."""
    g = _gen(seed)
    nblk_ctx = (num_tokens + block_size - 1) // block_size
    assert nblk_ctx <= num_blocks
    table = torch.randperm(num_blocks, generator=g)[:nblk_ctx].to(torch.int32).numpy()[None, :].copy()
    vals = torch.randn((num_blocks * block_size * ENTRY,), generator=g, dtype=torch.float32)
    if cache_dtype == 0:
        cache = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        fp8 = torch.float8_e4m3fn if cache_dtype == 1 else torch.float8_e5m2
        cache = vals.to(fp8).view(torch.uint8).numpy()
    if row_stride is None:
        row_stride = num_heads * (nope + v_dim) + 64
    nchunks = (num_tokens + chunk - 1) // chunk
    bufs = []
    for c in range(nchunks if distinct_chunks else 1):
        rows = min(chunk, num_tokens - c * chunk) if distinct_chunks else chunk
        bufs.append(_bf16_normal(g, (rows, row_stride)))
    return PackWorkload(num_tokens, chunk, num_heads, nope, v_dim, row_stride, cache_dtype,
                        num_blocks, block_size, np.ascontiguousarray(cache), np.ascontiguousarray(table),
                        bufs)
