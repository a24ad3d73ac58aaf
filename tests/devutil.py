"""Device-side plumbing for the GPU parity tests: numpy <-> torch transfers,
guard-banded cache buffers, and one runner per entry point that calls the
CUDA library through its Python binding (pack_mla_cache_gb300.ops).

Nothing here computes any part of the method; the CUDA path does it all."""
from __future__ import annotations

import numpy as np
import torch

from pack_mla_cache_gb300 import ops
from pack_mla_cache_gb300 import workloads as W

GUARD = 512  # canary bytes on each side of every cache / output buffer
CANARY = 0xA5


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).cpu().numpy()


class Guarded:
    """A device byte buffer with canary bands before and after the payload."""

    def __init__(self, nbytes: int, fill: int = CANARY):
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), fill, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + nbytes]

    def ptr(self) -> int:
        return self.t.data_ptr()

    def guards_intact(self) -> bool:
        g = torch.cat([self.buf[:GUARD], self.buf[GUARD + self.nbytes:]])
        return bool((g == CANARY).all().item())

    def host(self) -> np.ndarray:
        return host_u8(self.t)


def gpu_insert(wl: W.InsertWorkload, *, cos_sin: torch.Tensor | None = None,
               slot_shared_1d: bool = True, fill: int = 0, err: torch.Tensor | None = None,
               kv_c: torch.Tensor | None = None, k_pe: torch.Tensor | None = None,
               caches: list | None = None):
    """Run the grouped insert on the GPU; returns (caches as numpy in the cache
    element type, guard check, list of Guarded)."""
    esz = wl.elt_size
    nbytes = wl.num_blocks * wl.block_size * W.ENTRY * esz
    if caches is None:
        caches = [Guarded(nbytes) for _ in range(wl.num_layers)]
        for c in caches:
            c.t.fill_(fill)
    ptrs = torch.tensor([c.ptr() for c in caches], dtype=torch.int64, device="cuda")
    if kv_c is None:
        kv_c = dev_bf16(wl.kv_c)
    if k_pe is None:
        k_pe = dev_bf16(wl.k_pe)
    if wl.shared_slots and slot_shared_1d:
        slots = dev(np.ascontiguousarray(wl.slot_mapping[0]))
    else:
        slots = dev(wl.slot_mapping)
    scales = dev(wl.k_scales) if wl.k_scales is not None else None
    gamma = dev_bf16(wl.gamma) if wl.gamma is not None else None
    pos = dev(wl.positions) if wl.positions is not None else None
    ops.mla_cache_insert_grouped(kv_c, k_pe, slots, ptrs, scales, wl.cache_dtype, wl.num_blocks,
                                 wl.block_size, wl.block_stride, wl.entry_stride, gamma=gamma,
                                 eps=wl.eps, positions=pos, cos_sin_cache=cos_sin, err_word=err)
    torch.cuda.synchronize()
    out = []
    for c in caches:
        h = c.host()
        out.append(h.view(np.uint16) if esz == 2 else h)
    return out, all(c.guards_intact() for c in caches), caches


def gpu_rope_table(max_position=W.MAX_POSITION, rot_dim=W.PE_DIM, base=W.ROPE_BASE):
    t = torch.empty((max_position, rot_dim), dtype=torch.float32, device="cuda")
    ops.mla_rope_cos_sin_cache(t, base)
    return t
