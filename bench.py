"""Benchmark of the MLA latent-KV data-movement hot path on one GPU per rank.

One step = one pass of the whole path over one batch, the large workload:
  * grouped insert: 65536 tokens x 5 layers, RMSNorm (eps 1e-6) + neox RoPE
    (positions in [0, 32768)), fp8 e4m3 caches of 2048 blocks x 64 x 576, one
    shared slot mapping;
  * chunked-context pack of 131072 context tokens = 16 chunks of 8192: per
    chunk a gather of the latent rows from an fp8 e4m3 paged cache (2048
    blocks, random block table) into a workspace, then the K/V pack of that
    chunk's kv_b_proj output [8192, 16 x (128 + 128)] bf16 (row stride 4160)
    into a contiguous fp8 e4m3 key [8192, 16, 192] and V [8192, 16, 128]
    (scale 0.01).  The chunk loop is software-pipelined: the gather of chunk 0,
    then per chunk c one launch that packs c and gathers c + 1 into the other
    of two workspaces (mla_context_kv_pack_gather); the unfused loop (a gather
    and a pack launch per chunk) is timed beside it.
The step's inputs (insert 377 MB, kv_b_proj 1.09 GB, cache 75 MB) are larger
than L2, so no flush is needed between steps.  value = algorithmic bytes of a
step / device time of a step (CUDA-graph replay, CUDA events on the launching
stream).  Algorithmic bytes read every input once and write every output once:
insert 1728 B per (token, layer) + 272 B per token; gather 1152 B per token;
pack 13376 B per token.

``--impl reference`` times the CPU oracle (plain C, its independent rows split
over the host's cores) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L_LAYERS, T_INSERT, NB_INSERT = 5, 65536, 2048
T_CTX, CHUNK, NB_CTX, HEADS, ROW_STRIDE = 131072, 8192, 2048, 16, 4160
ENTRY, BS = 576, 64
OUT_SCALE = 0.01
FALLBACK_HBM_GBS = 6800.0

B_INSERT_ROW = 1152 + 576           # per (token, layer)
B_INSERT_TOK = 8 + 8 + 256          # slot, position, cos/sin per token
B_GATHER_TOK = 576 + 576            # fp8 row read + raw write
B_PACK_TOK = HEADS * 256 * 2 + 64 + HEADS * 192 + HEADS * 128  # 13376
B_PACK_TOK_BF16 = HEADS * 256 * 2 + 128 + 2 * (HEADS * 192 + HEADS * 128)  # 18560 (bf16 k_pe)

METRIC = "grouped MLA insert & context K/V pack: HBM GB/s (% of peak), tokens·layers/s"
WORKLOAD = ("grouped 5-layer fp8 e4m3 insert of 65536 tokens with RMSNorm+RoPE into caches of "
            "2048 blocks x 64 x 576 + context pack of 131072 tokens (16 chunks of 8192, 16 heads, "
            "kv_b_proj row stride 4160) gathered from an fp8 e4m3 paged cache, fp8 e4m3 out "
            "(scale 0.01)")


def insert_bytes(T, L):
    return T * (L * B_INSERT_ROW + B_INSERT_TOK)


def step_bytes():
    return (insert_bytes(T_INSERT, L_LAYERS) + T_CTX * B_GATHER_TOK + (T_CTX // BS) * 4
            + T_CTX * B_PACK_TOK)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if the
    summary was taken on the kernel source as it is now (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel)
        if not d:
            return None
        h = hashlib.sha1()
        for f in d["sources"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != d["sha1"]:
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = str(gpu_index)
        try:
            import torch
            u = str(torch.cuda.get_device_properties(gpu_index).uuid)
            self.idx = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.idx, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.05)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        except Exception:
            pass
        finally:
            try:
                os.remove(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- GPU workload
class Workload:
    """Device-resident inputs/outputs of one step, built from the seeded
    generators."""

    def __init__(self, seed: int):
        import torch
        from pack_mla_cache_gb300 import ops
        from pack_mla_cache_gb300 import workloads as W

        self.ops = ops
        dev = torch.device("cuda")
        wl = W.insert_workload(L_LAYERS, T_INSERT, 1, num_blocks=NB_INSERT, block_size=BS,
                               norm=True, rope=True, seed=seed, slot_pool=NB_INSERT * BS)
        self.wl = wl

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

        self.h_kv_c = bf16(wl.kv_c)
        self.h_k_pe = bf16(wl.k_pe)
        self.kv_c = self.h_kv_c.to(dev)
        self.k_pe = self.h_k_pe.to(dev)
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.slot_mapping[0])).to(dev)
        self.positions = torch.from_numpy(wl.positions).to(dev)
        self.scales = torch.from_numpy(wl.k_scales).to(dev)
        self.gamma = bf16(wl.gamma).to(dev)
        self.caches = [torch.zeros(NB_INSERT * BS * ENTRY, dtype=torch.uint8, device=dev)
                       for _ in range(L_LAYERS)]
        self.cache_ptrs = torch.tensor([c.data_ptr() for c in self.caches], dtype=torch.int64,
                                       device=dev)
        self.cos_sin = torch.empty((W.MAX_POSITION, W.PE_DIM), dtype=torch.float32, device=dev)
        ops.mla_rope_cos_sin_cache(self.cos_sin, W.ROPE_BASE)

        pw = W.pack_workload(T_CTX, CHUNK, num_blocks=NB_CTX, block_size=BS, num_heads=HEADS,
                             row_stride=ROW_STRIDE, seed=seed + 1)
        self.pw = pw
        self.ctx_cache = torch.from_numpy(pw.cache).to(dev)
        self.block_table = torch.from_numpy(pw.block_table).to(dev)
        self.cu = torch.tensor([0, CHUNK], dtype=torch.int32, device=dev)
        self.starts = [torch.tensor([c * CHUNK], dtype=torch.int32, device=dev)
                       for c in range(pw.num_chunks)]
        self.h_kvb = [bf16(b) for b in pw.kv_b_proj]
        # one contiguous kv_b_proj output, key and V for the whole context; the
        # chunks are views of them (the one-launch pack reads them whole)
        self.kvb_all = torch.cat([b.to(dev) for b in self.h_kvb])
        self.kvb = [self.kvb_all[c * CHUNK:(c + 1) * CHUNK] for c in range(pw.num_chunks)]
        self.ws = torch.empty((CHUNK, ENTRY), dtype=torch.uint8, device=dev)
        self.key_all = torch.empty((T_CTX, HEADS, 192), dtype=torch.uint8, device=dev)
        self.vout_all = torch.empty((T_CTX, HEADS, 128), dtype=torch.uint8, device=dev)
        self.key = [self.key_all[c * CHUNK:(c + 1) * CHUNK] for c in range(pw.num_chunks)]
        self.vout = [self.vout_all[c * CHUNK:(c + 1) * CHUNK] for c in range(pw.num_chunks)]
        # the gather tables are uploaded once, before any step: the gathers may
        # read them before their programmatic-launch wait
        ops.mla_set_gather_early_tables(True)
        self.out_scale = torch.tensor([OUT_SCALE], dtype=torch.float32, device=dev)
        self.err = torch.zeros(2, dtype=torch.int32, device=dev)

    # one kernel each ----------------------------------------------------
    def insert(self):
        self.ops.mla_cache_insert_grouped(
            self.kv_c, self.k_pe, self.slots, self.cache_ptrs, self.scales, 1, NB_INSERT, BS,
            BS * ENTRY, ENTRY, gamma=self.gamma, eps=self.wl.eps, positions=self.positions,
            cos_sin_cache=self.cos_sin, err_word=self.err[0:1])

    def gather(self, c):
        self.ops.mla_context_gather(self.ctx_cache, 1, NB_CTX, BS, BS * ENTRY, ENTRY, ENTRY,
                                    self.block_table, self.cu, self.starts[c], self.ws, 1,
                                    err_word=self.err[1:2])

    def pack(self, c):
        heads = self.kvb[c][:, :HEADS * 256].view(CHUNK, HEADS, 256)
        self.ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:], self.ws[:, 512:],
                                     self.key[c], self.vout[c], 1, kpe_dtype=1,
                                     out_scale=self.out_scale)

    def step(self):
        self.insert()
        for c in range(self.pw.num_chunks):
            self.gather(c)
            self.pack(c)

    # the chunk loop software-pipelined: chunk c's pack and chunk c + 1's gather
    # in one launch, the gathers alternating between two workspaces
    def pipelined_setup(self):
        import torch
        ops = self.ops
        if getattr(self, "fused_descs", None):
            return
        self.ws_pair = [self.ws, torch.empty_like(self.ws)]
        n = self.pw.num_chunks
        cu_empty = torch.tensor([0, 0], dtype=torch.int32, device=self.ws.device)
        self.fused_descs = []
        for c in range(n):
            heads = self.kvb[c][:, :HEADS * 256].view(CHUNK, HEADS, 256)
            pk = ops.kv_pack_desc(heads[:, :, :128], heads[:, :, 128:], self.ws_pair[c % 2][:, 512:],
                                  self.key[c], self.vout[c], 1, kpe_dtype=1,
                                  out_scale=self.out_scale)
            nxt = c + 1 < n
            gd = ops.context_gather_desc(self.ctx_cache, 1, NB_CTX, BS, BS * ENTRY, ENTRY, ENTRY,
                                         self.block_table, self.cu if nxt else cu_empty,
                                         self.starts[c + 1 if nxt else c],
                                         self.ws_pair[(c + 1) % 2], 1,
                                         num_tokens=CHUNK if nxt else 0)
            self.fused_descs.append((pk, gd))
        self._keep = cu_empty

    def pack_gather(self, c):
        pk, gd = self.fused_descs[c]
        self.ops.mla_context_kv_pack_gather(pk, gd, err_word=self.err[1:2])

    def step_pipelined(self):
        self.insert()
        self.ops.mla_context_gather(self.ctx_cache, 1, NB_CTX, BS, BS * ENTRY, ENTRY, ENTRY,
                                    self.block_table, self.cu, self.starts[0], self.ws_pair[0], 1,
                                    err_word=self.err[1:2])
        for c in range(self.pw.num_chunks):
            self.pack_gather(c)

    # the whole context in one launch each (the grid-capped grid-stride loop)
    def one_launch_setup(self):
        import torch
        dev = self.kvb_all.device
        self.ws_all = torch.empty((T_CTX, ENTRY), dtype=torch.uint8, device=dev)
        self.ws_all16 = torch.empty((T_CTX, ENTRY), dtype=torch.bfloat16, device=dev)
        cu = torch.tensor([0, T_CTX], dtype=torch.int32, device=dev)
        st = torch.tensor([0], dtype=torch.int32, device=dev)
        for ws, odt in ((self.ws_all, 1), (self.ws_all16, 0)):
            self.ops.mla_context_gather(self.ctx_cache, 1, NB_CTX, BS, BS * ENTRY, ENTRY, ENTRY,
                                        self.block_table, cu, st, ws, odt)
        self.key16 = torch.empty((T_CTX, HEADS, 192), dtype=torch.bfloat16, device=dev)
        self.v16 = torch.empty((T_CTX, HEADS, 128), dtype=torch.bfloat16, device=dev)

    def pack_one_launch(self, bf16_out=False):
        heads = self.kvb_all[:, :HEADS * 256].view(T_CTX, HEADS, 256)
        if bf16_out:
            self.ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:],
                                         self.ws_all16[:, 512:], self.key16, self.v16, 0,
                                         kpe_dtype=0)
        else:
            self.ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:],
                                         self.ws_all[:, 512:], self.key_all, self.vout_all, 1,
                                         kpe_dtype=1, out_scale=self.out_scale)

    launches_per_step = 1 + 2 * (T_CTX // CHUNK)
    launches_per_step_pipelined = 2 + T_CTX // CHUNK


def graph_of(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm (occupancy caches, lazy module loading) outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, stream, reps):
    """ms per replay; replay() launches on the current stream, so the replays
    and both events run on `stream`."""
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        s.record(stream)
        for _ in range(reps):
            g.replay()
        e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / reps


# ----------------------------------------------------------- CPU oracle leg
class OracleSample:
    """A bounded sample of the step for the CPU oracle (as it stands): an
    insert of `tokens_insert` tokens x 5 layers and a gather + fp8 pack of
    `tokens_pack` context tokens, from the same seeded generators."""

    def __init__(self, seed: int, tokens_insert: int, tokens_pack: int):
        import oracle as orc
        from pack_mla_cache_gb300 import workloads as W

        orc.build()
        self.orc = orc
        self.ti, self.tp = tokens_insert, tokens_pack
        self.wl = W.insert_workload(L_LAYERS, tokens_insert, 1, num_blocks=NB_INSERT,
                                    block_size=BS, norm=True, rope=True, seed=seed,
                                    slot_pool=NB_INSERT * BS)
        self.pw = W.pack_workload(tokens_pack, tokens_pack,
                                  num_blocks=max(1, -(-tokens_pack // BS)) + 1, block_size=BS,
                                  num_heads=HEADS, row_stride=ROW_STRIDE, seed=seed + 1)
        self.caches = self.wl.empty_caches()
        self.table = orc.rope_cos_sin_cache(W.MAX_POSITION, W.PE_DIM, W.ROPE_BASE)
        self.ws = np.zeros((tokens_pack, ENTRY), np.uint8)
        self.slots = np.ascontiguousarray(self.wl.slot_mapping[0])
        self.nbytes = (insert_bytes(tokens_insert, L_LAYERS) + tokens_pack * B_GATHER_TOK
                       + tokens_pack * B_PACK_TOK)

    def run(self, threads: int = 1) -> float:
        """Seconds for one pass; threads > 1 splits each function's independent
        rows over that many host threads (the unchanged oracle per range, a
        byte-identical result)."""
        orc, wl, pw, tp = self.orc, self.wl, self.pw, self.tp
        kvb = pw.kv_b_proj[0]
        cu, st = np.array([0, tp], np.int32), np.array([0], np.int32)
        t0 = time.perf_counter()
        if threads <= 1:
            orc.insert_grouped(wl.kv_c, wl.k_pe, self.slots, 0, self.caches, wl.k_scales, 1,
                               NB_INSERT, BS, BS * ENTRY, ENTRY, wl.gamma, wl.eps, wl.positions,
                               self.table)
            orc.context_gather(pw.cache, 1, pw.num_blocks, BS, BS * ENTRY, ENTRY, ENTRY,
                               pw.block_table, cu, st, self.ws, 1)
            orc.context_kv_pack(kvb, ROW_STRIDE, 256, kvb[:, 128:], ROW_STRIDE, 256,
                                self.ws[:, 512:], ENTRY, 1, tp, HEADS, 128, 64, 128, 1, OUT_SCALE)
        else:
            orc.insert_grouped_split(threads, wl.kv_c, wl.k_pe, self.slots, 0, self.caches,
                                     wl.k_scales, 1, NB_INSERT, BS, BS * ENTRY, ENTRY, wl.gamma,
                                     wl.eps, wl.positions, self.table)
            orc.context_gather_split(threads, pw.cache, 1, pw.num_blocks, BS, BS * ENTRY, ENTRY,
                                     ENTRY, pw.block_table, cu, st, self.ws, 1)
            orc.context_kv_pack_split(threads, kvb, ROW_STRIDE, 256, kvb[:, 128:], ROW_STRIDE,
                                      256, self.ws[:, 512:], ENTRY, 1, tp, HEADS, 128, 64, 128, 1,
                                      OUT_SCALE)
        return time.perf_counter() - t0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle

    cores = oracle.host_threads()
    # one step = this bounded sample of the workload (~1/32 of the insert and
    # the pack), its rows split over every host core
    ti, tp = 2048, 4096
    smp = OracleSample(0, ti, tp)
    for _ in range(args.warmup):
        smp.run(cores)
    times, nbytes = [], smp.nbytes
    for _ in range(args.steps):
        times.append(smp.run(cores))
    tot = sum(times)
    value = nbytes * len(times) / tot / 1e9
    sample = (f"per step: insert of {ti} tokens x 5 layers (RMSNorm+RoPE, e4m3) + gather and "
              f"fp8 pack of {tp} context tokens (16 heads), from the same generators; the C "
              f"oracle's independent rows split over {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / len(times) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp8 e4m3 out, f64 math",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample,
                                            "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- multi-rank
def max_over_ranks(value: float, world: int) -> float:
    """The largest of every rank's value (the slowest rank's time); the
    identity on one rank.  Works with any process-group backend: the tensor
    lives on the GPU for NCCL and on the CPU otherwise."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, world: int, ms_max: float) -> float:
    """Whole-job GB/s: every rank moves its own shard (no exchange), the job
    takes as long as its slowest rank."""
    return bytes_per_rank_step * world / (ms_max * 1e-3) / 1e9


# ----------------------------------------------------------------- main arm
def run(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()

    w = Workload(seed=1000 + rank)
    w.pipelined_setup()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            w.step_pipelined()
    torch.cuda.synchronize()
    step_graph = graph_of(w.step_pipelined, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: K steps, device time on the launching stream
    with ClockSampler(local) as clk:
        # keep the GPU busy with untimed steps while the sampler starts, so its
        # samples fall under load (the K timed steps alone last a few ms)
        t_load = time.perf_counter() + 0.8
        while time.perf_counter() < t_load:
            with torch.cuda.stream(stream):
                for _ in range(32):
                    step_graph.replay()
            stream.synchronize()
        barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                step_graph.replay()
            end.record(stream)
        end.synchronize()
        barrier()
        ms = start.elapsed_time(end) / args.steps
        # per-kernel average launch durations, same launch configurations
        nch = w.pw.num_chunks
        g_ins = graph_of(w.insert, stream)
        g_gat = graph_of(lambda: [w.gather(c) for c in range(nch)], stream)
        g_pack = graph_of(lambda: [w.pack(c) for c in range(nch)], stream)
        g_pg = graph_of(lambda: [w.pack_gather(c) for c in range(nch)], stream)
        g_plain = graph_of(w.step, stream)
        reps = max(3, args.steps)
        ms_insert = time_graph(g_ins, stream, reps)
        ms_gather = time_graph(g_gat, stream, reps) / nch
        ms_pack = time_graph(g_pack, stream, reps) / nch
        ms_pg = time_graph(g_pg, stream, reps) / nch
        ms_plain = time_graph(g_plain, stream, reps)
        # the whole 131072-token context packed by ONE launch (fp8 and bf16 out)
        w.one_launch_setup()
        g_one = graph_of(lambda: w.pack_one_launch(False), stream)
        g_one16 = graph_of(lambda: w.pack_one_launch(True), stream)
        ms_one = time_graph(g_one, stream, max(3, args.steps // 4))
        ms_one16 = time_graph(g_one16, stream, max(3, args.steps // 4))
    clocks = clk.summary()

    ms = max_over_ranks(ms, world)
    sbytes = step_bytes()
    value = job_throughput(sbytes, world, ms)
    errs = w.err.cpu().tolist()
    assert errs == [0, 0], f"kernels reported skipped rows: {errs}"

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(w, stream, max(2, min(args.steps, 5)))
    e2e["ms"] = max_over_ranks(e2e["ms"], world)

    if rank != 0:
        dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peak()
    b_pack_launch = CHUNK * B_PACK_TOK
    b_ins_launch = insert_bytes(T_INSERT, L_LAYERS)
    b_gat_launch = CHUNK * B_GATHER_TOK + (CHUNK // BS) * 4
    nch = w.pw.num_chunks
    # the fused launches of a step: every one packs a chunk, all but the last
    # also gather the next chunk (average bytes per launch)
    b_pg_launch = b_pack_launch + b_gat_launch * (nch - 1) / nch
    ach = b_pg_launch / (ms_pg * 1e-3) / 1e9

    def kline(b, m):
        a = b / (m * 1e-3) / 1e9
        return {"us_per_launch": m * 1e3, "bytes_per_launch": b, "achieved_gbs": a,
                "frac": a / peak}

    cpu = None
    if world == 1:
        import oracle

        cores = oracle.host_threads()
        smp = OracleSample(0, 8192, 32768)
        what = ("insert of 8192 tokens x 5 layers (RMSNorm+RoPE, e4m3) + gather and fp8 pack of "
                "32768 context tokens (16 heads)")
        reps1 = 2  # about 6 s of CPU work on one host core
        dt1 = sum(smp.run(1) for _ in range(reps1))
        repsn = 8
        smp.run(cores)
        dtn = sum(smp.run(cores) for _ in range(repsn))
        v1, vn = reps1 * smp.nbytes / dt1 / 1e9, repsn * smp.nbytes / dtn / 1e9
        cpu = {"value": vn, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{repsn} x ({what}), the C oracle's independent rows split over "
                         f"{cores} host threads (byte-identical output), {dtn:.1f} s",
               "single_core": {"value": v1, "unit": "GB/s", "cores": 1,
                               "sample": f"{reps1} x (the same), single-threaded, {dt1:.1f} s"}}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp8 e4m3 out, fp32 math", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (1.55 GB read per step), no flush",
                   "timing": "CUDA-graph replay of whole steps, CUDA events on the stream",
                   "step": ("insert; gather of chunk 0; then per chunk c one launch packing c "
                            "and gathering c + 1 (two workspaces)"),
                   "ms_per_step_unfused": ms_plain,
                   "step_bytes": sbytes, "frac_of_peak": value / world / peak,
                   "peak_gbs": peak, "peak_kind": peak_kind,
                   "tokens_layers_per_s_insert": T_INSERT * L_LAYERS * world / (ms * 1e-3),
                   "context_tokens_per_s": T_CTX * world / (ms * 1e-3)},
        "roofline": {"bound": "hbm", "kernel": "pack_gather_kernel<e4m3,e4m3,bf16>",
                     "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "traffic": profile_traffic("pack_gather_fp8_h16"),
                     "traffic_basis": ("ncu, one launch with its gather: dram__bytes_read.sum + "
                                       "lts__t_sectors_srcunit_tex_op_write.sum x 32 (every stored "
                                       "byte reaches DRAM; dram__bytes_write.sum sees only the "
                                       "write-backs inside the launch)")},
        "kernels": {"insert": kline(b_ins_launch, ms_insert),
                    "pack_gather": kline(b_pg_launch, ms_pg),
                    "gather": kline(b_gat_launch, ms_gather),
                    "pack": kline(b_pack_launch, ms_pack),
                    "pack_one_launch_131072": kline(T_CTX * B_PACK_TOK, ms_one),
                    "pack_one_launch_131072_bf16": kline(T_CTX * B_PACK_TOK_BF16, ms_one16)},
        "cpu_baseline": cpu,
        "e2e": {"value": job_throughput(sbytes, world, e2e["ms"]), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e["ms"], "runs_ms": [round(r, 3) for r in e2e["reps_ms"]],
                "bound": "pinned H2D over the host link (about 210 GB/s measured host to GB300)"},
        "gpu_launches": Workload.launches_per_step_pipelined * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(w, stream, steps):
    """Whole step through the public API from pinned host buffers: H2D of the
    step's inputs, the 18 calls, D2H of the packed key/V; wall time between
    synchronisations.  Copies and kernels overlap as a serving loop would run
    them: inputs stream in on one stream, the kernels run on the compute stream
    as each chunk's input lands (event waits), results stream out on a third;
    the chunks go first and the insert last, so its 377 MB of input arrive
    while the chunks compute."""
    import torch
    h_kv_c = w.h_kv_c.pin_memory()
    h_k_pe = w.h_k_pe.pin_memory()
    h_kvb = [b.pin_memory() for b in w.h_kvb]
    h_key = [torch.empty_like(k, device="cpu").pin_memory() for k in w.key]
    h_v = [torch.empty_like(v, device="cpu").pin_memory() for v in w.vout]
    h2d = h_kv_c.numel() * 2 + h_k_pe.numel() * 2 + sum(b.numel() * 2 for b in h_kvb)
    d2h = sum(k.numel() for k in h_key) + sum(v.numel() for v in h_v)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n = w.pw.num_chunks

    def one():
        ev_in = [torch.cuda.Event() for _ in range(n + 1)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        s_in.wait_stream(stream)  # the previous step's kernels have read their inputs
        with torch.cuda.stream(s_in):
            for c in range(n):
                w.kvb[c].copy_(h_kvb[c], non_blocking=True)
                ev_in[c].record(s_in)
            w.kv_c.copy_(h_kv_c, non_blocking=True)
            w.k_pe.copy_(h_k_pe, non_blocking=True)
            ev_in[n].record(s_in)
        with torch.cuda.stream(stream):
            w.ops.mla_context_gather(w.ctx_cache, 1, NB_CTX, BS, BS * ENTRY, ENTRY, ENTRY,
                                     w.block_table, w.cu, w.starts[0], w.ws_pair[0], 1)
            for c in range(n):
                stream.wait_event(ev_in[c])
                w.pack_gather(c)
                ev_done[c].record(stream)
            stream.wait_event(ev_in[n])
            w.insert()
        with torch.cuda.stream(s_out):
            for c in range(n):
                s_out.wait_event(ev_done[c])
                h_key[c].copy_(w.key[c], non_blocking=True)
                h_v[c].copy_(w.vout[c], non_blocking=True)
        stream.synchronize()
        s_out.synchronize()
        s_in.synchronize()

    one()
    reps = []
    for _ in range(3):  # the median of three timed runs (host-link hiccups)
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        reps.append((time.perf_counter() - t0) / steps * 1e3)
    ms = sorted(reps)[1]
    return {"ms": ms, "h2d": h2d, "d2h": d2h, "reps_ms": reps}


def run_profile_case(name: str, launches: int, tokens: int | None = None,
                     graph: bool = False) -> int:
    """A few launches of ONE kernel on a mid-size case (inputs larger than L2,
    a few hundred MB on the device), for ncu captures:
      insert  32768 tokens x 5 layers, e4m3, RMSNorm+RoPE, 2048-block caches
      insert_raw the same without RMSNorm / RoPE
      insert_plain the insert with the bulk-copy pipeline shape disabled (row per warp)
      gather  262144 context rows from a 4096-block fp8 cache, raw
      gather_scaled  the gather widened to bf16 times a k_scale
      gather_bf16    the gather widened exactly to bf16
      gather_kv_c    the raw gather of the 512 kv_c columns only
      pack    32768 tokens, 16 heads, fp8 e4m3 out, fp8 k_pe
      pack_bf16  the same with bf16 output and a bf16 k_pe
      pack_f16   the fp8 pack of an fp16 kv_b_proj output
      pack_paged the fp8 pack reading k_pe from a 4096-block fp8 cache
      pack_gather the fp8 pack of 8192 tokens and the gather of the next 8192
                 rows into a second workspace, one launch
      norm_rope  65536 tokens x 5 layers of the [T, L, 576] projection, RMSNorm +
                 RoPE into layer-major outputs"""
    import torch
    from pack_mla_cache_gb300 import ops
    from pack_mla_cache_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    if name in ("insert", "insert_raw", "insert_plain"):
        T = tokens or 32768
        raw = name == "insert_raw"
        ops.mla_set_bulk_copy(0 if name == "insert_plain" else 1)
        kv_c = torch.randn((L_LAYERS, T, 512), generator=g, device=dev).to(torch.bfloat16)
        k_pe = torch.randn((L_LAYERS, T, 64), generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(NB_INSERT * BS, generator=g, device=dev)[:T]
        pos = torch.randint(0, W.MAX_POSITION, (T,), generator=g, device=dev)
        gamma = (1 + 0.1 * torch.randn((L_LAYERS, 512), generator=g, device=dev)).to(torch.bfloat16)
        scales = torch.rand(L_LAYERS, generator=g, device=dev) * 0.015 + 0.005
        caches = [torch.zeros(NB_INSERT * BS * ENTRY, dtype=torch.uint8, device=dev)
                  for _ in range(L_LAYERS)]
        ptrs = torch.tensor([c.data_ptr() for c in caches], dtype=torch.int64, device=dev)
        table = torch.empty((W.MAX_POSITION, 64), dtype=torch.float32, device=dev)
        ops.mla_rope_cos_sin_cache(table, W.ROPE_BASE)
        fn = lambda: ops.mla_cache_insert_grouped(kv_c, k_pe, slots, ptrs, scales, 1, NB_INSERT,
                                                  BS, BS * ENTRY, ENTRY,
                                                  gamma=None if raw else gamma, eps=1e-6,
                                                  positions=None if raw else pos,
                                                  cos_sin_cache=None if raw else table)
        nbytes = insert_bytes(T, L_LAYERS)
    elif name in ("gather", "gather_scaled", "gather_bf16", "gather_kv_c"):
        T, nb = tokens or 262144, 4096
        cache = torch.randint(0, 126, (nb * BS * ENTRY,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        table = torch.randperm(nb, generator=g, device=dev).to(torch.int32)[None, :].contiguous()
        cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
        st = torch.tensor([0], dtype=torch.int32, device=dev)
        if name == "gather_scaled":
            out = torch.empty((T, ENTRY), dtype=torch.bfloat16, device=dev)
            ks = torch.tensor([0.0137], dtype=torch.float32, device=dev)
            fn = lambda: ops.mla_context_gather_scaled(cache, 1, nb, BS, BS * ENTRY, ENTRY, ENTRY,
                                                       table, cu, st, out, ks)
            nbytes = T * (ENTRY + 2 * ENTRY) + (T // BS) * 4
        elif name == "gather_bf16":
            out = torch.empty((T, ENTRY), dtype=torch.bfloat16, device=dev)
            fn = lambda: ops.mla_context_gather(cache, 1, nb, BS, BS * ENTRY, ENTRY, ENTRY, table,
                                                cu, st, out, 0)
            nbytes = T * (ENTRY + 2 * ENTRY) + (T // BS) * 4
        else:
            cols = 512 if name == "gather_kv_c" else ENTRY
            out = torch.empty((T, cols), dtype=torch.uint8, device=dev)
            fn = lambda: ops.mla_context_gather(cache, 1, nb, BS, BS * ENTRY, ENTRY, cols, table,
                                                cu, st, out, 1)
            nbytes = T * 2 * cols + (T // BS) * 4
    elif name in ("pack", "pack_bf16", "pack_f16"):
        T = tokens or 32768
        bf = name == "pack_bf16"
        kvb = torch.randn((T, ROW_STRIDE), generator=g, device=dev).to(
            torch.float16 if name == "pack_f16" else torch.bfloat16)
        heads = kvb[:, :HEADS * 256].view(T, HEADS, 256)
        if bf:
            ws = torch.randn((T, ENTRY), generator=g, device=dev).to(torch.bfloat16)
        else:
            ws = torch.randint(0, 126, (T, ENTRY), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        odt = torch.bfloat16 if bf else torch.uint8
        key = torch.empty((T, HEADS, 192), dtype=odt, device=dev)
        vo = torch.empty((T, HEADS, 128), dtype=odt, device=dev)
        sc = None if bf else torch.tensor([OUT_SCALE], dtype=torch.float32, device=dev)
        fn = lambda: ops.mla_context_kv_pack(heads[:, :, :128], heads[:, :, 128:], ws[:, 512:],
                                             key, vo, 0 if bf else 1, kpe_dtype=0 if bf else 1,
                                             out_scale=sc)
        nbytes = T * (HEADS * 512 + (128 if bf else 64) + HEADS * 320 * (2 if bf else 1))
    elif name == "norm_rope":
        T = tokens or 65536
        kv = torch.randn((T, L_LAYERS, ENTRY), generator=g, device=dev).to(torch.bfloat16)
        pos = torch.randint(0, W.MAX_POSITION, (T,), generator=g, device=dev)
        gamma = (1 + 0.1 * torch.randn((L_LAYERS, 512), generator=g, device=dev)).to(torch.bfloat16)
        table = torch.empty((W.MAX_POSITION, 64), dtype=torch.float32, device=dev)
        ops.mla_rope_cos_sin_cache(table, W.ROPE_BASE)
        oc = torch.empty((L_LAYERS, T, 512), dtype=torch.bfloat16, device=dev)
        op = torch.empty((L_LAYERS, T, 64), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.mla_norm_rope_grouped(kv[:, :, :512], kv[:, :, 512:],
                                               oc.transpose(0, 1), op.transpose(0, 1),
                                               gamma=gamma, eps=1e-6, positions=pos,
                                               cos_sin_cache=table)
        nbytes = T * L_LAYERS * 2 * ENTRY * 2 + T * (8 + 256)
    elif name == "pack_paged":
        T, nb = tokens or 32768, 4096
        assert T <= nb * BS
        kvb = torch.randn((T, ROW_STRIDE), generator=g, device=dev).to(torch.bfloat16)
        heads = kvb[:, :HEADS * 256].view(T, HEADS, 256)
        cache = torch.randint(0, 126, (nb * BS * ENTRY,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        table = torch.randperm(nb, generator=g, device=dev).to(torch.int32)[None, :].contiguous()
        cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
        st = torch.tensor([0], dtype=torch.int32, device=dev)
        key = torch.empty((T, HEADS, 192), dtype=torch.uint8, device=dev)
        vo = torch.empty((T, HEADS, 128), dtype=torch.uint8, device=dev)
        sc = torch.tensor([OUT_SCALE], dtype=torch.float32, device=dev)
        fn = lambda: ops.mla_context_kv_pack_paged(heads[:, :, :128], heads[:, :, 128:], cache, 1,
                                                   nb, BS, BS * ENTRY, ENTRY, table, cu, st, key,
                                                   vo, 1, out_scale=sc)
        nbytes = T * (HEADS * 512 + 64 + HEADS * 320) + (T // BS) * 4
    elif name == "pack_gather":
        # the pack of T tokens (fp8 out, 16 heads, k_pe from workspace A) and
        # the gather of the next T rows into workspace B, one launch
        T, nb = tokens or 8192, 4096
        assert 2 * T <= nb * BS
        kvb = torch.randn((T, ROW_STRIDE), generator=g, device=dev).to(torch.bfloat16)
        heads = kvb[:, :HEADS * 256].view(T, HEADS, 256)
        cache = torch.randint(0, 126, (nb * BS * ENTRY,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        table = torch.randperm(nb, generator=g, device=dev).to(torch.int32)[None, :].contiguous()
        cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
        st = torch.tensor([T], dtype=torch.int32, device=dev)
        ws_a = torch.randint(0, 126, (T, ENTRY), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        ws_b = torch.empty((T, ENTRY), dtype=torch.uint8, device=dev)
        key = torch.empty((T, HEADS, 192), dtype=torch.uint8, device=dev)
        vo = torch.empty((T, HEADS, 128), dtype=torch.uint8, device=dev)
        sc = torch.tensor([OUT_SCALE], dtype=torch.float32, device=dev)
        pk = ops.kv_pack_desc(heads[:, :, :128], heads[:, :, 128:], ws_a[:, 512:], key, vo, 1,
                              kpe_dtype=1, out_scale=sc)
        gd = ops.context_gather_desc(cache, 1, nb, BS, BS * ENTRY, ENTRY, ENTRY, table, cu, st,
                                     ws_b, 1)
        fn = lambda: ops.mla_context_kv_pack_gather(pk, gd)
        nbytes = T * B_PACK_TOK + T * B_GATHER_TOK + (T // BS) * 4
    else:
        raise SystemExit(f"unknown profile case {name}")
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:  # the launches replayed from one CUDA graph: no host gaps between them
        stream = torch.cuda.Stream()
        g = graph_of(lambda: [fn() for _ in range(launches)], stream)
        us = time_graph(g, stream, 3) / launches * 1e3
    else:
        s.record()
        for _ in range(launches):
            fn()
        e.record()
        e.synchronize()
        us = s.elapsed_time(e) / launches * 1e3
    print(json.dumps({"profile_case": name, "tokens": T, "graph": graph, "launches": launches,
                      "us_per_launch": us,
                      "bytes_per_launch": nbytes, "gbs": nbytes / us / 1e3}), flush=True)
    return 0


def host_cost_row(T, kv_c, k_pe, slots, ptrs, scales, graph_us):
    """Host cost of a decode-size insert without a CUDA graph: wall time per
    call of 1000 back-to-back calls (then one synchronize), best of 5.
      api      through the Python binding (argument marshalling included);
      abi      the C entry point called through ctypes with its arguments
               built once (what a C caller pays, plus the ctypes call);
      floor    the same call with num_tokens = 0, which returns after the
               argument checks that need no CUDA call (ctypes + validation);
    each for one grouped call and for five single-layer calls, with the
    per-call device-pointer checks on (default) and off."""
    import torch
    from pack_mla_cache_gb300 import ops

    L = kv_c.shape[0]
    lib = ops.lib()
    fn = lib.mla_cache_insert_grouped
    st = torch.cuda.current_stream().cuda_stream

    def args_of(l0, nl, t):
        return (kv_c[l0].data_ptr(), 512, T * 512, k_pe[l0].data_ptr(), 64, T * 64, t, nl, 512,
                64, slots.data_ptr(), 0, ptrs[l0:].data_ptr(), scales[l0:].data_ptr(), 1, 64, 64,
                64 * ENTRY, ENTRY, None, None, st)

    grouped_args = args_of(0, L, T)
    layer_args = [args_of(l, 1, T) for l in range(L)]
    floor_args = args_of(0, L, 0)

    def host_us(call, n=1000):
        for _ in range(50):
            call()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(5):
            t0 = time.perf_counter()
            for _ in range(n):
                call()
            torch.cuda.synchronize()
            best = min(best, (time.perf_counter() - t0) / n * 1e6)
        return best

    def abi_grouped():
        assert fn(*grouped_args) == 0

    def abi_layers():
        for a in layer_args:
            fn(*a)

    row = {"small_batch": f"host_L{L}_T{T}_e4m3", "graph_grouped_us": graph_us,
           "api_grouped_us": host_us(lambda: ops.mla_cache_insert_grouped(
               kv_c, k_pe, slots, ptrs, scales, 1, 64, 64, 64 * ENTRY, ENTRY)),
           "abi_floor_us": host_us(lambda: fn(*floor_args)),
           "abi_grouped_us": host_us(abi_grouped),
           "abi_five_single_layer_us": host_us(abi_layers)}
    prev = ops.mla_set_pointer_checks(False)
    try:
        row["abi_grouped_no_ptr_checks_us"] = host_us(abi_grouped)
        row["abi_five_single_layer_no_ptr_checks_us"] = host_us(abi_layers)
    finally:
        ops.mla_set_pointer_checks(prev)
    row["note"] = ("wall time per call of 1000 back-to-back calls; the kernel itself takes "
                   "graph_grouped_us")
    return row


def run_small_batch() -> int:
    """The small-batch inserts, each timed over 200 calls replayed from one CUDA
    graph (one JSON line each):
      * L=1, T=64, bf16 cache of 16 blocks x 64 x 576, raw insert;
      * L=5, T in {1, 2, 4, 8}, e4m3 caches of 64 blocks x 64 x 576, one shared
        mapping: one grouped call against five single-layer calls of the same
        library (the comparison "PR #55356 [Kimi Perf] Group fp8 mla cache
        insertion" makes for its small-batch speedup);
      * L=5, T=4096 with RMSNorm + RoPE, e4m3 / e5m2, shared / per-layer
        mapping, with one input set (L2-resident) and 6 rotating sets;
      * 32768 context tokens in 4 chunks of 8192: gather + pack per chunk,
        fp8 e4m3 and bf16 output."""
    import torch
    from pack_mla_cache_gb300 import ops
    from pack_mla_cache_gb300 import workloads as Wl
    import __graft_entry__
    __graft_entry__.build()
    W_MAX_POSITION = lambda: Wl.MAX_POSITION  # noqa: E731
    dev = torch.device("cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    stream = torch.cuda.Stream()
    calls = 200

    def timed(fn):
        gr = graph_of(lambda: [fn() for _ in range(calls)], stream)
        return min(time_graph(gr, stream, 3) for _ in range(5)) / calls * 1e3  # us per call

    # L=1, T=64 raw bf16
    kv_c = torch.randn((1, 64, 512), generator=g, device=dev).to(torch.bfloat16)
    k_pe = torch.randn((1, 64, 64), generator=g, device=dev).to(torch.bfloat16)
    cache = torch.zeros(16 * 64 * ENTRY, dtype=torch.bfloat16, device=dev)
    ptrs = torch.tensor([cache.data_ptr()], dtype=torch.int64, device=dev)
    slots = torch.randperm(1024, generator=g, device=dev)[:64]
    us = timed(lambda: ops.mla_cache_insert_grouped(kv_c, k_pe, slots, ptrs, None, 0, 16, 64,
                                                    64 * ENTRY, ENTRY))
    print(json.dumps({"small_batch": "L1_T64_bf16_raw", "us_per_call": us,
                      "tokens_layers_per_s": 64 / (us * 1e-6),
                      "bytes_per_call": 64 * (1152 + 8 + 1152)}), flush=True)
    # L=5, T=1..8 e4m3, grouped vs per layer
    L = 5
    caches = [torch.zeros(64 * 64 * ENTRY, dtype=torch.uint8, device=dev) for _ in range(L)]
    ptrs = torch.tensor([c.data_ptr() for c in caches], dtype=torch.int64, device=dev)
    scales = torch.rand(L, generator=g, device=dev) * 0.015 + 0.005
    for T in (1, 2, 4, 8):
        kv_c = torch.randn((L, T, 512), generator=g, device=dev).to(torch.bfloat16)
        k_pe = torch.randn((L, T, 64), generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(4096, generator=g, device=dev)[:T]
        grouped = timed(lambda: ops.mla_cache_insert_grouped(kv_c, k_pe, slots, ptrs, scales, 1,
                                                             64, 64, 64 * ENTRY, ENTRY))

        def per_layer():
            for l in range(L):
                ops.mla_cache_insert_grouped(kv_c[l:l + 1], k_pe[l:l + 1], slots, ptrs[l:l + 1],
                                             scales[l:l + 1], 1, 64, 64, 64 * ENTRY, ENTRY)
        five = timed(per_layer)
        print(json.dumps({"small_batch": f"L5_T{T}_e4m3", "grouped_us": grouped,
                          "five_single_layer_us": five, "speedup": five / grouped,
                          "tokens_layers_per_s": L * T / (grouped * 1e-6)}), flush=True)
        print(json.dumps(host_cost_row(T, kv_c, k_pe, slots, ptrs, scales, grouped)), flush=True)
    # L=5, T=4096, RMSNorm + RoPE into 512-block caches: e4m3 / e5m2 x shared / per-layer
    # mapping; one input and cache set (L2-resident) and 6 rotating sets (219 MB > L2)
    T, NB = 4096, 512
    table = torch.empty((W_MAX_POSITION(), 64), dtype=torch.float32, device=dev)
    ops.mla_rope_cos_sin_cache(table, 1e4)
    gamma = (1 + 0.1 * torch.randn((L, 512), generator=g, device=dev)).to(torch.bfloat16)

    def make_set(shared):
        kv_c = torch.randn((L, T, 512), generator=g, device=dev).to(torch.bfloat16)
        k_pe = torch.randn((L, T, 64), generator=g, device=dev).to(torch.bfloat16)
        rows = 1 if shared else L
        sl = torch.stack([torch.randperm(NB * 64, generator=g, device=dev)[:T] for _ in range(rows)])
        sl = sl[0] if shared else sl
        pos = torch.randint(0, W_MAX_POSITION(), (T,), generator=g, device=dev)
        cs = [torch.zeros(NB * 64 * ENTRY, dtype=torch.uint8, device=dev) for _ in range(L)]
        pt = torch.tensor([c.data_ptr() for c in cs], dtype=torch.int64, device=dev)
        return kv_c, k_pe, sl, pos, cs, pt

    # the per-layer pointer arrays and scales are uploaded once, up front: the
    # row shape may build its per-layer table before the launch wait (the
    # stream-order figure is reported beside it)
    prev_early = ops.mla_set_insert_early_tables(True)
    for fmt in (1, 2):
        for shared in (True, False):
            sets = [make_set(shared) for _ in range(6)]
            per_tok = 8 + 256 + (8 if shared else 8 * L)
            nbytes = T * L * (1152 + 576) + T * per_tok

            def call(st):
                kv_c, k_pe, sl, pos, _, pt = st
                ops.mla_cache_insert_grouped(kv_c, k_pe, sl, pt, scales, fmt, NB, 64, 64 * ENTRY,
                                             ENTRY, gamma=gamma, eps=1e-6, positions=pos,
                                             cos_sin_cache=table)
            resident = timed(lambda: call(sets[0]))
            rot_graph = graph_of(lambda: [call(sets[i % 6]) for i in range(calls)], stream)
            rotating = min(time_graph(rot_graph, stream, 3) for _ in range(5)) / calls * 1e3
            ops.mla_set_insert_early_tables(False)
            so_graph = graph_of(lambda: [call(sets[i % 6]) for i in range(calls)], stream)
            rotating_so = min(time_graph(so_graph, stream, 3) for _ in range(5)) / calls * 1e3
            ops.mla_set_insert_early_tables(True)
            del so_graph
            print(json.dumps({"small_batch": f"L5_T4096_norm_rope_{'e4m3' if fmt == 1 else 'e5m2'}_"
                              f"{'shared' if shared else 'per_layer'}_slots",
                              "bytes_per_call": nbytes,
                              "l2_resident_us": resident, "l2_resident_gbs": nbytes / resident / 1e3,
                              "rotating_6_sets_us": rotating,
                              "rotating_gbs": nbytes / rotating / 1e3,
                              "rotating_6_sets_stream_order_us": rotating_so}), flush=True)
            del sets
    ops.mla_set_insert_early_tables(prev_early)
    # cfg 4: one sequence of 32768 context tokens in 4 chunks of 8192 from a 1024-block fp8
    # cache; per chunk a gather then a pack, fp8 e4m3 out (raw fp8 k_pe) and bf16 out (the
    # gather widens to bf16 for a bf16 kv_b_proj)
    C, NC, NBC = 8192, 4, 1024
    ops.mla_set_gather_early_tables(True)  # the tables below are uploaded once, up front
    ctx = torch.randint(0, 126, (NBC * 64 * ENTRY,), generator=g, device=dev,
                        dtype=torch.int32).to(torch.uint8)
    btab = torch.randperm(NBC, generator=g, device=dev)[:NC * C // 64].to(torch.int32)[None, :].contiguous()
    cu = torch.tensor([0, C], dtype=torch.int32, device=dev)
    starts = [torch.tensor([c * C], dtype=torch.int32, device=dev) for c in range(NC)]
    kvbs = [torch.randn((C, ROW_STRIDE), generator=g, device=dev).to(torch.bfloat16)
            for _ in range(NC)]
    sc = torch.tensor([OUT_SCALE], dtype=torch.float32, device=dev)
    for out in ("e4m3", "bf16"):
        bf = out == "bf16"
        ws = torch.empty((C, ENTRY), dtype=torch.bfloat16 if bf else torch.uint8, device=dev)
        odt = torch.bfloat16 if bf else torch.uint8
        keys = [torch.empty((C, HEADS, 192), dtype=odt, device=dev) for _ in range(NC)]
        vs = [torch.empty((C, HEADS, 128), dtype=odt, device=dev) for _ in range(NC)]

        def chunks():
            for c in range(NC):
                ops.mla_context_gather(ctx, 1, NBC, 64, 64 * ENTRY, ENTRY, ENTRY, btab, cu,
                                       starts[c], ws, 0 if bf else 1)
                h = kvbs[c][:, :HEADS * 256].view(C, HEADS, 256)
                ops.mla_context_kv_pack(h[:, :, :128], h[:, :, 128:], ws[:, 512:], keys[c], vs[c],
                                        0 if bf else 1, kpe_dtype=0 if bf else 1,
                                        out_scale=None if bf else sc)
        # the same chunk loop with each pack and the next chunk's gather in one launch
        # (two workspaces): 5 launches instead of 8
        ws2 = [ws, torch.empty_like(ws)]
        cu0 = torch.tensor([0, 0], dtype=torch.int32, device=dev)
        descs = []
        for c in range(NC):
            h = kvbs[c][:, :HEADS * 256].view(C, HEADS, 256)
            pk = ops.kv_pack_desc(h[:, :, :128], h[:, :, 128:], ws2[c % 2][:, 512:], keys[c], vs[c],
                                  0 if bf else 1, kpe_dtype=0 if bf else 1,
                                  out_scale=None if bf else sc)
            nxt = c + 1 < NC
            gd = ops.context_gather_desc(ctx, 1, NBC, 64, 64 * ENTRY, ENTRY, ENTRY, btab,
                                         cu if nxt else cu0, starts[c + 1 if nxt else c],
                                         ws2[(c + 1) % 2], 0 if bf else 1,
                                         num_tokens=C if nxt else 0)
            descs.append((pk, gd))

        def chunks_fused():
            ops.mla_context_gather(ctx, 1, NBC, 64, 64 * ENTRY, ENTRY, ENTRY, btab, cu, starts[0],
                                   ws2[0], 0 if bf else 1)
            for pk, gd in descs:
                ops.mla_context_kv_pack_gather(pk, gd)
        per_tok = (576 + (1152 if bf else 576) + 4 / 64 + (B_PACK_TOK_BF16 if bf else B_PACK_TOK))
        nbytes = NC * C * per_tok
        for suffix, fn, launches in (("", chunks, 2 * NC), ("_fused", chunks_fused, NC + 1)):
            gr = graph_of(fn, stream)
            ms = min(time_graph(gr, stream, 5) for _ in range(5))
            print(json.dumps({"small_batch": f"cfg4_32768_context_4x8192_{out}{suffix}",
                              "launches": launches, "us": ms * 1e3, "bytes": nbytes,
                              "gbs": nbytes / (ms * 1e-3) / 1e9,
                              "context_tokens_per_s": NC * C / (ms * 1e-3)}), flush=True)
            del gr
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--profile-case", default=None,
                    help="run a few launches of one kernel (see run_profile_case)")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=None, help="tokens of the profile case")
    ap.add_argument("--graph", action="store_true", help="replay the profile case's launches from a CUDA graph")
    ap.add_argument("--small-batch", action="store_true",
                    help="time the small-batch inserts (grouped vs five single-layer calls)")
    args = ap.parse_args()
    if args.small_batch:
        return run_small_batch()
    if args.profile_case:
        return run_profile_case(args.profile_case, args.launches, args.tokens, args.graph)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run(args)


if __name__ == "__main__":
    sys.exit(main())
