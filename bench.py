"""Benchmark: paged decode attention KV GB/s (% of HBM peak) and decode tokens/s.

Workload: the large-batch decode workload -- batch 256, 32 query heads / 8 KV
heads, head_dim 128, block 16, 32 layers, context lengths U[128, 4096],
physical blocks interleaved across sequences, bf16 pool of about 71 GB.

One step = one decode step of the whole model's attention: for each of the 32
layers, append the new token's K/V (pa_write_kv, into the last context slot) and
run pa_decode_attention over the context (split-K + combine when partitioned).
Each layer reads ~2.2 GB of K/V, far more than the 129 MB L2, so no flush is
needed between steps.  By default the K timed steps run as one CUDA graph
replay (the calls captured once, each decode call bracketed by event-record
nodes for its per-call time); --no-graph launches every call from the host.

After the headline line's own measurements, the same run measures the other
workloads one at a time (graph-timed, each with its clock record) and adds them
to the line as "workloads": the batched gather on the large-batch pool, the
mini-infer-shaped 24-layer step, the long-context call, the large-batch lengths
with 16- to 128-query-head groups (the tcgen05 kernel), and the append +
decode loop with the free stack on the device.  --no-workloads skips them.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
Under torchrun every rank runs an independent replica (weak scaling, no
collective on the data path); the timed region is bracketed by barriers and the
max over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

METRIC = "paged decode attention KV GB/s"
UNIT = "GB/s"
WORKLOAD_CFG = 3


# ------------------------------------------------------------------ helpers


def decode_bytes(wl) -> int:
    """Algorithmic bytes of one pa_decode_attention call (one layer): K and V
    of every context token, q, the fp32 output, the table entries used and the
    lengths."""
    lens = wl.context_lens.astype(np.int64)
    kv = int(lens.sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    qb = wl.batch * wl.num_heads * wl.head_dim * wl.elem_bytes
    ob = wl.batch * wl.num_heads * wl.head_dim * 4
    tb = int(sum(-(-int(n) // wl.block_size) for n in lens)) * 4
    return kv + qb + ob + tb + wl.batch * 4


def append_bytes(wl) -> int:
    """Algorithmic bytes of one layer's KV append: the new K and V rows read and
    written, and the positions."""
    return 2 * 2 * wl.batch * wl.num_kv_heads * wl.head_dim * wl.elem_bytes + wl.batch * 4


def kernel_name(B, kind: int) -> str:
    """The decode kernel's name for a PA_DECODE_* kind."""
    return {B.PA_DECODE_CUDA_CORES: "pa_decode_kernel",
            B.PA_DECODE_TENSOR_CORES: "pa_decode_mma_kernel",
            B.PA_DECODE_TCGEN05: "pa_decode_umma_kernel"}[kind]


def decode_flops(wl) -> int:
    return int(wl.context_lens.astype(np.int64).sum()) * 4 * wl.num_heads * wl.head_dim


# DRAM bytes (read + write) of one layer's pa_write_kv_and_decode call on this
# workload, one ncu capture per kernel on the 1-layer pool (--metrics
# dram__bytes_read.sum,dram__bytes_write.sum, -k one kernel, -c 2):
# pa_decode_mma_kernel with the fused append 2,231,443,968 read + 6,390,784
# written, pa_combine_kernel 9,848,064 read + 0 written; see profiles/.  Valid
# only for the sources they were taken from (the kernels, the shared device
# code, and the dispatch / partition choice in pa_api.cpp).
DECODE_TRAFFIC = {
    "bytes_per_launch": 2231443968 + 6390784 + 9848064,
    "sources_sha256": "e8553c7561bc99f0d93bcf519ca31ec7d25ef9f18a7ddd6e270573826241a3c1",
}
DECODE_SOURCES = ["pa_decode_mma.cuh", "pa_decode_mma.cu", "pa_decode.cuh", "pa_device.cuh",
                  "pa_internal.h", "pa_api.cpp", "pa_fused_append.cuh"]


def decode_sources_sha256() -> str:
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(REPO, "paged_kv_cache_239_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def decode_traffic():
    """Per-launch DRAM traffic of the decode kernel, or None if it changed since the capture."""
    if decode_sources_sha256() == DECODE_TRAFFIC["sources_sha256"]:
        return DECODE_TRAFFIC["bytes_per_launch"]
    return None


# The GB300's nominal HBM3e bandwidth (8 stacks, ~7.9 TB/s): the denominator of
# the "fraction of HBM peak" the target is stated in.  The roofline itself is
# taken against the measured copy bandwidth (MEASURED_PEAKS.json), which a
# read-mostly stream can exceed.
NOMINAL_HBM_GBS = 7900.0


def measured_peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(values, world: int, device="cpu"):
    """Element-wise max of per-rank timings (a host-side reduction of a few
    scalars; the data path itself has no collective)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def l2_note(wl, L) -> str:
    kv = int(wl.context_lens.astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    if kv > 129e6:
        return f"inputs larger than L2 ({kv / 1e9:.2f} GB of K/V per layer vs 129 MB L2), no flush"
    return (f"K/V per layer {kv / 1e6:.1f} MB < L2; consecutive layers read disjoint pool "
            f"slices ({kv * L / 1e6:.0f} MB per step), no flush")


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(wl, nseq: int, pool_getter, q_getter, layer: int = 0):
    """Times the oracle on the first `nseq` sequences of one layer.  Returns
    (bytes, seconds, threads)."""
    import oracle
    from paged_kv_cache_239_gb300 import workloads as W

    tables, lens = [], []
    blocks = []
    for b in range(nseq):
        n = int(wl.context_lens[b])
        nblk = -(-n // wl.block_size)
        ids = list(range(len(blocks), len(blocks) + nblk))
        blocks.extend(int(x) for x in wl.block_tables[b, :nblk])
        row = np.full(wl.max_blocks, -1, np.int32)
        row[:nblk] = ids
        tables.append(row)
        lens.append(n)
    sub_pool = pool_getter(blocks, layer)          # [len(blocks), 2, 1, Hkv, B, D]
    q = q_getter(nseq, layer)                      # [nseq, H, D]
    tables = np.stack(tables)
    lens = np.array(lens, np.int32)
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.decode_attention(W.as_oracle_array(q), W.as_oracle_array(sub_pool), 0, tables, lens,
                            wl.num_heads, wl.scale, threads=threads)
    dt = time.perf_counter() - t0
    sub = W.Workload(wl.name, wl.dtype, 1, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                     wl.block_size, lens, tables, len(blocks), wl.scale, wl.seed)
    return decode_bytes(sub), dt, threads


# --------------------------------------------------------------- reference


def run_reference(args, rank: int, world: int) -> None:
    """The oracle as the reference arm: each step is one layer of a bounded
    sample of the workload's sequences, on the host cores."""
    if rank != 0:
        return
    import torch

    from paged_kv_cache_239_gb300 import workloads as W

    wl = W.named(WORKLOAD_CFG)
    nseq = args.ref_seqs
    # inputs for the sampled sequences only, drawn on the CPU with the seeded generators
    nblk = [-(-int(n) // wl.block_size) for n in wl.context_lens[:nseq]]
    sub = W.custom(wl.name, wl.dtype, 1, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                   wl.block_size, wl.context_lens[:nseq], seed=wl.seed, max_blocks=wl.max_blocks)
    assert sub.num_blocks == sum(nblk)
    pool = W.make_pool(sub)
    q = W.make_queries(sub, 1)[0]

    def pool_getter(blocks, layer):
        return pool.index_select(0, torch.tensor(blocks, dtype=torch.long))

    def q_getter(n, layer):
        return q[:n]

    times, nbytes, threads = [], 0, 1
    for i in range(args.warmup + args.steps):
        nbytes, dt, threads = oracle_sample(sub, nseq, pool_getter, q_getter)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{wl.name} (sample: first {nseq} sequences, one layer per step)",
                   "batch": nseq, "num_heads": wl.num_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "block_size": wl.block_size},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{nseq} sequences x 1 layer per step, fp64 C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm


def run_gpu(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import torch.distributed as dist

    from paged_kv_cache_239_gb300 import _build_lib
    from paged_kv_cache_239_gb300 import binding as B
    from paged_kv_cache_239_gb300 import workloads as W

    _build_lib.build()
    B.lib()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    wl = W.named(args.workload)
    if args.num_heads > 0:     # same lengths and tables; another query-head count
        wl.num_heads = args.num_heads
    if args.kv_heads > 0:      # same lengths, tables and query heads; another group size
        wl.num_kv_heads = args.kv_heads
    if wl.num_heads % wl.num_kv_heads:
        raise SystemExit("the KV heads must divide the query heads")
    if args.pool_layers > 0:   # smaller pool (same lengths/tables) for profiler captures
        wl.num_layers = min(args.pool_layers, wl.num_layers)
    L = wl.num_layers if args.layers <= 0 else min(args.layers, wl.num_layers)
    pool = W.make_pool(wl, device=dev, seed_offset=rank)
    qs = W.make_queries(wl, L, device=dev, seed_offset=rank)
    ks, vs = W.make_new_tokens(wl, L, device=dev, seed_offset=rank)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    positions = (lens - 1).contiguous()   # the new token takes the last context slot
    h = B.pa_pool_create(pool, wl.num_blocks, wl.num_layers, wl.num_kv_heads, wl.block_size,
                         wl.head_dim, pool.dtype)
    pb = B.pa_decode_partition_blocks(h, wl.batch, wl.num_heads, wl.max_blocks)
    ws_bytes = B.pa_decode_workspace_size(h, wl.batch, wl.num_heads, wl.max_blocks, 0)
    kernel_kind = B.pa_decode_kernel_choice(h, wl.num_heads)
    decode_kernel = kernel_name(B, kernel_kind)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    outs = torch.empty((L, wl.batch, wl.num_heads, wl.head_dim), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cur = {"sp": stream.cuda_stream, "stream": stream}
    lib = B.lib()
    # a second (combine) kernel runs exactly when the call needs a workspace
    launches_per_step = L * ((1 if args.fused else 2) + (1 if ws_bytes > 0 else 0))

    sets = [dict(q=qs, k=ks, v=vs, bt=bt, lens=lens, pos=positions, out=outs)]

    def layer_call(l, ev=None, bs=None):
        bs = sets[0] if bs is None else bs
        if args.fused:
            if ev is not None:
                ev[0].record(cur["stream"])
            rc = lib.pa_write_kv_and_decode(bs["out"][l].data_ptr(), bs["q"][l].data_ptr(), h, l,
                                            bs["k"][l].data_ptr(), bs["v"][l].data_ptr(),
                                            bs["pos"].data_ptr(), bs["bt"].data_ptr(),
                                            wl.max_blocks, bs["lens"].data_ptr(), wl.batch,
                                            wl.block_size, wl.num_heads, wl.num_kv_heads,
                                            wl.head_dim, wl.scale, 0, ws.data_ptr(), ws_bytes,
                                            cur["sp"])
            if rc:
                raise RuntimeError(B.last_error())
            if ev is not None:
                ev[1].record(cur["stream"])
            return
        rc = lib.pa_write_kv(h, l, bs["k"][l].data_ptr(), bs["v"][l].data_ptr(),
                             bs["bt"].data_ptr(), wl.max_blocks, bs["pos"].data_ptr(), wl.batch,
                             cur["sp"])
        if rc:
            raise RuntimeError(B.last_error())
        if ev is not None:
            ev[0].record(cur["stream"])
        rc = lib.pa_decode_attention(bs["out"][l].data_ptr(), bs["q"][l].data_ptr(), h, l,
                                     bs["bt"].data_ptr(), wl.max_blocks, bs["lens"].data_ptr(),
                                     wl.batch, wl.block_size, wl.num_heads, wl.num_kv_heads,
                                     wl.head_dim, wl.scale, ws.data_ptr(), ws_bytes, cur["sp"])
        if rc:
            raise RuntimeError(B.last_error())
        if ev is not None:
            ev[1].record(cur["stream"])

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- warm-up ----
    for _ in range(args.warmup):
        for l in range(L):
            layer_call(l)
    torch.cuda.synchronize()
    st = B.pa_get_status()
    if st:
        raise RuntimeError(f"device status {st:#x} after warm-up")

    # ---- CUDA graphs (default): the timed K steps as one graph whose decode
    #      calls are bracketed by event-record nodes, and a one-step graph for
    #      the end-to-end leg ----
    use_graph = not args.no_graph
    graph = step_graph = None
    ev_kw = {"enable_timing": True, "external": True} if use_graph else {"enable_timing": True}
    evs = [[(torch.cuda.Event(**ev_kw), torch.cuda.Event(**ev_kw)) for _ in range(L)]
           for _ in range(args.steps)]

    def capture(body):
        g_ = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            cur["sp"] = side.cuda_stream
            cur["stream"] = side
            with torch.cuda.graph(g_, stream=side):
                body()
            cur["sp"] = stream.cuda_stream
            cur["stream"] = stream
        stream.wait_stream(side)
        return g_

    if use_graph:
        def all_steps():
            for s in range(args.steps):
                for l in range(L):
                    layer_call(l, evs[s][l])

        def one_step():
            for l in range(L):
                layer_call(l)

        graph = capture(all_steps)
        step_graph = capture(one_step)
        for _ in range(args.warmup):
            step_graph.replay()
        graph.replay()   # untimed: the first launch of a graph uploads it to the device
        torch.cuda.synchronize()

    # ---- timed region: device-resident inputs.  With graphs, `value` comes from
    #      K replays of the uninstrumented one-step graph; the per-call times
    #      for the roofline from a second timed replay of the K-step graph whose
    #      decode calls are bracketed by event nodes (the nodes cost ~3%). ----
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    instrumented_ms = None
    with ClockSampler(torch.cuda.current_device()) as clocks:
        t_start.record(stream)
        if graph is not None:
            for _ in range(args.steps):
                step_graph.replay()
        else:
            for s in range(args.steps):
                for l in range(L):
                    layer_call(l, evs[s][l])
        t_end.record(stream)
        torch.cuda.synchronize()
        if graph is not None:
            i0 = torch.cuda.Event(enable_timing=True)
            i1 = torch.cuda.Event(enable_timing=True)
            i0.record(stream)
            graph.replay()
            i1.record(stream)
            torch.cuda.synchronize()
            instrumented_ms = i0.elapsed_time(i1)
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    call_ms = [a.elapsed_time(b) for row in evs for (a, b) in row]
    st = B.pa_get_status()
    if st:
        raise RuntimeError(f"device status {st:#x} after the timed region")

    # ---- end to end through the C ABI: every step copies its inputs (q, new
    #      K/V, tables, lengths, positions) from pinned host memory and every
    #      layer's output back.  Two device buffer sets and two copy streams:
    #      step s+1's uploads and step s-1's download overlap step s. ----
    e2e_ms, h2d, d2h = float("nan"), 0, 0
    if not args.no_e2e:
        host = dict(q=qs.cpu().pin_memory(), k=ks.cpu().pin_memory(), v=vs.cpu().pin_memory(),
                    bt=bt.cpu().pin_memory(), lens=lens.cpu().pin_memory(),
                    pos=positions.cpu().pin_memory())
        out_h = torch.empty(outs.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_h.numel() * out_h.element_size()
        sets.append({k_: t.clone() for k_, t in sets[0].items()})
        graphs = None
        if use_graph:
            graphs = [step_graph]
            for x in (1,):
                graphs.append(capture(lambda x=x: [layer_call(l, bs=sets[x]) for l in range(L)]))
        up = torch.cuda.Stream(dev)
        down = torch.cuda.Stream(dev)
        comp_done = [torch.cuda.Event(), torch.cuda.Event()]
        down_done = [torch.cuda.Event(), torch.cuda.Event()]
        up_done = [torch.cuda.Event(), torch.cuda.Event()]
        for e_ in comp_done + down_done:
            e_.record(stream)

        def e2e_step(si):
            x = si % 2
            bs = sets[x]
            up.wait_event(comp_done[x])            # step si-2 no longer reads set x
            with torch.cuda.stream(up):
                for key, t in host.items():
                    bs[key].copy_(t, non_blocking=True)
            up_done[x].record(up)
            stream.wait_event(up_done[x])
            stream.wait_event(down_done[x])        # step si-2's outputs have left
            if graphs is not None:
                graphs[x].replay()
            else:
                for l in range(L):
                    layer_call(l, bs=bs)
            comp_done[x].record(stream)
            down.wait_event(comp_done[x])
            with torch.cuda.stream(down):
                out_h.copy_(bs["out"], non_blocking=True)
            down_done[x].record(down)

        for i in range(max(2, args.warmup // 2)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(up)
        for i in range(args.steps):
            e2e_step(i)
        e1.record(down)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = e0.elapsed_time(e1)

    # ---- max over ranks ----
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], world, dev)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cache = {}

        def pool_getter(blocks, layer):
            if layer not in cache:
                ids = torch.tensor(blocks, dtype=torch.long, device=dev)
                cache[layer] = pool.index_select(0, ids)[:, :, layer:layer + 1].contiguous().cpu()
            return cache[layer]

        def q_getter(n, layer):
            return qs[layer, :n].cpu()

        # one layer of the first cpu_seqs sequences, repeated until about
        # cpu_seconds of oracle work have been timed
        nbytes, dt, threads, reps = 0, 0.0, 1, 0
        while reps < 2 or (dt < args.cpu_seconds and reps < 200):
            nb_, dt_, threads = oracle_sample(wl, args.cpu_seqs, pool_getter, q_getter, 0)
            nbytes += nb_
            dt += dt_
            reps += 1
        cpu = {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {args.cpu_seqs} of {wl.batch} sequences, layer 0, x{reps} "
                         f"repeats, fp64 C oracle ({dt:.1f} s)"}

    if rank != 0:
        B.pa_pool_destroy(h)
        return
    per_call = decode_bytes(wl)
    # the timed launch of a layer: the fused call also moves the appended rows
    launch_bytes = per_call + (append_bytes(wl) if args.fused else 0)
    steps = args.steps
    value = per_call * L * steps * world / (total_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    call_avg_ms = sum(call_ms) / len(call_ms)
    achieved = launch_bytes / (call_avg_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "num_layers": L,
            "context_lens": f"seed {wl.seed}, min {wl.context_lens.min()}, max "
                            f"{wl.context_lens.max()}, mean {wl.context_lens.mean():.0f}",
            "cuda_graph": use_graph,
            "append": ("fused into the decode launch (pa_write_kv_and_decode)" if args.fused
                       else "separate pa_write_kv launch before each decode"),
            "pool_gb": round(wl.pool_bytes() / 1e9, 1),
            "decode_kernel": decode_kernel,
            "partition_blocks": (pb if kernel_kind != B.PA_DECODE_TCGEN05 else
                                 "none: equal 128-token tile shares per persistent CTA"),
            "l2": l2_note(wl, L),
            "parallelism": f"replicas x{world}",
        },
        "pct_of_measured_copy_peak": 100.0 * value / peak,
        "pct_of_nominal_hbm_peak": 100.0 * value / NOMINAL_HBM_GBS,
        "decode_tokens_per_s": wl.batch * steps * world / (total_ms / 1e3),
        "roofline": {"bound": "hbm",
                     "kernel": ("pa_write_kv_and_decode (append + decode + combine)" if args.fused
                                else "pa_decode_attention (decode + combine)"),
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     # the captured counters belong to the default workload only
                     "traffic": (decode_traffic() if args.workload == WORKLOAD_CFG and
                                 args.kv_heads <= 0 and args.num_heads <= 0 and args.fused
                                 else None),
                     "traffic_kernel": (decode_kernel + (" (with the fused append)" if args.fused
                                                       else "") +
                                        " + pa_combine_kernel, ncu dram read+write per call"),
                     "algorithmic_bytes_per_call": launch_bytes,
                     "avg_call_ms": call_avg_ms,
                     "timing": ("CUDA events around every decode call, recorded as event nodes "
                                "of a graph replay of the same K steps"
                                if instrumented_ms is not None else
                                "CUDA events around every decode call of the timed region"),
                     "instrumented_step_ms": (instrumented_ms / steps
                                              if instrumented_ms is not None else None)},
        "cpu_baseline": cpu,
        "e2e": {"value": per_call * L * steps * world / (e2e_ms / 1e3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / steps,
                "overlap": "two device buffer sets; uploads and downloads on their own streams "
                           "overlap the neighbouring steps' compute"},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks.summary(),
    }
    if not args.no_workloads and world == 1:
        # the other workloads, each measured alone after the headline (the
        # gather on this pool first, then the pool is freed)
        extra = [measure_gather(B, torch, wl, pool, h, bt, lens, dev,
                                layers=min(4, wl.num_layers))]
        B.pa_pool_destroy(h)
        h = None
        del pool, qs, ks, vs, outs, ws, sets, graph, step_graph
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        extra += run_extra_workloads(args, B, torch, W, dev)
        line["workloads"] = extra
    print(json.dumps(line), flush=True)
    if h is not None:
        B.pa_pool_destroy(h)


def timed_graph_calls(torch, dev, call, ncalls, target_s=0.5):
    """CUDA-graph replays of `ncalls` calls (call(i)), warmed up, repeated
    until about target_s seconds have been timed with CUDA events on the
    replaying stream; returns (ms per call, clock summary)."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for i in range(ncalls):       # warm-up, outside the graph
            call(i, side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(ncalls):
                call(i, side)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    reps = max(3, min(200, int(target_s * 1e3 / max(e0.elapsed_time(e1), 1e-3))))
    with ClockSampler(torch.cuda.current_device()) as clocks:
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (reps * ncalls), clocks.summary()


def measure_step(B, torch, W, dev, wl, name, note=""):
    """Fused append + decode over every layer of a workload's pool (the
    benchmark step's call), graph-timed."""
    pool = W.make_pool(wl, device=dev)
    L = wl.num_layers
    qs = W.make_queries(wl, L, device=dev)
    ks, vs = W.make_new_tokens(wl, L, device=dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    pos = (lens - 1).contiguous()
    h = B.pa_pool_create(pool, wl.num_blocks, L, wl.num_kv_heads, wl.block_size, wl.head_dim,
                         pool.dtype)
    try:
        kind = B.pa_decode_kernel_choice(h, wl.num_heads)
        need = B.pa_decode_workspace_size(h, wl.batch, wl.num_heads, wl.max_blocks, 0)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        outs = torch.empty((L, wl.batch, wl.num_heads, wl.head_dim), dtype=torch.float32,
                           device=dev)
        lib = B.lib()

        def call(i, stream):
            l = i % L
            rc = lib.pa_write_kv_and_decode(outs[l].data_ptr(), qs[l].data_ptr(), h, l,
                                            ks[l].data_ptr(), vs[l].data_ptr(), pos.data_ptr(),
                                            bt.data_ptr(), wl.max_blocks, lens.data_ptr(),
                                            wl.batch, wl.block_size, wl.num_heads,
                                            wl.num_kv_heads, wl.head_dim, wl.scale, 0,
                                            ws.data_ptr(), need, stream.cuda_stream)
            if rc:
                raise RuntimeError(B.last_error())

        ms, clk = timed_graph_calls(torch, dev, call, max(L, 8))
        st = B.pa_get_status()
        if st:
            raise RuntimeError(f"device status {st:#x} in workload {name}")
    finally:
        B.pa_pool_destroy(h)
    peak, kind_p = measured_peaks()
    nbytes = decode_bytes(wl)
    gbs = nbytes / (ms / 1e3) / 1e9
    res = {"workload": name, "value": gbs, "unit": UNIT,
           "frac_of_measured_copy_peak": gbs / peak, "frac_of_nominal_hbm_peak":
           gbs / NOMINAL_HBM_GBS, "ms_per_call": ms, "decode_kernel": kernel_name(B, kind),
           "decode_tokens_per_s": wl.batch / (ms * L / 1e3),
           "shape": {"batch": wl.batch, "num_heads": wl.num_heads,
                     "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                     "block_size": wl.block_size, "num_layers": L},
           "timing": "graph replays of the fused append + decode call over the pool's layers, "
                     "CUDA events", "clocks": clk}
    if note:
        res["note"] = note
    del pool, qs, ks, vs, outs, ws
    torch.cuda.empty_cache()
    return res


def measure_gather(B, torch, wl, pool, h, bt, lens, dev, layers):
    """Row N1: pa_gather_kv of `layers` layers of a workload's pool, graph-timed."""
    T = int(wl.context_lens.max())
    shape = (wl.batch, T, wl.num_kv_heads, wl.head_dim)
    k = torch.empty(shape, dtype=pool.dtype, device=dev)
    v = torch.empty(shape, dtype=pool.dtype, device=dev)
    m = torch.empty((wl.batch, T), dtype=torch.uint8, device=dev)
    lib = B.lib()

    def call(i, stream):
        rc = lib.pa_gather_kv(k.data_ptr(), v.data_ptr(), m.data_ptr(), h, i % layers,
                              bt.data_ptr(), wl.max_blocks, lens.data_ptr(), wl.batch, T,
                              stream.cuda_stream)
        if rc:
            raise RuntimeError(B.last_error())

    ms, clk = timed_graph_calls(torch, dev, call, layers)
    assert B.pa_get_status() == 0
    rd = int(wl.context_lens.astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    wr = 2 * wl.batch * T * wl.num_kv_heads * wl.head_dim * wl.elem_bytes + wl.batch * T
    nb = rd + wr + int(sum(-(-int(n) // wl.block_size) for n in wl.context_lens)) * 4
    peak, _ = measured_peaks()
    gbs = nb / (ms / 1e3) / 1e9
    del k, v, m
    torch.cuda.empty_cache()
    return {"workload": f"gather_kv ({wl.name} layers)", "value": gbs, "unit": UNIT,
            "frac_of_measured_copy_peak": gbs / peak,
            "frac_of_nominal_hbm_peak": gbs / NOMINAL_HBM_GBS, "ms_per_call": ms,
            "bytes_per_call": nb, "timing": "graph replays of pa_gather_kv over 4 layers",
            "clocks": clk}


def run_extra_workloads(args, B, torch, W, dev):
    """The named workloads other than the headline, and the large-batch
    lengths with the large query groups the tcgen05 kernel serves."""
    res = []
    res.append(measure_step(B, torch, W, dev, W.named(2), "mini_infer_bf16",
                            "K/V per layer below L2; consecutive layers read disjoint slices"))
    res.append(measure_step(B, torch, W, dev, W.named(4), "long_context_bf16",
                            "one layer: every call re-reads the same 1.35 GB (10x L2)"))
    for H, Hkv in ((32, 2), (32, 1), (48, 1), (64, 1), (96, 1), (128, 1)):
        wl = W.named(3)
        wl.num_heads, wl.num_kv_heads, wl.num_layers = H, Hkv, 16 if Hkv == 1 else 8
        res.append(measure_step(B, torch, W, dev, wl,
                                f"large_batch_bf16 lengths, {H} query / {Hkv} KV heads "
                                f"(group {H // Hkv})"))
    res.append(measure_loop(B, torch, W, dev))
    return res


def measure_loop(B, torch, W, dev):
    """Workload 5, the append + decode loop with the free stack on the device,
    each run of 64 steps one CUDA graph."""
    import types

    a = types.SimpleNamespace(workload=5, warmup=3, steps=16, device_alloc=True)
    buf = {}
    run_loop(a, dev.index or 0, _result=buf)
    return buf["result"]


def _setup(args, local_rank, cfg):
    import torch

    from paged_kv_cache_239_gb300 import _build_lib
    from paged_kv_cache_239_gb300 import binding as B
    from paged_kv_cache_239_gb300 import workloads as W

    _build_lib.build()
    B.lib()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    return torch, B, W, dev, W.named(cfg)


def run_gather(args, local_rank: int) -> None:
    """Row N1: bandwidth of pa_gather_kv over every layer of a workload."""
    torch, B, W, dev, wl = _setup(args, local_rank, args.workload)
    pool = W.make_pool(wl, device=dev)
    h = B.pa_pool_create(pool, wl.num_blocks, wl.num_layers, wl.num_kv_heads, wl.block_size,
                         wl.head_dim, pool.dtype)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    T = int(wl.context_lens.max())
    shape = (wl.batch, T, wl.num_kv_heads, wl.head_dim)
    k = torch.empty(shape, dtype=pool.dtype, device=dev)
    v = torch.empty(shape, dtype=pool.dtype, device=dev)
    m = torch.empty((wl.batch, T), dtype=torch.uint8, device=dev)
    L = wl.num_layers

    def step():
        for l in range(L):
            B.pa_gather_kv(k, v, m, h, l, bt, wl.max_blocks, lens, wl.batch, T)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (args.steps * L)
    rd = int(wl.context_lens.astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    wr = 2 * wl.batch * T * wl.num_kv_heads * wl.head_dim * wl.elem_bytes + wl.batch * T
    nb = rd + wr + int(sum(-(-int(n) // wl.block_size) for n in wl.context_lens)) * 4
    peak, kind = measured_peaks()
    gbs = nb / (ms / 1e3) / 1e9
    assert B.pa_get_status() == 0
    print(json.dumps({"row": "gather", "workload": wl.name, "value": gbs, "unit": UNIT,
                      "ms_per_call": ms, "bytes_per_call": nb, "read_bytes": rd,
                      "write_bytes": wr, "frac_of_peak": gbs / peak,
                      "peak": peak, "peak_source": f"{kind} hbm_gbs", "steps": args.steps,
                      "layers": L}), flush=True)
    B.pa_pool_destroy(h)


def run_loop(args, local_rank: int, _result=None) -> None:
    """The append+decode loop (workload 5 by default): every step takes a block
    for each sequence crossing a block boundary (host free stack), copies the
    changed table rows, appends one token per sequence and decodes over n+1.
    One run = `steps_per_run` steps from the initial state; the allocator and
    tables are reset between runs (untimed)."""
    torch, B, W, dev, wl = _setup(args, local_rank, 5 if args.workload == WORKLOAD_CFG
                                  else args.workload)
    nsteps = wl.steps or 64
    pool = W.make_pool(wl, device=dev)
    ks, vs = W.make_new_tokens(wl, nsteps, device=dev)
    qs = W.make_queries(wl, nsteps, device=dev)
    h = B.pa_pool_create(pool, wl.num_blocks, wl.num_layers, wl.num_kv_heads, wl.block_size,
                         wl.head_dim, pool.dtype)
    used = sorted(int(x) for x in wl.block_tables[wl.block_tables >= 0])
    order = list(wl.free_stack) + used
    bt = torch.from_numpy(wl.block_tables.copy()).to(dev)
    lens_d = torch.empty(wl.batch, dtype=torch.int32, device=dev)
    pos_d = torch.empty(wl.batch, dtype=torch.int32, device=dev)
    out = torch.empty((wl.batch, wl.num_heads, wl.head_dim), dtype=torch.float32, device=dev)
    ws_b = B.pa_decode_workspace_size(h, wl.batch, wl.num_heads, wl.max_blocks, 0)
    ws = torch.empty(max(ws_b, 1), dtype=torch.uint8, device=dev)
    lens_pin = torch.empty(wl.batch, dtype=torch.int32).pin_memory()
    pos_pin = torch.empty(wl.batch, dtype=torch.int32).pin_memory()
    row_pin = torch.empty(wl.max_blocks, dtype=torch.int32).pin_memory()

    def reset():
        torch.cuda.synchronize()
        nonlocal h
        B.pa_pool_destroy(h)
        h = B.pa_pool_create(pool, wl.num_blocks, wl.num_layers, wl.num_kv_heads,
                             wl.block_size, wl.head_dim, pool.dtype)
        B.pa_pool_seed_free_stack(h, order)
        for _ in used:
            B.pa_alloc_block(h)
        bt.copy_(torch.from_numpy(wl.block_tables))
        torch.cuda.synchronize()

    def run():
        lens = wl.context_lens.copy()
        tables = wl.block_tables.copy()
        for s in range(nsteps):
            for b in np.nonzero(lens % wl.block_size == 0)[0]:
                blk = B.pa_alloc_block(h)
                j = lens[b] // wl.block_size
                tables[b, j] = blk
                bt[b, j:j + 1].copy_(torch.tensor([blk], dtype=torch.int32), non_blocking=True)
            pos_pin.copy_(torch.from_numpy(lens))
            pos_d.copy_(pos_pin, non_blocking=True)
            B.pa_write_kv(h, 0, ks[s], vs[s], bt, wl.max_blocks, pos_d, wl.batch)
            lens = lens + 1
            lens_pin.copy_(torch.from_numpy(lens))
            lens_d.copy_(lens_pin, non_blocking=True)
            B.pa_decode_attention(out, qs[s], h, 0, bt, wl.max_blocks, lens_d, wl.batch,
                                  wl.block_size, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                  wl.scale, ws, ws_b)
            torch.cuda.current_stream().synchronize()   # host reuses the pinned rows
        return lens

    if args.device_alloc:
        return run_loop_device(args, B, torch, wl, pool, ks, vs, qs, h, used, order, nsteps, dev,
                               _result)
    for _ in range(max(1, args.warmup // 3)):
        reset()
        run()
    times = []
    for _ in range(max(1, args.steps // 8)):
        reset()
        t0 = time.perf_counter()
        lens_end = run()
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    assert B.pa_get_status() == 0
    tot = sum(times)
    runs = len(times)
    # decode bytes summed over the loop's growing lengths
    kv = 0
    for s in range(nsteps):
        n = wl.context_lens.astype(np.int64) + s + 1
        kv += int(n.sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    peak, kind = measured_peaks()
    print(json.dumps({"row": "loop", "workload": wl.name, "steps_per_run": nsteps, "runs": runs,
                      "decode_tokens_per_s": wl.batch * nsteps * runs / tot,
                      "kv_gbs_wall": kv * runs / tot / 1e9, "ms_per_step": 1e3 * tot / (runs * nsteps),
                      "peak": peak, "timing": "host wall clock incl. allocation, H2D table "
                      "updates and a stream sync per step"}), flush=True)
    B.pa_pool_destroy(h)


def run_loop_device(args, B, torch, wl, pool, ks, vs, qs, h, used, order, nsteps, dev,
                    _result=None):
    """The same loop with the free stack on the device: each step is
    pa_device_alloc_blocks_step (the allocation and the next lengths, run a
    step ahead on a second stream) + pa_write_kv_and_decode, and a whole run of
    `nsteps` steps is one CUDA graph replay (no host round trip)."""
    B.pa_pool_seed_free_stack(h, order)
    for _ in used:
        B.pa_alloc_block(h)
    stack = torch.empty(wl.num_blocks + 1, dtype=torch.int32, device=dev)
    B.pa_device_stack_upload(h, stack)
    stack0 = stack.clone()
    bt0 = torch.from_numpy(wl.block_tables.copy()).to(dev)
    lens0 = torch.from_numpy(wl.context_lens.copy()).to(dev)
    bt = bt0.clone()
    # three length arrays in turn: step t's positions, its lengths (= step t +
    # 1's positions), and the one step t + 1's allocation writes meanwhile
    bufs = (lens0.clone(), lens0.clone(), lens0.clone())
    out = torch.empty((wl.batch, wl.num_heads, wl.head_dim), dtype=torch.float32, device=dev)
    maxlen_blocks = wl.max_blocks
    pb = B.pa_decode_partition_blocks(h, wl.batch, wl.num_heads, maxlen_blocks)
    need = B.pa_decode_workspace_size(h, wl.batch, wl.num_heads, maxlen_blocks, pb)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    B.pa_get_status()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    side = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            side.wait_stream(s)
            ev_alloc = [torch.cuda.Event() for _ in range(nsteps)]
            ev_dec = [torch.cuda.Event() for _ in range(nsteps)]

            def alloc(t):
                # step t's blocks and lengths (positions + 1) in one launch, on
                # a second stream a step ahead of the decodes; it waits for the
                # decode that last read the array it writes
                with torch.cuda.stream(side):
                    if t >= 2:
                        side.wait_event(ev_dec[t - 2])
                    B.pa_device_alloc_blocks_step(h, stack, bt, wl.max_blocks, bufs[t % 3],
                                                  bufs[(t + 1) % 3], wl.batch, stream=side)
                    ev_alloc[t].record(side)

            alloc(0)
            for t in range(nsteps):
                if t + 1 < nsteps:
                    alloc(t + 1)
                s.wait_event(ev_alloc[t])
                B.pa_write_kv_and_decode(out, qs[t], h, 0, ks[t], vs[t], bufs[t % 3], bt,
                                         wl.max_blocks, bufs[(t + 1) % 3], wl.batch,
                                         wl.block_size, wl.num_heads, wl.num_kv_heads,
                                         wl.head_dim, wl.scale, pb, ws, need, stream=s)
                ev_dec[t].record(s)
            s.wait_stream(side)
    torch.cuda.current_stream(dev).wait_stream(s)

    def reset():
        stack.copy_(stack0)
        bt.copy_(bt0)
        bufs[0].copy_(lens0)

    for _ in range(max(1, args.warmup)):
        reset()
        g.replay()
    torch.cuda.synchronize()
    runs = max(1, args.steps // 4)
    ms = 0.0
    with ClockSampler(torch.cuda.current_device()) as clocks:
        for _ in range(runs):
            reset()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
    st = B.pa_get_status()
    assert st == 0, st
    kv = 0
    for t in range(nsteps):
        n = wl.context_lens.astype(np.int64) + t + 1
        kv += int(n.sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    peak, kind = measured_peaks()
    gbs = kv * runs / (ms / 1e3) / 1e9
    res = {"workload": wl.name, "value": gbs, "unit": UNIT, "steps_per_run": nsteps,
           "runs": runs, "decode_tokens_per_s": wl.batch * nsteps * runs / (ms / 1e3),
           "frac_of_measured_copy_peak": gbs / peak,
           "frac_of_nominal_hbm_peak": gbs / NOMINAL_HBM_GBS,
           "ms_per_step": ms / (runs * nsteps), "partition_blocks": pb,
           "decode_kernel": kernel_name(B, B.pa_decode_kernel_choice(h, wl.num_heads)),
           "timing": "CUDA events around one graph replay per run (device allocation with "
                     "the length update a step ahead on a second stream, fused append+decode)",
           "clocks": clocks.summary()}
    B.pa_device_stack_download(h, stack)
    B.pa_pool_destroy(h)
    if _result is not None:
        _result["result"] = res
        return
    print(json.dumps({"row": "loop_device", **res}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--layers", type=int, default=0, help="layers per step (0 = all)")
    ap.add_argument("--workload", type=int, default=WORKLOAD_CFG, choices=[1, 2, 3, 4, 5],
                    help="named workload (default: the large-batch one, the headline)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every call from the host instead of replaying CUDA graphs")
    ap.add_argument("--row", choices=["step", "gather", "loop"], default="step",
                    help="step: append+decode per layer (headline); gather: pa_gather_kv "
                         "bandwidth; loop: the append+decode loop with block allocation")
    ap.add_argument("--cpu-seqs", type=int, default=256, help="sequences in the oracle sample")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate oracle time for the CPU baseline")
    ap.add_argument("--ref-seqs", type=int, default=96, help="sequences per reference step")
    ap.add_argument("--device-alloc", action="store_true",
                    help="with --row loop: free stack on the device, one CUDA graph per run")
    ap.add_argument("--separate", action="store_true",
                    help="step mode: pa_write_kv then pa_decode_attention per layer instead of "
                         "the fused pa_write_kv_and_decode (the default)")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="override the workload's KV heads (query heads unchanged): group-size "
                         "sweeps, e.g. --kv-heads 1 for one KV head per 32 query heads")
    ap.add_argument("--num-heads", type=int, default=0,
                    help="override the workload's query heads (with --kv-heads: any group, e.g. "
                         "--num-heads 64 --kv-heads 1 for the tcgen05 kernel)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads measured after the headline")
    ap.add_argument("--pool-layers", type=int, default=0,
                    help="build the pool with this many layers (0 = the workload's 32); "
                         "for small profiler captures, not for reported numbers")
    args = ap.parse_args()
    args.fused = not args.separate
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but {world} process(es): for N > 1 launch one "
                         f"process per GPU with torch.distributed.run (WORLD_SIZE = N)")
    if world > 1:
        import torch.distributed as dist

        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch

            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.row == "gather":
            run_gather(args, local_rank)
        elif args.row == "loop":
            run_loop(args, local_rank)
        else:
            run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
