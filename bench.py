"""Benchmark: paged decode attention KV GB/s (% of HBM peak) and decode tokens/s.

Workload: the large-batch decode workload -- batch 256, 32 query heads / 8 KV
heads, head_dim 128, block 16, 32 layers, context lengths U[128, 4096],
physical blocks interleaved across sequences, bf16 pool of about 71 GB.

One step = one decode step of the whole model's attention: for each of the 32
layers, append the new token's K/V (pa_write_kv, into the last context slot) and
run pa_decode_attention over the context (split-K + combine when partitioned).
Each layer reads ~2.2 GB of K/V, far more than the 129 MB L2, so no flush is
needed between steps.

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


def decode_flops(wl) -> int:
    return int(wl.context_lens.astype(np.int64).sum()) * 4 * wl.num_heads * wl.head_dim


# DRAM bytes (read + write) of one pa_decode_kernel launch on this workload,
# from `ncu --set full` (profiles/pa_decode_kernel__large_batch_*.md), valid only
# for the kernel sources they were taken from.
DECODE_TRAFFIC = {
    "bytes_per_launch": 2223014000 + 6228480,
    "sources_sha256": "d472b81370cc6a2abb2460c285814a52cd86a657cb4dfc3aef8672e6c3a4cbce",
}
DECODE_SOURCES = ["pa_decode.cuh", "pa_decode_launch.cuh", "pa_decode_bf16.cu", "pa_device.cuh"]


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
    wl = W.named(WORKLOAD_CFG)
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
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    outs = torch.empty((L, wl.batch, wl.num_heads, wl.head_dim), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    lib = B.lib()
    cmax = -(-wl.max_blocks // pb)
    launches_per_step = L * (2 + (1 if cmax > 1 else 0))

    def layer_call(l, ev=None):
        rc = lib.pa_write_kv(h, l, ks[l].data_ptr(), vs[l].data_ptr(), bt.data_ptr(),
                             wl.max_blocks, positions.data_ptr(), wl.batch, sp)
        if rc:
            raise RuntimeError(B.last_error())
        if ev is not None:
            ev[0].record(stream)
        rc = lib.pa_decode_attention(outs[l].data_ptr(), qs[l].data_ptr(), h, l, bt.data_ptr(),
                                     wl.max_blocks, lens.data_ptr(), wl.batch, wl.block_size,
                                     wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.scale,
                                     ws.data_ptr(), ws_bytes, sp)
        if rc:
            raise RuntimeError(B.last_error())
        if ev is not None:
            ev[1].record(stream)

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

    # ---- timed region: device-resident inputs ----
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(L)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        t_start.record(stream)
        for s in range(args.steps):
            for l in range(L):
                layer_call(l, evs[s][l])
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    call_ms = [a.elapsed_time(b) for row in evs for (a, b) in row]
    st = B.pa_get_status()
    if st:
        raise RuntimeError(f"device status {st:#x} after the timed region")

    # ---- end to end through the C ABI: inputs from pinned host memory ----
    e2e_ms, h2d, d2h = float("nan"), 0, 0
    if not args.no_e2e:
        q_h = qs.cpu().pin_memory()
        k_h = ks.cpu().pin_memory()
        v_h = vs.cpu().pin_memory()
        bt_h = bt.cpu().pin_memory()
        lens_h = lens.cpu().pin_memory()
        pos_h = positions.cpu().pin_memory()
        out_h = torch.empty(outs.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h, bt_h, lens_h, pos_h))
        d2h = out_h.numel() * out_h.element_size()

        def e2e_step():
            qs.copy_(q_h, non_blocking=True)
            ks.copy_(k_h, non_blocking=True)
            vs.copy_(v_h, non_blocking=True)
            bt.copy_(bt_h, non_blocking=True)
            lens.copy_(lens_h, non_blocking=True)
            positions.copy_(pos_h, non_blocking=True)
            for l in range(L):
                layer_call(l)
            out_h.copy_(outs, non_blocking=True)

        for _ in range(max(1, args.warmup // 2)):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
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
    steps = args.steps
    value = per_call * L * steps * world / (total_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    call_avg_ms = sum(call_ms) / len(call_ms)
    achieved = per_call / (call_avg_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "num_layers": L,
            "context_lens": f"U[128,4096] seed {wl.seed}, mean {wl.context_lens.mean():.0f}",
            "pool_gb": round(wl.pool_bytes() / 1e9, 1), "partition_blocks": pb,
            "l2": "inputs larger than L2 (2.2 GB of K/V per layer vs 129 MB L2), no flush",
            "parallelism": f"replicas x{world}",
        },
        "pct_hbm_peak": 100.0 * value / peak,
        "decode_tokens_per_s": wl.batch * steps * world / (total_ms / 1e3),
        "roofline": {"bound": "hbm", "kernel": "pa_decode_attention (decode + combine)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs", "traffic": decode_traffic(),
                     "traffic_kernel": "pa_decode_kernel (ncu dram read+write per launch)",
                     "algorithmic_bytes_per_call": per_call,
                     "avg_call_ms": call_avg_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": per_call * L * steps * world / (e2e_ms / 1e3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / steps},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    B.pa_pool_destroy(h)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--layers", type=int, default=0, help="layers per step (0 = all 32)")
    ap.add_argument("--cpu-seqs", type=int, default=256, help="sequences in the oracle sample")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate oracle time for the CPU baseline")
    ap.add_argument("--ref-seqs", type=int, default=96, help="sequences per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--pool-layers", type=int, default=0,
                    help="build the pool with this many layers (0 = the workload's 32); "
                         "for small profiler captures, not for reported numbers")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
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
        else:
            run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
