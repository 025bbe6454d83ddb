#!/usr/bin/env python
"""Paged decode attention benchmark — prints one JSON line.

A step is one pass of the whole hot path over one decode batch: the host
block manager's slot assignment (done once; the workload is the same every
step, so each step rewrites the same slots), copy-on-write copies when the
batch has any, the append of every sequence's new K/V token, and paged decode
attention (with its split merge) over every cached token.

Default workload: 64 sequences with lengths U[128,2048] (+1 appended token),
32 query / 8 KV heads, head_dim 128, block 16, pool 1.25x the blocks needed
with shuffled physical ids, fp16 K/V/q drawn N(0,1) from a fixed seed.

value      KV GB/s: bytes of the K and V rows attended per step / device step
           time (CUDA events on the launching stream; between steps, outside
           the events, L2 is flushed by writing one 512 MB buffer and reading
           another, so no input and no dirty line is left in it)
e2e        the same metric through the public API with pinned host buffers:
           every step uploads q, new K/V, slot mapping, block table and
           lengths and downloads the output inside the timed region
roofline   the attention kernel alone: algorithmic bytes / mean launch time,
           against the measured HBM copy bandwidth
cpu_baseline  the fp64 CPU oracle, as it stands, on whole-batch passes

--impl reference times the CPU oracle instead (the only reference this
method has) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged decode attention: KV GB/s (fraction of GB300 HBM peak) and tokens attended/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20


def workload(name: str, seed_offset: int = 0):
    import synthetic
    if name == "gqa4_u128_2048":
        return synthetic.config2_gqa_batch(seed=2 + 1000 * seed_offset)
    if name == "mha32_lognormal800":
        return synthetic.config3_mha_lognormal(seed=3 + 1000 * seed_offset)
    if name == "shared_prefix_cow":
        return synthetic.config4_shared_prefix(seed=4 + 1000 * seed_offset)
    if name.startswith("long32k_gqa8_bs"):
        return synthetic.config5_long_context(block_size=int(name[len("long32k_gqa8_bs"):]),
                                              seed=5 + 1000 * seed_offset)
    raise SystemExit(f"unknown workload {name}")


def describe(b, kv_dtype: str = "fp16", lens=None) -> dict:
    lens = b.attended_lens if lens is None else np.asarray(lens)
    return {
        "workload": b.name,
        "num_seqs": int(b.num_seqs),
        "seq_len": f"{int(lens.min())}..{int(lens.max())} (mean {float(lens.mean()):.0f})",
        "tokens_attended": int(lens.sum()),
        "num_q_heads": b.num_q_heads,
        "num_kv_heads": b.num_kv_heads,
        "head_dim": b.head_dim,
        "block_size": b.block_size,
        "num_blocks": int(b.num_blocks),
        "kv_storage": "fp16" if kv_dtype == "fp16" else "fp8 e4m3 bytes, fp32 scale per KV head",
        "l2": "flushed between steps outside the timed events (512 MB write, then 512 MB read of another buffer)",
    }


def kv_bytes(b) -> int:
    return int(b.attended_lens.astype(np.int64).sum()) * b.num_kv_heads * b.head_dim * 2 * 2


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor rate, burst (a kernel timed alone); fp16 has the same
    nominal rate on this GPU."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def strip_c_comments(src: str) -> str:
    """C/C++ source with its comments removed and each run of whitespace
    collapsed to one space; string and character literals are kept whole."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


DECODE_SOURCES = ("pa_decode.cu", "pa_device.cuh")
PREFIX_SOURCES = ("pa_prefix.cu", "pa_device.cuh")


def kernel_source_hash(names=DECODE_SOURCES) -> str:
    """Identifies a kernel's code (comments and layout excluded), so that
    recorded ncu traffic is used only for the code it was taken on."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_40_gb300", "csrc", name),
                  encoding="utf-8") as f:
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str, sources=DECODE_SOURCES):
    """DRAM bytes per attention launch from a committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload_name)
    if not ent or ent.get("kernel_source_sha256_16") != kernel_source_hash(sources):
        return None
    return int(ent["dram_bytes_per_launch"])


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid.replace("GPU-", "").lower()
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[0].replace("GPU-", "").lower() == self.uuid:
                self.rows.append(parts)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------- distributed --
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def _reduce(x: float, world: int, op: str) -> float:
    """All-reduce one float over the ranks (on the GPU under NCCL, on the host
    under gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def reduce_max(x: float, world: int) -> float:
    return _reduce(x, world, "max")


def reduce_sum(x: float, world: int) -> float:
    return _reduce(x, world, "sum")


def aggregate(kv_bytes: int, tokens: int, steps: int, seconds: float, world: int):
    """Whole-job throughput of a weakly scaled run: every rank processed its
    own batch `steps` times in `seconds`; the job's time is the slowest
    rank's, its work the sum over ranks. Returns (KV GB/s, tokens/s, job
    seconds)."""
    t = reduce_max(seconds, world)
    kv = reduce_sum(float(kv_bytes) * steps, world)
    tok = reduce_sum(float(tokens) * steps, world)
    return kv / t / 1e9, tok / t, t


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------- CPU oracle --
def oracle_step_inputs(b):
    """(q, k_pool, v_pool, block_table, seq_lens) of the workload's decode
    step, from the oracle's own block manager."""
    import oracle
    if hasattr(b, "prefix_len"):
        # shared prefix: sequence 0 holds it, the others are forks; one step
        a = oracle.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
        a.add_seq(0, int(b.prefix_len))
        for c in range(1, b.num_seqs):
            a.fork(0, c)
        active = list(range(b.num_seqs))
        for s_ in active:
            a.append_slot(s_)
        mb = -(-(int(b.prefix_len) + 1) // b.block_size)
        table = np.asarray(a.dense_table(active, mb), np.int32)
        lens = np.full(b.num_seqs, int(b.prefix_len) + 1, np.int32)
        return b.step_inputs(0, b.num_seqs)[0], b.k_pool, b.v_pool, table, lens
    ref = oracle.decode_step(b, compute_attention=False)
    return b.q, ref.k_pool, ref.v_pool, ref.block_table, ref.seq_lens


def time_oracle(b, budget_s: float, max_seqs=None, fp8=None):
    """Time the CPU oracle's attention on whole-batch passes (or the first
    `max_seqs` sequences) until `budget_s` seconds have passed. With `fp8` (an
    E4M3 cache for the batch) the oracle's attention over that cache is timed."""
    import oracle
    q, kp, vp, table, seq_lens = oracle_step_inputs(b)
    seqs = list(range(b.num_seqs if max_seqs is None else min(max_seqs, b.num_seqs)))
    lens = np.asarray(seq_lens).astype(np.int64)
    esize = 1 if fp8 is not None else 2
    bytes_per_pass = int(lens[seqs].sum()) * b.num_kv_heads * b.head_dim * esize * 2
    tokens_per_pass = int(lens[seqs].sum())
    passes, t0 = 0, time.perf_counter()
    while True:
        if fp8 is not None:
            oracle.decode_attention_fp8(q, fp8.k_pool, fp8.v_pool, fp8.k_scale, fp8.v_scale,
                                        table, seq_lens, b.scale, seqs=seqs)
        else:
            oracle.decode_attention(q, kp, vp, table, seq_lens, b.scale, seqs=seqs)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"seconds": el, "passes": passes, "bytes": bytes_per_pass * passes,
            "tokens": tokens_per_pass * passes, "seqs": len(seqs)}


def run_reference(args, world, rank):
    if rank != 0:
        return
    b = workload(args.workload)
    fp8 = None
    if args.kv_dtype == "fp8":
        import synthetic
        fp8 = synthetic.fp8_cache(b)
    sample_seqs = args.ref_sample_seqs
    for _ in range(args.warmup):
        time_oracle(b, 0.0, max_seqs=sample_seqs, fp8=fp8)
    t_total, byt, tok = 0.0, 0, 0
    for _ in range(args.steps):
        r = time_oracle(b, 0.0, max_seqs=sample_seqs, fp8=fp8)
        t_total += r["seconds"]
        byt += r["bytes"]
        tok += r["tokens"]
    gbs = byt / t_total / 1e9
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(b, args.kv_dtype, oracle_step_inputs(b)[4]),
        "tokens_per_s": round(tok / t_total, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"first {sample_seqs} of {b.num_seqs} sequences, all heads, "
                                   f"attention only, per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- swapping --
def run_swap(args):
    """Swap half of the batch's sequences out to a pinned host pool and back
    in, each step: the block manager's pairs, then pa_swap_blocks each way."""
    import torch
    import paged_kv_cache_40_gb300 as pa
    from paged_kv_cache_40_gb300 import build as pa_build
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner

    pa_build.build()
    dev = torch.device("cuda", 0)
    b = workload(args.workload)
    run = DecodeBatchRunner(b, device=dev)
    run.plan_step()
    a = run.alloc
    a.add_host_pool(b.num_blocks)
    hk = torch.empty(tuple(run.k_pool.shape), dtype=run.k_pool.dtype).pin_memory()
    hv = torch.empty(tuple(run.v_pool.shape), dtype=run.v_pool.dtype).pin_memory()
    seqs = list(range(0, b.num_seqs, 2))
    stream = torch.cuda.current_stream(dev)
    block_bytes = run.k_pool[0].numel() * run.k_pool.element_size()

    def step(ev=None):
        t0 = time.perf_counter()
        out = [p for s_ in seqs for p in a.swap_out(s_)]
        t1 = time.perf_counter()
        po = torch.tensor(out, dtype=torch.int32).pin_memory()
        if ev:
            ev[0].record(stream)
        pa.pa_swap_blocks(run.k_pool, run.v_pool, hk, hv, po)
        if ev:
            ev[1].record(stream)
        t2 = time.perf_counter()
        back = [p for s_ in seqs for p in a.swap_in(s_)]
        t3 = time.perf_counter()
        pi = torch.tensor(back, dtype=torch.int32).pin_memory()
        pa.pa_swap_blocks(hk, hv, run.k_pool, run.v_pool, pi)
        if ev:
            ev[2].record(stream)
        return len(out), (t1 - t0) + (t3 - t2)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    host_s, nblk = 0.0, 0
    for k in range(K):
        nblk, hs = step(evs[k])
        host_s += hs
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    out_ms = [e[0].elapsed_time(e[1]) for e in evs]
    in_ms = [e[1].elapsed_time(e[2]) for e in evs]
    moved = nblk * block_bytes * 2
    gbs_out = moved / (statistics.mean(out_ms) / 1e3) / 1e9
    gbs_in = moved / (statistics.mean(in_ms) / 1e3) / 1e9
    print(json.dumps({
        "metric": "swap: K/V block bytes per second between the device pool and pinned host "
                  "memory (pa_swap_blocks)",
        "value": round(2 * moved / ((statistics.mean(out_ms) + statistics.mean(in_ms)) / 1e3) / 1e9,
                       2),
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "higher_is_better": True, "data": "synthetic",
        "config": {"workload": b.name, "sequences_swapped": len(seqs), "blocks_per_step": nblk,
                   "bytes_each_way": moved},
        "out_gbs": round(gbs_out, 2), "in_gbs": round(gbs_in, 2),
        "out_us": round(1e3 * statistics.mean(out_ms), 2),
        "in_us": round(1e3 * statistics.mean(in_ms), 2),
        "host_block_manager_us_per_step": round(1e6 * host_s / K, 1),
    }), flush=True)


# ------------------------------------------------- end to end with planning --
def time_planned(args, b, fp8, dev, stream, flush, world, steps):
    """Decode steps whose timed region includes the host block manager.

    serial: per step, with the stream idle, an event, then the step planned
    (pa_alloc_plan_step into pinned host memory), its kernels launched and a
    second event: planning, launch and the kernels, one after the other;
    L2 flushed between steps outside the events.
    overlap: steps back to back with no wait, step k+1 planned on the host
    while the kernels of step k run (two rotating sets of plan buffers); one
    event before the first step and one after the last. Inputs (the K/V the
    steps read) are larger than L2, which is not flushed in this loop.
    Both report KV GB/s over the bytes the steps actually attended (the
    sequences grow by one token a step)."""
    import torch
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    # the tokens every sequence may grow by in the batch's pool, and the
    # steps of each loop that fit (both loops and their warm-up grow them)
    bs = b.block_size
    lens0 = [int(L) for L in b.prefill_lens]
    free = int(b.num_blocks) - sum(-(-L // bs) for L in lens0)
    grow = 0
    while sum(-(-(L + grow + 1) // bs) - -(-L // bs) for L in lens0) <= free:
        grow += 1
    steps = min(steps, grow // 2 - args.warmup)
    if steps < 10:
        return {"skipped": f"the pool leaves room for {grow} more tokens per sequence"}
    mb = int(max(-(-(L + grow) // bs) for L in lens0))
    kw = dict(device=dev, partition_tokens=args.partition, layout=args.layout, max_blocks=mb)
    if fp8 is not None:
        kw.update(kv_dtype="fp8", k_pool=fp8.k_pool, v_pool=fp8.v_pool, k_scale=fp8.k_scale,
                  v_scale=fp8.v_scale)
    run = DecodeBatchRunner(b, **kw)
    h2d = run.host_planned(sets=2)
    out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
    run.out = out_h
    esize = 1 if fp8 is not None else 2
    per_tok = b.num_kv_heads * b.head_dim * esize * 2
    # pa_decode_step / pa_decode_step_fp8: plan, copies, append, attention in
    # one library call per step
    run.prepare_native_steps(stream)

    def one():
        plan = run.run_native_step()
        return int(plan.seq_lens.astype(np.int64).sum())

    # a set of plan buffers is rewritten two steps after the step that read
    # it: that step must have completed (the flush makes the device the slow
    # side, so without the wait the host would plan over a set still queued)
    for _ in range(args.warmup):
        flush()
        torch.cuda.synchronize(dev)
        one()
    torch.cuda.synchronize(dev)
    barrier(world)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    toks, host_s = 0, 0.0
    for k in range(steps):
        flush()
        torch.cuda.synchronize(dev)
        ev[k][0].record(stream)
        t0 = time.perf_counter()
        toks += one()
        host_s += time.perf_counter() - t0
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    serial_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    serial_gbs, _, t_serial = aggregate(toks * per_tok, 0, 1, sum(serial_ms) / 1e3, world)
    # overlapped: plan k+1 while step k runs; a set of plan buffers is reused
    # only after the step that read it has completed
    done = [torch.cuda.Event() for _ in range(steps)]
    flush()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    toks_o = 0
    e0.record(stream)
    for k in range(steps):
        if k >= 2:
            done[k - 2].synchronize()
        toks_o += one()
        done[k].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    over_ms = e0.elapsed_time(e1)
    over_gbs, _, t_over = aggregate(toks_o * per_tok, 0, 1, over_ms / 1e3, world)
    import paged_kv_cache_40_gb300 as pa
    assert pa.pa_device_error() == 0
    d2h = out_h.numel() * out_h.element_size()
    return {
        "call": ("pa_decode_step_fp8" if fp8 is not None else "pa_decode_step")
                + " (one library call per step)",
        "value": round(serial_gbs, 2), "unit": "GB/s", "steps": steps,
        "ms_per_step": round(1e3 * t_serial / steps, 5),
        "host_plan_and_launch_us_per_step": round(1e6 * host_s / steps, 2),
        "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
        "path": "per step with the stream idle: block-manager plan (one call) into pinned host "
                "memory, then the step's kernels reading it in place; events around both; L2 "
                "flushed between steps outside the events",
        "overlap": {"value": round(over_gbs, 2), "unit": "GB/s",
                    "ms_per_step": round(1e3 * t_over / steps, 5),
                    "path": "steps back to back, step k+1 planned while step k runs (two sets "
                            "of plan buffers); events around the whole loop; no L2 flush "
                            "(the K/V read per step exceed L2)"},
    }


# ----------------------------------------------------------------- our arm --
def run_ours(args, world, rank, local):
    import torch
    import paged_kv_cache_40_gb300 as pa
    from paged_kv_cache_40_gb300 import build as pa_build
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner

    pa_build.build()
    pa.lib()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for the libpa arm")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    b = workload(args.workload, seed_offset=rank)
    fp8 = None
    shared = args.workload == "shared_prefix_cow"
    if shared:
        from paged_kv_cache_40_gb300.engine import SharedPrefixRunner
        if args.kv_dtype != "fp16":
            raise SystemExit("the shared-prefix step is measured on an fp16 cache")
        run = SharedPrefixRunner(b, device=dev, partition_tokens=args.partition,
                                 prefix_aware=not args.plain_decode, layout=args.layout)
    elif args.kv_dtype == "fp8":
        import synthetic
        fp8 = synthetic.fp8_cache(b, seed=100 + 1000 * rank)
        run = DecodeBatchRunner(b, device=dev, partition_tokens=args.partition, kv_dtype="fp8",
                                k_pool=fp8.k_pool, v_pool=fp8.v_pool, k_scale=fp8.k_scale,
                                v_scale=fp8.v_scale, layout=args.layout)
    else:
        run = DecodeBatchRunner(b, device=dev, partition_tokens=args.partition,
                                layout=args.layout)
    plan = run.plan_step()
    # host slot assignment (block manager) cost for this batch, measured on a
    # second allocator holding the same placement
    from paged_kv_cache_40_gb300 import BlockAllocator
    a = BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    if shared:
        a.add_seq(0, int(b.prefix_len))
        for c in range(1, b.num_seqs):
            a.fork(0, c)
    else:
        for op in b.churn:
            if op.kind == "alloc":
                a.add_seq(op.owner, op.nblocks * b.block_size)
            else:
                a.free_seq(op.owner)
        for i in range(b.num_seqs):
            a.add_seq(i, int(b.prefill_lens[i]))
    # the binding's first-call costs (imports, ctypes set-up) are paid by calls
    # that change no state: an empty batch and a table build
    ids = np.arange(b.num_seqs, dtype=np.int64)
    width = run.max_blocks + 2 + 11 // b.block_size  # room for eleven more tokens
    bufs = (np.empty(b.num_seqs, np.int32), np.empty((b.num_seqs, 2), np.int32),
            np.empty((b.num_seqs, width), np.int32), np.empty(b.num_seqs, np.int32))
    a.plan_step(ids[:0], width, out=bufs)
    host_us = []
    for _ in range(11):  # the step above, then ten more (the sequences grow)
        t_host0 = time.perf_counter()
        a.plan_step(ids, width, out=bufs)       # one call: slots, copy pairs, tables, lengths
        host_us.append((time.perf_counter() - t_host0) * 1e6)
    t_host_first, t_host = host_us[0], statistics.median(host_us[1:])
    a.close()
    stream = torch.cuda.current_stream(dev)
    # L2 flush between steps: write one buffer larger than L2, then read a
    # second one, so the timed step starts with L2 holding neither its inputs
    # nor dirty lines whose write-back it would pay for.
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # float32 so the reduction reads the buffer once (an int32 sum would first
    # convert the whole buffer to int64)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        flush_w.fill_(1)
        torch.sum(flush_r, dim=0, out=flush_sink)

    for _ in range(args.warmup):
        flush()
        run.run_step()
    torch.cuda.synchronize(dev)
    assert pa.pa_device_error() == 0

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(str(torch.cuda.get_device_properties(dev).uuid))
    sampler.start()
    time.sleep(0.15)
    barrier(world)
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    launches0 = pa.pa_kernel_launches()
    # the step as a caller issues it (DecodeBatchRunner.step): the copies if
    # any, then for an fp16 cache one kernel that appends the new rows and
    # attends (pa_decode_append_attention); for an E4M3 cache the append,
    # then the attention kernel as a programmatic dependent of it; for the
    # shared-prefix workload the copies, the append and the prefix-aware call
    for k in range(K):
        flush()
        ev[k][0].record(stream)
        run.step()
        ev[k][1].record(stream)
    launches = pa.pa_kernel_launches() - launches0
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - w0
    clocks = sampler.stop()
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    assert pa.pa_device_error() == 0
    # the attention call alone (the roofline's kernel), same number of steps
    eva = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for k in range(K):
        flush()
        eva[k][0].record(stream)
        run.attend()
        eva[k][1].record(stream)
    torch.cuda.synchronize(dev)
    attn_ms = [eva[k][0].elapsed_time(eva[k][1]) for k in range(K)]
    assert pa.pa_device_error() == 0

    # end to end through the public API with host memory, both ways the API
    # offers; each timed step moves the step's inputs (q, new K/V rows, slots,
    # copy pairs, table, lengths) from pinned host memory to the GPU and its
    # result back:
    #  - upload: the inputs packed in one pinned buffer go up with one copy
    #    (DecodeBatchRunner.pack_inputs / upload_inputs);
    #  - host (reported as e2e): the inputs stay in pinned host memory and
    #    the kernels read them through its device mapping over NVLink-C2C
    #    (host_inputs), no copy call.
    # Either way the attention kernel writes the result into pinned host
    # memory through its device mapping.
    out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
    dev_out = run.out
    run.out = out_h
    d2h = out_h.numel() * out_h.element_size()
    Ke = max(1, min(K, args.e2e_steps))

    def time_e2e(e2e_step):
        for _ in range(args.warmup):
            flush()
            e2e_step()
        torch.cuda.synchronize(dev)
        eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
        barrier(world)
        for k in range(Ke):
            flush()
            eev[k][0].record(stream)
            e2e_step()
            eev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        assert pa.pa_device_error() == 0
        return [eev[k][0].elapsed_time(eev[k][1]) for k in range(Ke)]

    run.pack_inputs()
    h2d_up = int(run.host_arena.numel())
    e2e_up_ms = time_e2e(lambda: (run.upload_inputs(), run.run_step()))
    h2d = run.host_inputs()
    e2e_ms = time_e2e(run.run_step)
    run.out = dev_out

    # end to end with the block manager inside the timed region: a decode
    # loop on a second copy of the batch whose sequences grow by one token a
    # step; each step is planned by one block-manager call straight into
    # pinned host memory, which the kernels read in place
    planned = None
    if not shared:
        planned = time_planned(args, b, fp8, dev, stream, flush, world, Ke)

    kvb = run.kv_bytes()
    tokens = int(plan.seq_lens.astype(np.int64).sum())
    value, tok_per_s, t_steps = aggregate(kvb, tokens, K, sum(step_ms) / 1e3, world)
    value_e2e, _, t_e2e = aggregate(kvb, tokens, Ke, sum(e2e_ms) / 1e3, world)
    value_up, _, t_up = aggregate(kvb, tokens, Ke, sum(e2e_up_ms) / 1e3, world)
    attn_mean_s = statistics.mean(attn_ms) / 1e3
    peak, peak_kind = hbm_peak()
    achieved = run.io_bytes() / attn_mean_s / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle(b, args.cpu_budget, fp8=fp8)
        cpu = {"value": round(r["bytes"] / r["seconds"] / 1e9, 4), "unit": "GB/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{r['passes']} whole-batch pass(es) of the same {b.num_seqs}-sequence "
                         f"batch, attention only, fp64 numpy, BLAS default threads",
               "tokens_per_s": round(r["tokens"] / r["seconds"], 1)}
    if rank != 0:
        return
    config = describe(b, args.kv_dtype, plan.seq_lens)
    if args.layout == "records":
        config["pool_layout"] = ("one pool of per-block records (K rows then V rows), "
                                 "block stride two blocks")
    if shared:
        config.update({
            "prefix_len": int(b.prefix_len),
            "cow_copies_per_step": int(len(plan.cow_pairs)),
            "attention": "prefix-aware (prefix blocks read once per KV head for all sequences)"
                         if run.prefix_aware else "generic paged decode",
            "unique_kv_bytes": run.unique_kv_bytes(),
            "note": "every sequence attends the same 2040-token prefix; bytes are logical "
                    "(per sequence), the prefix's blocks are served from L2 after the first read",
        })
    if shared and run.prefix_aware:
        # one launch of the prefix kernel (every suffix is short): its
        # contraction runs on the tensor cores and it reads the prefix once,
        # so the tensor roof bounds it, not HBM
        flops = run.prefix_flops()
        tpeak, tpeak_kind = tensor_peak()
        tf = flops / attn_mean_s / 1e12
        roofline = {"bound": "tensor", "achieved": round(tf, 2), "peak": tpeak,
                    "unit": "TFLOP/s", "frac": round(tf / tpeak, 4),
                    "traffic": recorded_traffic(b.name, PREFIX_SOURCES),
                    "peak_source": tpeak_kind + " (dense bf16 burst; fp16 has the same rate)",
                    "kernel": "paged_prefix_kernel", "flops_per_launch": flops,
                    "hbm_logical": {"achieved": round(achieved, 1), "peak": peak,
                                    "unit": "GB/s", "bytes_per_launch": run.io_bytes(),
                                    "note": "logical per-sequence bytes; the prefix is read "
                                            "once, so this is not a DRAM rate"}}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": recorded_traffic(b.name + ("_fp8" if fp8 is not None else "")
                                                + ("_records" if args.layout == "records"
                                                   else "")),
                    "peak_source": peak_kind,
                    "kernel": "paged_decode_kernel",
                    "bytes_per_launch": run.io_bytes()}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(1e3 * t_steps / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": config,
        "tokens_per_s": round(tok_per_s, 1),
        "frac_of_hbm_peak": {"measured": round(value / peak, 4),
                             "nominal_8tbs": round(value / 8000.0, 4)},
        "attention_us": {"mean": round(1e6 * attn_mean_s, 3),
                         "median": round(1e3 * statistics.median(attn_ms), 3),
                         "min": round(1e3 * min(attn_ms), 3)},
        "roofline": roofline,
        "e2e_planned": planned,
        "e2e": {"value": round(value_e2e, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(1e3 * t_e2e / Ke, 5), "steps": Ke,
                "path": "inputs in pinned host memory, read by the kernels over NVLink-C2C; "
                        "output written by the attention kernel into pinned host memory",
                "upload_path": {"value": round(value_up, 2), "unit": "GB/s",
                                "ms_per_step": round(1e3 * t_up / Ke, 5),
                                "h2d_bytes_per_step": h2d_up,
                                "path": "inputs packed in one pinned buffer, one host-to-device "
                                        "copy per step; output as above"}},
        "cpu_baseline": cpu,
        "gpu_launches": launches,
        "clocks": clocks,
        "host_slot_assign_us": round(t_host, 1) if t_host is not None else None,
        "host_slot_assign_first_us": (round(t_host_first, 1) if t_host_first is not None
                                      else None),
        "wall_s_timed_region": round(wall, 4),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa4_u128_2048")
    ap.add_argument("--partition", type=int, default=0, help="tokens per split (0 = default)")
    ap.add_argument("--op", choices=["decode", "swap"], default="decode",
                    help="decode: the decode step (default); swap: swapping throughput")
    ap.add_argument("--plain-decode", action="store_true",
                    help="shared-prefix workload: attend with the generic call, not the "
                         "prefix-aware one")
    ap.add_argument("--kv-dtype", choices=["fp16", "fp8"], default="fp16",
                    help="KV cache storage: fp16, or E4M3 bytes with per-head scales")
    ap.add_argument("--layout", choices=["separate", "records"], default="separate",
                    help="KV pools: two separate pools, or one pool of per-block K/V records")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-sample-seqs", type=int, default=4)
    args = ap.parse_args()
    world, rank, local = dist_setup(args)
    if args.op == "swap" and args.impl != "reference":
        if rank == 0:
            run_swap(args)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
