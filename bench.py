"""Benchmark of one paged decode step on GB300 (driver contract: one JSON line).

A step is the whole hot path over one batch: pa_reshape_and_cache of the new
token of every sequence, then pa_decode (decode kernel + merge kernel), on
the Llama-3-8B-shaped workload (batch 64, 32 q / 8 kv heads, head_dim 128,
block_size 16, bf16, seq_lens uniform [512, 4096], shuffled blocks).

value  : algorithmic HBM GB/s of the step (bytes the step must move / device
         time per step), whole job (all ranks' bytes / slowest rank's time).
e2e    : the same metric through the public API with host buffers: q, k/v of
         the new tokens, slots, block tables and seq_lens sit in pinned host
         memory and the output goes to pinned host memory; the library's
         kernels read and write them in place over the CPU-GPU link (no copy
         engine), all inside the timed region. The same step with one packed
         H2D copy and one D2H copy is reported beside it (copy_engine).
roofline: the decode kernel alone (CUDA events around it on its stream).
cpu_baseline: the fp64 C oracle on this host's cores.

--config picks another named workload; the chunk workloads (num_queries > 1)
time pa_reshape_and_cache of the B * T new tokens + pa_prefill_chunk, with the
same byte model (each K/V row of a sequence's read range counted once).

--impl reference times the oracle (the CPU reference of this build) on a
bounded sample of the same workload with the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import generate, get_config  # noqa: E402

METRIC = "paged decode attention: μs/step, achieved HBM GB/s and % of GB300 peak"
# the other seeded decode workloads, reported beside the main one
DEFAULT_EXTRA_CONFIGS = "long_skew,fp8,prefix_window,tiny"
UNIT = "GB/s"


# ----------------------------------------------------------- byte models

def decode_bytes(w) -> dict:
    """Algorithmic bytes of one pa_decode (or pa_prefill_chunk): every K/V row
    of each sequence's read range once, q, out, the block-table entries of
    the touched blocks and seq_lens."""
    s = w.spec
    L = w.seq_lens.astype(np.int64)
    st = w.starts.astype(np.int64)
    n = L - st
    elt = 1 if s.kv_fp8 else 2
    kv = int(n.sum()) * s.num_kv_heads * 2 * s.head_dim * elt
    blocks = np.where(L > 0, -(-L // s.block_size) - st // s.block_size, 0)
    q = s.batch * s.num_queries * s.num_q_heads * s.head_dim * 2
    tables = 4 * int(blocks.sum()) + 4 * s.batch
    return {"kv": kv, "q": q, "out": q, "tables": tables,
            "kernel": kv + q + tables, "total": kv + 2 * q + tables,
            "tokens": int(n.sum())}


def attention_flops(w) -> float:
    """Algorithmic FLOPs of the attention: 2 D for q.k and 2 D for p.v per
    attended (query, q head, position); query t of a chunk attends to
    [max(0, p + 1 - W), p], p = L - T + t."""
    s = w.spec
    T, W = s.num_queries, s.window
    total = 0
    for L in w.seq_lens.astype(np.int64):
        p = L - T + np.arange(T)
        lo = np.where((W > 0) & (p + 1 > W), p + 1 - W, 0)
        total += int(np.where(p >= 0, p + 1 - lo, 0).sum())
    return 4.0 * s.head_dim * s.num_q_heads * total


def reshape_bytes(w) -> int:
    s = w.spec
    T = int((w.slot_new >= 0).sum().item())
    elt = 1 if s.kv_fp8 else 2
    per_row = s.num_kv_heads * s.head_dim
    return T * per_row * 2 * 2 + T * per_row * elt * 2 + 8 * w.slot_new.numel()


# ----------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- helpers

def measured_tensor_peak() -> tuple[float, str]:
    """Dense bf16 TFLOP/s (burst) measured on this machine, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the sources that make up the decode kernel (its code, the
    PTX wrappers, the step plan and the argument structs), comments and
    whitespace left out so that a change of wording keeps the profiles."""
    h = hashlib.sha256()
    for f in ("decode.cuh", "ptx.cuh", "plan.cuh", "pa_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_267_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)  # block comments
        src = re.sub(r"//[^\n]*", " ", src)                # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(config: str, decode_launch_bytes: float):
    """dram bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"decode_{config}_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def relaunch_under_torchrun(n_gpus: int) -> None:
    """`--gpus N` (N > 1) started without a launcher: run this same command
    as N processes under torch.distributed.run on this node (one per GPU),
    and exit with its status. Never runs one rank silently."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n_gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    sys.stdout.flush()
    sys.exit(subprocess.call(cmd))


def dist_setup(n_gpus: int):
    """Rank layout from the launcher's environment. With no launcher and
    `--gpus N > 1` the caller relaunches under torch.distributed.run first; a
    launcher whose world size differs from `--gpus` is an error."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if "WORLD_SIZE" in os.environ and world != n_gpus:
        raise SystemExit(f"bench.py: --gpus {n_gpus} but the launcher started {world} ranks")
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_spec(config: str, rank: int):
    """Each rank decodes its own batch (weak scaling): same shape, own seed."""
    s = get_config(config)
    return s.with_(seed=s.seed + 1000 * rank) if rank else s


# ----------------------------------------------------------- oracle timing

def oracle_baseline(w, kc_host, vc_host, budget_s: float, seq_subset=None,
                    queries=None) -> dict:
    """Times the oracle on sequences `seq_subset` (default all) and, for a
    chunk, query positions `queries` of each (default all), all heads. The
    bytes are the step's algorithmic bytes for that share: each sequence's
    K/V read range once, scaled by the share of its queries computed, plus q
    and out of the computed rows."""
    import oracle
    s = w.spec
    B = s.batch
    seqs = list(range(B)) if seq_subset is None else list(seq_subset)
    T = s.num_queries
    ts = list(range(T)) if queries is None else list(queries)
    pairs = np.array([(b, h) for b in seqs for h in range(s.num_q_heads)], np.int32)
    triples = np.array([(b, t, h) for b in seqs for t in ts
                        for h in range(s.num_q_heads)], np.int32)
    sel = np.zeros(B, bool)
    sel[seqs] = True
    L = w.seq_lens.astype(np.int64)
    n = (L - w.starts)[sel]
    elt = 1 if s.kv_fp8 else 2
    bytes_ = (int(n.sum()) * s.num_kv_heads * 2 * s.head_dim * elt * len(ts) / T
              + 2 * len(triples) * s.head_dim * 2)
    threads = oracle.default_threads()
    qh = w.q.cpu()
    reps, t0 = 0, time.perf_counter()
    kw = dict(num_kv_heads=s.num_kv_heads, scale=s.softmax_scale, block_size=s.block_size,
              window=s.window, q_dtype=s.dtype, cache_dtype="fp8" if s.kv_fp8 else s.dtype,
              k_scale=w.k_scale, v_scale=w.v_scale, threads=threads)
    while True:
        if T == 1:
            oracle.decode(qh, kc_host, vc_host, w.block_tables, w.seq_lens, pairs=pairs, **kw)
        else:
            oracle.decode_multi(qh, kc_host, vc_host, w.block_tables, w.seq_lens,
                                triples=triples, **kw)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    per = el / reps
    return {"value": bytes_ / per / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "seconds_per_sample": per,
            "sample": f"fp64 C oracle decode of {len(seqs)} of {B} sequences x "
                      f"{len(ts)} of {T} queries x {s.num_q_heads} heads ({int(n.sum())} "
                      f"tokens in the read ranges), {reps} run(s)"}


def bounded_sample(w, kc_host, vc_host, budget_s: float):
    """(sequences, queries) whose oracle run takes about `budget_s` or less:
    whole sequences while they fit, else evenly spaced query positions of the
    first sequence (a chunk's queries are independent rows)."""
    s = w.spec
    T = s.num_queries
    probe = oracle_baseline(w, kc_host, vc_host, 0.0, seq_subset=[0], queries=[T - 1])
    per_query = max(probe["seconds_per_sample"], 1e-6)  # the longest row of sequence 0
    per_seq = per_query * T
    if per_seq <= budget_s:
        nseq = int(max(1, min(s.batch, budget_s / per_seq)))
        return list(range(nseq)), None
    nq = int(max(1, min(T, budget_s / per_query)))
    if nq == 1:
        return [0], [(T - 1) // 2]  # the middle row: a chunk's rows grow with t
    return [0], sorted({int(round(i * (T - 1) / (nq - 1))) for i in range(nq)})


def host_caches(w, kc, vc):
    def h(t):
        t = t.cpu().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16):
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return h(kc), h(vc)


# ----------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    from oracle.build import build_oracle
    import oracle
    build_oracle()
    w = generate(rank_spec(args.config, 0), device="cpu")
    s = w.spec
    if s.kv_fp8:
        from workloads.gen import E4M3_NAN
        shape = (w.num_blocks, s.num_kv_heads, s.block_size, s.head_dim)
        kc = np.full(shape, E4M3_NAN, np.uint8)
        vc = np.full(shape, E4M3_NAN, np.uint8)
        oracle.reshape_and_cache(w.k_hist, w.v_hist, kc, vc, w.slot_hist.numpy(), s.dtype, "fp8",
                                 w.k_scale, w.v_scale)
    else:
        kc, vc = host_caches(w, w.key_cache, w.value_cache)
    oracle.reshape_and_cache(w.k_new, w.v_new, kc, vc, w.slot_new.numpy(), s.dtype,
                             "fp8" if s.kv_fp8 else s.dtype, w.k_scale, w.v_scale)
    # bounded sample per step, sized so the whole run stays short
    total_budget = 120.0
    per_step = max(0.01, total_budget / max(1, args.steps + args.warmup))
    subset, queries = bounded_sample(w, kc, vc, per_step)
    nseq = len(subset)
    for _ in range(args.warmup):
        oracle_baseline(w, kc, vc, 0.0, subset, queries)
    times, vals = [], []
    for _ in range(args.steps):
        r = oracle_baseline(w, kc, vc, 0.0, subset, queries)
        times.append(r["seconds_per_sample"])
        vals.append(r["value"])
    ms = 1e3 * statistics.mean(times)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.config}: {workload_desc(s)}",
                       "sample_per_step": (f"{nseq} of {s.batch} sequences, all heads" if queries is None
                                           else f"{len(queries)} of {s.num_queries} queries of "
                                                f"sequence 0, all heads")},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": r["cores"],
                             "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_desc(s) -> str:
    d = (f"batch {s.batch}, {s.num_q_heads} q / {s.num_kv_heads} kv heads, head_dim "
         f"{s.head_dim}, block_size {s.block_size}, {s.dtype}")
    if s.kv_fp8:
        d += ", e4m3 KV"
    if s.window:
        d += f", window {s.window}"
    if s.shared_prefix:
        d += f", shared prefix {s.shared_prefix}"
    if s.num_queries > 1:
        d += f", {s.num_queries} causal queries per sequence"
    return d


# ----------------------------------------------------------- our arm

def unique_kv_bytes(w) -> int:
    """K/V bytes of the distinct cache rows the step reads: a physical slot
    read by several sequences (a shared prefix block) counts once."""
    s = w.spec
    L = w.seq_lens.astype(np.int64)
    st = w.starts.astype(np.int64)
    slots = []
    for b in range(s.batch):
        if L[b] <= st[b]:
            continue
        pos = np.arange(st[b], L[b], dtype=np.int64)
        slots.append(w.block_tables[b, pos // s.block_size].astype(np.int64) * s.block_size
                     + pos % s.block_size)
    n = int(np.unique(np.concatenate(slots)).size) if slots else 0
    elt = 1 if s.kv_fp8 else 2
    return n * s.num_kv_heads * 2 * s.head_dim * elt


class StepCtx:
    """One named workload on the device, ready to step: the write path of its
    new tokens, then pa_decode (or pa_prefill_chunk for a chunk)."""

    def __init__(self, pa, name: str, rank: int, dev):
        self.pa = pa
        self.name = name
        w = generate(rank_spec(name, rank), device=dev)
        s = w.spec
        self.w, self.s = w, s
        self.kv = "fp8" if s.kv_fp8 else "auto"
        if s.kv_fp8:
            self.kc, self.vc = w.empty_fp8_cache()
            pa.reshape_and_cache(w.k_hist, w.v_hist, self.kc, self.vc, w.slot_hist, self.kv,
                                 w.k_scale, w.v_scale)
            w.k_hist = w.v_hist = w.slot_hist = None
        else:
            self.kc, self.vc = w.key_cache, w.value_cache
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.sl = torch.from_numpy(w.seq_lens).to(dev)
        self.out = torch.empty_like(w.q)
        self.kw = dict(num_kv_heads=s.num_kv_heads, scale=s.softmax_scale,
                       block_size=s.block_size, window=s.window, kv_dtype=self.kv,
                       k_scale=w.k_scale, v_scale=w.v_scale, out=self.out)
        self.attend = pa.decode if s.num_queries == 1 else pa.prefill_chunk
        self.dbytes = decode_bytes(w)
        self.rbytes = reshape_bytes(w)
        self.step_bytes = self.dbytes["total"] + self.rbytes

    def step(self):
        w = self.w
        self.pa.reshape_and_cache(w.k_new, w.v_new, self.kc, self.vc, w.slot_new, self.kv,
                                  w.k_scale, w.v_scale)
        self.attend(w.q, self.kc, self.vc, self.bt, self.sl, **self.kw)

    def attend_only(self):
        self.attend(self.w.q, self.kc, self.vc, self.bt, self.sl, **self.kw)


class L2Flush:
    """Write a buffer four times the L2 size (evicts every line), then read
    another one as large, so the timed step starts with a cold L2 that holds
    no dirty lines whose write-back would land inside the timed region (with
    only twice the L2 size some dirty lines survived and slowed the next step
    measurably)."""

    def __init__(self, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(4 * l2, 512 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.r = torch.ones(n // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


# The device is held by a bounded spin kernel (torch.cuda._sleep) while the
# host enqueues the timed iterations: 500,000 cycles (about 250 us at 2 GHz)
# per iteration, several times what the host takes to enqueue one (the L2
# flush, two events, the step's launches). Without it, the first iteration
# after an idle spell sometimes waited inside its events for the host's
# launches (one step of 231 us among steps of 114 us).
SPIN_CYCLES_PER_ITER = 500_000
QUEUE_CHUNK = 32


def queued(n: int, enqueue) -> None:
    """Enqueue iterations 0..n-1 (enqueue(i) issues one) in chunks, each
    behind a spin long enough for the host to enqueue the whole chunk, so
    that CUDA events around an iteration time the device's work alone."""
    for c0 in range(0, n, QUEUE_CHUNK):
        c1 = min(n, c0 + QUEUE_CHUNK)
        torch.cuda._sleep(SPIN_CYCLES_PER_ITER * (c1 - c0))
        for i in range(c0, c1):
            enqueue(i)


def timed_steps(ctx: StepCtx, flush, stream, steps: int, warmup: int, local: int,
                world: int, quick: bool) -> dict:
    """Device time per step (CUDA events on the launching stream, L2 flushed
    before every step outside the events) and the clocks sampled over the
    timed window, kept open for about a second of identical work."""
    pa = ctx.pa
    for _ in range(max(3, warmup)):
        ctx.step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.15)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    n0 = pa.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()

    def one(i):
        flush()
        starts[i].record(stream)
        ctx.step()
        ends[i].record(stream)

    queued(steps, one)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    launches = pa.launch_count() - n0
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    extra = 0
    while not quick and time.perf_counter() - t_wall < 1.0 and extra < 20000:
        flush()
        ctx.step()
        extra += 1
        if extra % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop()
    return {"ms": max_over_ranks(statistics.mean(step_ms), world), "clocks": clk,
            "launches": launches, "wall": wall}


def timed_kernel(ctx: StepCtx, flush, steps: int, world: int) -> float:
    """Mean duration (ms) of the attention kernel alone: events recorded by
    the library right around its launch, on its stream."""
    pa = ctx.pa
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    def one(i):
        flush()
        pa.profile_events(ev_a[i], ev_b[i])
        ctx.attend_only()

    queued(steps, one)
    pa.profile_events(None, None)
    torch.cuda.synchronize()
    return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)), world)


def extra_config(pa, name, args, world, rank, local, dev, flush, stream, peak) -> dict:
    """The step and its attention kernel on another seeded workload, with
    its own clock record."""
    ctx = StepCtx(pa, name, rank, dev)
    t = timed_steps(ctx, flush, stream, args.steps, args.warmup, local, world, args.quick)
    k_ms = timed_kernel(ctx, flush, args.steps, world)
    if pa.check_device_error():
        raise RuntimeError(f"device error flag during the {name} benchmark")
    total = sum_over_ranks(float(ctx.step_bytes), world)
    gbs = total / (t["ms"] * 1e-3) / 1e9
    achieved = ctx.dbytes["kernel"] / (k_ms * 1e-3) / 1e9
    entry = {"workload": workload_desc(ctx.s), "us_per_step": t["ms"] * 1e3,
             "value": gbs, "unit": UNIT, "pct_of_peak": 100.0 * gbs / world / peak,
             "bytes_per_step_per_rank": ctx.step_bytes,
             "attended_tokens_per_rank": ctx.dbytes["tokens"],
             "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel",
                          "kernel_us": k_ms * 1e3, "bytes_per_launch": ctx.dbytes["kernel"],
                          "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak,
                          "traffic": profiled_traffic(name, ctx.dbytes["kernel"])},
             "gpu_launches": t["launches"], "clocks": t["clocks"]}
    if ctx.s.shared_prefix:
        # shared prefix blocks: logical bytes count them once per sequence that
        # reads them (the metric's bytes), unique bytes once per step
        entry["kv_bytes_logical"] = ctx.dbytes["kv"]
        entry["kv_bytes_unique"] = unique_kv_bytes(ctx.w)
    del ctx
    torch.cuda.empty_cache()
    return entry


def run_ours(args, world, rank, local):
    import paged_kv_cache_267_gb300 as pa
    from paged_kv_cache_267_gb300.build import build_library
    build_library()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    ctx = StepCtx(pa, args.config, rank, dev)
    w, s = ctx.w, ctx.s
    kv, kc, vc, bt, sl, out, kw = ctx.kv, ctx.kc, ctx.vc, ctx.bt, ctx.sl, ctx.out, ctx.kw
    attend = ctx.attend
    stream = torch.cuda.current_stream()
    dbytes, step_bytes = ctx.dbytes, ctx.step_bytes
    flush = L2Flush(dev)

    t = timed_steps(ctx, flush, stream, args.steps, args.warmup, local, world, args.quick)
    ms, clk, launches, wall = t["ms"], t["clocks"], t["launches"], t["wall"]
    total_bytes = sum_over_ranks(float(step_bytes), world)
    value = total_bytes / (ms * 1e-3) / 1e9

    # ---- roofline: decode kernel alone, events around it on the launch stream
    k_ms = timed_kernel(ctx, flush, args.steps, world)
    peak, peak_kind = measured_peak()
    achieved = dbytes["kernel"] / (k_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.config, dbytes["kernel"])
    flops = attention_flops(w)
    tpeak, tpeak_kind = measured_tensor_peak()
    # bound: whichever of bytes and FLOPs takes longer at its measured peak
    tensor_bound = flops / (tpeak * 1e12) > dbytes["kernel"] / (peak * 1e9)

    # ---- end to end through the public API with host buffers. The step's
    # host inputs (q, new k/v, slots, block tables, seq_lens) and its output
    # live in pinned host memory; the kernels use them in place.
    host_in = {n: t_.detach().cpu().contiguous().pin_memory() for n, t_ in
               (("q", w.q), ("k", w.k_new), ("v", w.v_new), ("slot", w.slot_new), ("bt", bt),
                ("sl", sl))}
    host_res = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    kw_host = dict(kw, out=host_res)
    h2d_direct = sum(t_.numel() * t_.element_size() for t_ in host_in.values())
    d2h_direct = host_res.numel() * host_res.element_size()

    def e2e_direct():
        pa.reshape_and_cache(host_in["k"], host_in["v"], kc, vc, host_in["slot"], kv, w.k_scale,
                             w.v_scale)
        attend(host_in["q"], kc, vc, host_in["bt"], host_in["sl"], **kw_host)

    # The same with the copy engine: one packed pinned staging buffer (each
    # input at a 256-byte aligned offset) moved by one H2D copy, the library
    # on device views of it, and one D2H copy of the output.
    parts = [(n, t_.detach().contiguous()) for n, t_ in
             (("q", w.q), ("k", w.k_new), ("v", w.v_new), ("slot", w.slot_new),
              ("bt", bt), ("sl", sl))]
    offs, off = {}, 0
    for n, t_ in parts:
        offs[n] = off
        off += (t_.numel() * t_.element_size() + 255) // 256 * 256
    host_stage = torch.empty(off, dtype=torch.uint8, pin_memory=True)
    dev_stage = torch.empty(off, dtype=torch.uint8, device=dev)
    dev_in = {}
    for n, t_ in parts:
        nb = t_.numel() * t_.element_size()
        host_stage[offs[n]:offs[n] + nb].copy_(t_.cpu().view(torch.uint8).reshape(-1))
        dev_in[n] = dev_stage[offs[n]:offs[n] + nb].view(t_.dtype).view(t_.shape)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = off  # bytes moved, alignment padding included
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        dev_stage.copy_(host_stage, non_blocking=True)
        pa.reshape_and_cache(dev_in["k"], dev_in["v"], kc, vc, dev_in["slot"], kv, w.k_scale,
                             w.v_scale)
        attend(dev_in["q"], kc, vc, dev_in["bt"], dev_in["sl"], **kw)
        host_out.copy_(out, non_blocking=True)

    # The host-buffer steps are enqueued one by one, without the spin: a
    # host-side delay inside a step counts here.
    def timed_mean_ms(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            e_s[i].record(stream)
            fn()
            e_e[i].record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(e_s, e_e)), world)

    e2e_ms = timed_mean_ms(e2e_direct)
    e2e_value = total_bytes / (e2e_ms * 1e-3) / 1e9
    # same inputs as the device step: equal up to the summation order the
    # dynamic pool may change
    if (host_res.float() - out.float().cpu()).abs().max().item() > 1e-2:
        raise RuntimeError("the host-buffer step disagrees with the device step")
    copy_ms = timed_mean_ms(e2e_step)

    # ---- the same step captured once in a CUDA graph and replayed (the L2
    # flush stays outside the graph, events around each replay)
    gstream = torch.cuda.Stream(device=dev)
    gstream.wait_stream(stream)
    with torch.cuda.stream(gstream):
        for _ in range(3):
            ctx.step()  # the library's workspace for this stream exists before capture
    gstream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        ctx.step()
    g_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    def replay(i):
        flush()
        g_s[i].record(stream)
        graph.replay()
        g_e[i].record(stream)

    queued(args.steps, replay)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(g_s, g_e)), world)
    del graph

    bad = pa.check_device_error()
    if bad:
        raise RuntimeError(f"device error flag {bad} during the benchmark")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        kch, vch = host_caches(w, kc, vc)
        subset, queries = bounded_sample(w, kch, vch, args.cpu_budget / 2)
        cpu = oracle_baseline(w, kch, vch, budget_s=args.cpu_budget, seq_subset=subset,
                              queries=queries)
        del kch, vch

    # ---- the other seeded workloads, each with its own timed window
    extras = {}
    names = [n for n in (args.configs.split(",") if args.configs else []) if n and n != args.config]
    if names:
        del ctx, w, kc, vc, host_in, host_res, host_stage, dev_stage, dev_in, host_out, parts
        kw = kw_host = None
        torch.cuda.empty_cache()
        for name in names:
            extras[name] = extra_config(pa, name, args, world, rank, local, dev, flush, stream,
                                        peak)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "us_per_step": ms * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if s.dtype == "bf16" else "f16",
        "data": "synthetic",
        "config": {"workload": f"{args.config}: {workload_desc(s)}",
                   "global_batch": s.batch * world, "parallelism": f"replicas{world}",
                   "step": ("pa_reshape_and_cache (1 new token per sequence) + pa_decode"
                            if s.num_queries == 1 else
                            f"pa_reshape_and_cache ({s.num_queries} new tokens per sequence) + "
                            "pa_prefill_chunk"),
                   "attended_tokens_per_rank": dbytes["tokens"],
                   "bytes_per_step_per_rank": step_bytes,
                   "l2": "flushed between timed steps, outside the events: write 4x L2, then read 4x L2",
                   "queue": "timed device steps enqueued behind a bounded spin kernel, so no step waits for host launches; the e2e steps are not"},
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": ({"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                      "frac": achieved / peak, "traffic": traffic,
                      "kernel": "paged_decode_kernel", "kernel_us": k_ms * 1e3,
                      "bytes_per_launch": dbytes["kernel"], "peak_kind": peak_kind}
                     if not tensor_bound else
                     {"bound": "tensor", "achieved": flops / (k_ms * 1e-3) / 1e12,
                      "peak": tpeak, "unit": "TFLOP/s",
                      "frac": flops / (k_ms * 1e-3) / 1e12 / tpeak, "traffic": None,
                      "kernel": "chunk_attn_tc128_kernel", "kernel_us": k_ms * 1e3,
                      "flops_per_launch": flops, "peak_kind": tpeak_kind + " bf16 burst"}),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d_direct,
                "d2h_bytes_per_step": d2h_direct, "ms_per_step": e2e_ms,
                "transfer": "kernels read the inputs from and write the output to pinned "
                            "host memory in place (CPU-GPU link)",
                "copy_engine": {"value": total_bytes / (copy_ms * 1e-3) / 1e9,
                                "ms_per_step": copy_ms, "h2d_bytes_per_step": h2d,
                                "d2h_bytes_per_step": d2h}},
        "graph": {"value": total_bytes / (graph_ms * 1e-3) / 1e9, "unit": UNIT,
                  "us_per_step": graph_ms * 1e3,
                  "what": "the step captured in one CUDA graph, replayed per step"},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if extras:
        line["configs"] = extras
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama8b")
    ap.add_argument("--configs", default=DEFAULT_EXTRA_CONFIGS,
                    help="other seeded workloads timed after the main one, each reported "
                         "under 'configs' in the JSON line (comma-separated; '' for none)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="no CPU baseline and no clock-sampling extension (for profiler runs)")
    args = ap.parse_args()
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        relaunch_under_torchrun(args.gpus)
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
