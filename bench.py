"""Decode-step benchmark: KV append + paged decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c1] [--impl ours|reference]

One step = one pass of the whole hot path over one batch: the KV append of the
step's new tokens (wllm_reshape_and_cache) followed by paged decode attention
for every sequence (wllm_paged_attention_decode), both through the C ABI.
Inputs are seeded synthetic decode steps (paged_kv_cache_185_gb300.workloads),
resident in HBM when timing starts.  L2 is flushed (a 512 MiB write) between
timed steps, outside the timed events.  Every step is timed with CUDA events on
the launching stream; per-kernel durations come from events around each launch.

Metric: decode-attention tokens/s (each sequence advances one token per step),
with the achieved HBM GB/s of the step and of the decode kernel (algorithmic
bytes: unique K/V bytes read + q + out + block-table entries + lengths).

With N > 1 (torchrun), every rank runs its own replica of the workload with its
own seed (sequences are independent: no collective on the data path); rank 0
prints one JSON line with the whole-job tokens/s over the slowest rank's time.

Extra fields of the line: "graph" (several layers' steps replayed from one CUDA
graph vs issued eagerly), "fp8" (the same decode and step over an E4M3 cache)
and "prefill" (chunked-prefill paged attention on
the workload's head geometry, against the measured bf16 tensor peak).

--impl reference times the fp64 CPU oracle on the host cores, on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_185_gb300 import workloads  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20
WORKLOAD_DESC = {
    "c0": "4 seqs L={7,16,33,50}, 4/2 heads, D 64, fp32",
    "c1": "64 seqs L~U[128,2048], 32/4 heads, D 64, fp16",
    "c2": "128 seqs L~U[1024,4096], 32/32 heads, D 128, bf16, 128 appends to free slots",
    "c3": "256 seqs in groups of 8 sharing 64 blocks, tails lognormal(1500, 0.5), 28/4 heads, D 128, bf16",
    "c4": "8 seqs L~U[32768,131072], 32/8 heads, D 128, bf16, ~120 GB pool, 1% keys x8",
    "gemma_mqa": "128 seqs L~U[1024,4096], 8/1 heads (MQA), D 256, bf16",
    "bs32": "128 seqs L~U[1024,4096], 32/32 heads, D 128, bf16, block_size 32, 128 appends to free slots",
}
DTYPE_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def graph_layers(args, case, dev, q, key, value, slots, bt, cl, flush, stream):
    """Several layers' decode steps (each layer its own K/V pools, the same step
    inputs) back to back, issued eagerly and replayed from one CUDA graph; the
    L2 is flushed between repetitions, outside the events.  Returns per-layer
    times, or None when the layers' pools would not fit the budget."""
    import paged_kv_cache_185_gb300 as wllm

    L = args.graph_layers
    if L <= 0 or L * 2 * case.pool_bytes() > (8 << 30) or case.dtype == torch.float32:
        return None
    B, Hq, Hkv, D, bs = case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    pools = [case.pool(dev) for _ in range(L)]
    outs = [torch.empty_like(q) for _ in range(L)]
    need = wllm.workspace_bytes(B, Hq, Hkv, D, case.max_blocks, bs)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    wllm.set_workspace(ws)
    try:
        def layers():
            for (kc, vc), o in zip(pools, outs):
                wllm.decode_step(o, q, key, value, kc, vc, slots, bt, cl, Hkv, case.scale, bs)

        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                layers()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layers()
        torch.cuda.synchronize()
        R = max(20, min(args.steps, 200))
        res = {}
        for name, fn in (("eager", layers), ("graph", g.replay)):
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
            for e in ev:
                flush.zero_()
                e[0].record(stream)
                fn()
                e[1].record(stream)
            torch.cuda.synchronize()
            res[name] = sum(e[0].elapsed_time(e[1]) for e in ev) / R * 1e3 / L
        return {"layers": L, "us_per_layer": res["graph"], "eager_us_per_layer": res["eager"],
                "note": "layers back to back, each on its own K/V pools; one CUDA graph replay vs eager calls"}
    finally:
        wllm.set_workspace(None)
        del pools


def fp8_decode(args, case, dev, q, key, value, slots, bt, cl, kc16, vc16, flush, stream):
    """The same decode step over an fp8 (E4M3) cache: codes drawn from the
    case's K/V (4x the values, read back with scales 1/4), the decode alone and
    the fused step timed like the main measurement.  None when the kernel has
    no fp8 form for this shape (fp32 queries, head_dim 64 with 8-token blocks)."""
    import paged_kv_cache_185_gb300 as wllm

    if (case.dtype == torch.float32 or case.head_dim not in (64, 128, 256) or args.fp8_reps <= 0
            or (case.head_dim == 64 and case.block_size < 16)):
        return None
    B, Hkv, bs = case.num_seqs, case.num_kv_heads, case.block_size
    pools = []
    for src in (kc16, vc16):  # input codes, drawn on the device block by block (not timed)
        dst = torch.empty(src.shape, dtype=torch.uint8, device=dev)
        for i in range(0, src.shape[0], 8192):
            dst[i:i + 8192] = (src[i:i + 8192].float() * 4.0).to(torch.float8_e4m3fn).view(torch.uint8)
        pools.append(dst)
    kc, vc = pools
    out = torch.empty_like(q)
    ks = vs = 0.25
    R = args.fp8_reps

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        return sum(e[0].elapsed_time(e[1]) for e in ev) / R

    dec_ms = timed(lambda: wllm.paged_attention_decode_fp8(out, q, kc, vc, bt, cl, Hkv, case.scale, ks, vs, bs))
    step_ms = timed(lambda: wllm.decode_step_fp8(out, q, key, value, kc, vc, slots, bt, cl, Hkv, case.scale, ks,
                                                 vs, bs))
    kv16 = case.kv_bytes_read()
    alg = case.algorithmic_bytes() - kv16 + kv16 // case.elt  # one byte per cached element
    peak, peak_kind = measured_peak()
    achieved = alg / (dec_ms / 1e3) / 1e9
    del pools, kc, vc
    return {"kv_dtype": "e4m3", "decode_us": dec_ms * 1e3, "step_us": step_ms * 1e3,
            "tokens_per_s": B / (step_ms / 1e3), "algorithmic_bytes": alg,
            "roofline": {"bound": "hbm", "kernel": "paged_decode_persistent<fp8> (decode + in-launch merge)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind},
            "reps": R, "note": "decode-only and fused-step times over E4M3 caches; L2 flushed between reps"}


def prefill_bench(args, case, dev, flush, stream):
    """Chunked prefill on the workload's head geometry: 8 sequences, each a
    512-token chunk after 0..2048 tokens of context (seeded), timed through
    wllm_paged_attention_prefill.  FLOPs are the causal attention's own
    (4 * D * (P + 1) per query row at position P), against the measured bf16
    tensor peak."""
    import numpy as np
    import paged_kv_cache_185_gb300 as wllm

    if case.dtype == torch.float32 or case.head_dim not in (64, 128) or args.prefill_reps <= 0:
        return None
    rng = np.random.default_rng(77)
    nseq, chunk = 8, 512
    prior = rng.integers(0, 2049, size=nseq)
    lens = [int(x) + chunk for x in prior]
    pc = workloads.custom_case("prefill", lens=lens, num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                               head_dim=case.head_dim, block_size=case.block_size, dtype=case.dtype, seed=77,
                               append="none")
    kc, vc = pc.pool(dev)
    T = nseq * chunk
    q = torch.from_numpy(workloads.normal(78, T * case.num_q_heads * case.head_dim)).reshape(
        T, case.num_q_heads, case.head_dim).to(case.dtype).to(dev)
    out = torch.empty_like(q)
    qsl = torch.arange(0, T + 1, chunk, dtype=torch.int32, device=dev)
    bt, cl = pc.block_tables.to(dev), pc.context_lens.to(dev)

    def call():
        wllm.paged_attention_prefill(out, q, kc, vc, bt, cl, qsl, case.num_kv_heads, case.scale, case.block_size)

    for _ in range(3):
        flush.zero_()
        call()
    R = args.prefill_reps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        call()
        e[1].record(stream)
    torch.cuda.synchronize()
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / R
    fp8_ms = None
    if case.head_dim == 128 or case.block_size >= 16:  # the same chunks over E4M3 codes of the same K/V
        k8 = (kc.float() * 4.0).to(torch.float8_e4m3fn).view(torch.uint8)
        v8 = (vc.float() * 4.0).to(torch.float8_e4m3fn).view(torch.uint8)

        def call8():
            wllm.paged_attention_prefill_fp8(out, q, k8, v8, bt, cl, qsl, case.num_kv_heads, case.scale, 0.25, 0.25,
                                             case.block_size)

        for _ in range(3):
            flush.zero_()
            call8()
        ev8 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
        for e in ev8:
            flush.zero_()
            e[0].record(stream)
            call8()
            e[1].record(stream)
        torch.cuda.synchronize()
        fp8_ms = sum(e[0].elapsed_time(e[1]) for e in ev8) / R
    flops = 0
    for p0 in prior:
        P = np.arange(int(p0), int(p0) + chunk)
        flops += int(4 * case.head_dim * (P + 1).sum()) * case.num_q_heads
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (bf16 burst)"
    except Exception:
        peak, kind = 1900.0, "fallback"
    achieved = flops / (ms / 1e3) / 1e12
    return {"workload": f"{nseq} seqs x {chunk}-token chunks after U[0,2048] context, "
                        f"{case.num_q_heads}/{case.num_kv_heads} heads, D {case.head_dim}",
            "us": ms * 1e3, "tokens_per_s": T / (ms / 1e3),
            "roofline": {"bound": "tensor", "kernel": "paged_prefill_kernel (mma.sync m16n8k16)",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_kind": kind, "flops": flops},
            "fp8_cache_us": None if fp8_ms is None else fp8_ms * 1e3,
            "fp8_cache_tflops": None if fp8_ms is None else flops / (fp8_ms / 1e3) / 1e12,
            "reps": R}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_185_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per decode launch from an ncu capture (profiles/decode_traffic.txt),
    used only while the kernel sources still hash to the captured version."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_sources_sha()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if kv.get("workload") == workload and kv.get("sources_sha") == sha:
                return int(kv["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        with open(self.file.name) as f:
            rows = [ln.strip().split(", ") for ln in f if ln.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for name, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def setup_dist(gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def all_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_case(workload: str, rank: int):
    """Rank r's replica: the named workload recipe with its own seed."""
    return workloads.make_case(workload, replica=rank)


def cpu_oracle_rate(case, budget_s: float, max_seqs=None, threads: int = 0):
    """Oracle decode (after its own append) on the host cores (all of them, or
    `threads`) over a bounded sample of sequences; returns (tokens/s, sample
    description, threads)."""
    import oracle
    kc, vc = case.pool("cpu")
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    threads = threads if threads > 0 else oracle.max_threads()
    B, Hq = case.num_seqs, case.num_q_heads
    # calibrate on one sequence, then size the sample to the budget
    t0 = time.perf_counter()
    oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.num_kv_heads,
                        case.scale, rows=list(range(Hq)), num_threads=threads)
    per_seq = max(time.perf_counter() - t0, 1e-6)
    n = int(min(B, max(1, budget_s / per_seq)))
    if max_seqs is not None:
        n = min(n, max_seqs)
    rows = list(range(n * Hq))
    t0 = time.perf_counter()
    oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.num_kv_heads,
                        case.scale, rows=rows, num_threads=threads)
    dt = time.perf_counter() - t0
    return n / dt, f"first {n} of {B} sequences of the workload, all {Hq} heads, one decode", threads


def run_reference(args):
    rank, world, _ = setup_dist(args.gpus)
    if rank != 0:
        return
    case = workloads.make_case(args.workload)
    import oracle
    kc, vc = case.pool("cpu")
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    Hq = case.num_q_heads
    t0 = time.perf_counter()
    oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.num_kv_heads,
                        case.scale, rows=list(range(Hq)))
    per_seq = max(time.perf_counter() - t0, 1e-6)
    budget = 90.0 / max(1, args.steps + args.warmup)  # whole run within ~1.5 min
    n = int(min(case.num_seqs, max(1, budget / per_seq)))
    rows = list(range(n * Hq))
    for _ in range(args.warmup):
        oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                            case.num_kv_heads, case.scale, rows=rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                            case.num_kv_heads, case.scale, rows=rows)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = n / (ms / 1e3)
    sample = f"first {n} of {case.num_seqs} sequences, all {Hq} heads, per step"
    line = {
        "impl": "reference", "metric": "decode-attn tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(case, args.workload, None),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(case, workload, part_tokens):
    return {
        "workload": case.name, "shape": WORKLOAD_DESC.get(workload, workload),
        "batch": case.num_seqs, "q_heads": case.num_q_heads, "kv_heads": case.num_kv_heads,
        "head_dim": case.head_dim, "block_size": case.block_size, "num_blocks": case.num_blocks,
        "context_tokens": int(case.context_lens.sum()), "unique_kv_tokens": case.meta["unique_tokens"],
        "appended_tokens": int(case.slot_mapping.numel()), "partition_tokens": part_tokens,
        "l2": "flushed between timed steps (512 MiB write, outside the timed events)",
    }


def run_ours(args):
    import paged_kv_cache_185_gb300 as wllm
    from paged_kv_cache_185_gb300 import build as wbuild
    rank, world, local = setup_dist(args.gpus)
    assert torch.cuda.is_available(), "bench needs a CUDA device"
    torch.cuda.set_device(local)
    if rank == 0:
        wbuild.build()
    barrier(world)
    wllm.load_library()
    dev = torch.device("cuda", local)

    case = replica_case(args.workload, rank)
    B, Hq, Hkv, D, bs = case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    kc, vc = case.pool(dev)
    q = case.q.to(dev)
    key, value, slots = case.key.to(dev), case.value.to(dev), case.slot_mapping.to(dev)
    bt, cl = case.block_tables.to(dev), case.context_lens.to(dev)
    out = torch.empty_like(q)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    part_tokens = wllm.partition_tokens(B, Hq, Hkv, D, case.max_blocks, bs, case.dtype)
    # our kernels per timed step: the fused step is one cooperative launch for
    # f16/bf16; fp32 runs the append kernel and the decode kernel
    launches_per_step = 1 if case.dtype != torch.float32 else (2 if case.slot_mapping.numel() else 1)

    def step():
        wllm.decode_step(out, q, key, value, kc, vc, slots, bt, cl, Hkv, case.scale, bs)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms_per_step = sum(step_ms) / K
    # the two calls separately (append, then decode), for the kernel breakdown
    sep = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(min(K, 200))]
    for e in sep:
        flush.zero_()
        e[0].record(stream)
        wllm.reshape_and_cache(key, value, kc, vc, slots)
        e[1].record(stream)
        wllm.paged_attention_decode(out, q, kc, vc, bt, cl, Hkv, case.scale, bs)
        e[2].record(stream)
    torch.cuda.synchronize()
    app_ms = [e[0].elapsed_time(e[1]) for e in sep]
    dec_ms = [e[1].elapsed_time(e[2]) for e in sep]
    ms_max = all_max(ms_per_step, world)
    tok_s = B * world / (ms_max / 1e3)

    # end to end through the public API with host buffers: pinned H2D of the
    # step's inputs, append + decode, D2H of the output, all inside the events
    h_in = {n: t.pin_memory() for n, t in (("q", case.q), ("key", case.key), ("value", case.value),
                                           ("slots", case.slot_mapping), ("bt", case.block_tables),
                                           ("cl", case.context_lens))}
    d_in = {"q": q, "key": key, "value": value, "slots": slots, "bt": bt, "cl": cl}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = h_out.numel() * h_out.element_size()
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K + max(3, args.warmup)):
        j = i - max(3, args.warmup)
        flush.zero_()
        if j >= 0:
            e2e_ev[j][0].record(stream)
        for n in d_in:
            d_in[n].copy_(h_in[n], non_blocking=True)
        wllm.decode_step(out, q, key, value, kc, vc, slots, bt, cl, Hkv, case.scale, bs)
        h_out.copy_(out, non_blocking=True)
        if j >= 0:
            e2e_ev[j][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = all_max(sum(e[0].elapsed_time(e[1]) for e in e2e_ev) / K, world)
    e2e_value = B * world / (e2e_ms / 1e3)

    graph = graph_layers(args, case, dev, q, key, value, slots, bt, cl, flush, stream)
    fp8 = fp8_decode(args, case, dev, q, key, value, slots, bt, cl, kc, vc, flush, stream)
    prefill = prefill_bench(args, case, dev, flush, stream)

    peak, peak_kind = measured_peak()
    alg = case.algorithmic_bytes()
    dec_mean = sum(dec_ms) / len(dec_ms)
    step_bytes = alg + case.append_bytes()
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9  # the fused step kernel: append + decode bytes
    traffic = recorded_traffic(args.workload)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, sample, threads = cpu_oracle_rate(case, budget_s=args.cpu_budget)
        rate1, sample1, _ = cpu_oracle_rate(case, budget_s=min(3.0, args.cpu_budget), threads=1)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample,
               "single_thread": {"value": rate1, "unit": "tokens/s", "sample": sample1}}
    line = {
        "metric": "decode-attn tokens/s", "value": tok_s, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[case.dtype], "data": "synthetic",
        "config": config_of(case, args.workload, part_tokens),
        "achieved_gbs": step_bytes / (ms_per_step / 1e3) / 1e9,
        "pct_of_8tbs": 100.0 * step_bytes / (ms_per_step / 1e3) / 8e12,
        "kernel_ms": {"step_fused": ms_per_step, "step_median": statistics.median(step_ms),
                      "append_separate": sum(app_ms) / len(app_ms), "decode_separate": dec_mean},
        "roofline": {"bound": "hbm", "kernel": "paged_decode_persistent (fused step: append + decode + combine)",
                     "achieved": achieved,
                     "peak": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes": step_bytes},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks.summary(),
        "graph": graph,
        "fp8": fp8,
        "prefill": prefill,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--graph-layers", type=int, default=8,
                    help="layers per CUDA-graph replay for the graph measurement (0: skip)")
    ap.add_argument("--fp8-reps", type=int, default=100,
                    help="repetitions of the fp8-cache measurement (0: skip)")
    ap.add_argument("--prefill-reps", type=int, default=50,
                    help="repetitions of the chunked-prefill measurement (0: skip)")
    ap.add_argument("--workload", default="c1", choices=list(workloads.CASE_NAMES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
