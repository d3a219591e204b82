"""Decode-step benchmark: KV append + paged decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4] [--impl ours|reference]

One step = one pass of the whole hot path over one batch: the KV append of the
step's new tokens followed by paged decode attention for every sequence, as
one fused launch through the C ABI (wllm_decode_step).  Inputs are seeded
synthetic decode steps (paged_kv_cache_185_gb300.workloads), resident in HBM
when timing starts.  L2 is flushed (a 512 MiB write) between timed steps,
outside the timed events.  Every step is timed with CUDA events on the
launching stream.

Metric: decode-attention tokens/s (each sequence advances one token per step),
with the achieved HBM GB/s of the step (algorithmic bytes: unique K/V bytes
read + q + out + block-table entries + lengths + the appended rows).

The headline line is the long-context batch (32K-128K tokens per sequence over
a ~120 GB pool), the largest that fits one GPU.  The same line carries a
"per_workload" record for every other workload, timed in the same process the
same way: the tiny fp32 step, the TinyLlama-, Llama-2-7B- and
Qwen2.5-7B-shaped batches, and the report rows (Gemma-shaped multi-query,
32-token blocks).  Each record holds its step time, tokens/s, algorithmic
bytes, roofline fraction against the measured HBM bandwidth, DRAM traffic
from an ncu capture (while the kernel sources still match it), an end-to-end
figure with host copies, the fp8 (E4M3) cache form and, for the small ones,
the fp64 oracle's own rate on the host cores.

With N > 1 (torchrun), every rank runs its own replica of the workload with its
own seed (sequences are independent: no collective on the data path); rank 0
prints one JSON line with the whole-job tokens/s over the slowest rank's time.

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
ALL_WORKLOADS = ("c0", "c1", "c2", "c3", "c4", "gemma_mqa", "bs32")


# ---------------------------------------------------------------------------
# small helpers
# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_185_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kind: str = "step"):
    """DRAM bytes per launch of the named workload's fused step (kind "step")
    or fp8 fused step ("fp8_step") from an ncu capture
    (profiles/decode_traffic.txt), used only while the kernel sources still
    hash to the captured version."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_sources_sha()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if (kv.get("workload") == workload and kv.get("sources_sha") == sha
                    and kv.get("kind", "step") == kind):
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


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def sample_rows(case):
    """Every (sequence, head) row once, cycling over the sequences first, so
    that any prefix of the order mixes short and long sequences."""
    B, Hq = case.num_seqs, case.num_q_heads
    return [(i % B) * Hq + (i // B) for i in range(B * Hq)]


def host_oracle_inputs(case):
    """The oracle's inputs: only the referenced blocks (the compact pool: the
    same tokens and sharing, renumbered; the full ~120 GB pool of the
    long-context batch is never built on the host), with this step's append
    already applied."""
    import oracle
    kc, vc, bt, slots = case.compact()
    if slots.numel():
        oracle.reshape_and_cache(case.key, case.value, kc, vc, slots)
    return kc, vc, bt


class OracleSample:
    """The oracle's decode over a bounded sample of rows of one workload."""

    def __init__(self, case, threads: int = 0):
        import oracle
        self.oracle = oracle
        self.case = case
        self.kc, self.vc, self.bt = host_oracle_inputs(case)
        self.order = sample_rows(case)
        self.threads = threads if threads > 0 else oracle.max_threads()

    def run(self, n: int) -> float:
        c = self.case
        t0 = time.perf_counter()
        self.oracle.paged_decode(c.q, self.kc, self.vc, self.bt, c.context_lens, c.num_kv_heads, c.scale,
                                 rows=self.order[:n], num_threads=self.threads)
        return time.perf_counter() - t0

    def rows_for(self, budget_s: float) -> int:
        """Rows whose decode takes about budget_s (at least one)."""
        k = min(len(self.order), self.threads)
        dt = max(self.run(k), 1e-6)
        n = int(k * budget_s / dt)
        return max(1, min(len(self.order), n))

    def describe(self, n: int) -> str:
        c = self.case
        return (f"{n} of {c.num_seqs * c.num_q_heads} (sequence, head) rows cycling over the {c.num_seqs} "
                f"sequences, one decode each (after the step's append), over the referenced blocks; "
                f"tokens/s = rows/s / {c.num_q_heads} heads")

    def cores(self, n: int) -> int:
        return min(n, self.threads)


def cpu_oracle_rate(case, budget_s: float, threads: int = 0):
    """Oracle decode (after its own append) on the host cores (all of them, or
    `threads`) over a bounded sample of rows; returns the cpu_baseline record."""
    s = OracleSample(case, threads)
    n = s.rows_for(budget_s)
    dt = s.run(n)
    return {"value": n / case.num_q_heads / dt, "unit": "tokens/s", "cores": s.cores(n), "kind": "oracle",
            "sample": s.describe(n), "seconds": dt}


def run_reference(args):
    rank, world, _ = setup_dist(args.gpus)
    if rank != 0:
        return
    case = workloads.make_case(args.workload)
    s = OracleSample(case)
    budget = 90.0 / max(1, args.steps + args.warmup)  # whole run within ~1.5 min of oracle time
    n = s.rows_for(budget)
    for _ in range(args.warmup):
        s.run(n)
    times = [s.run(n) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = n / case.num_q_heads / (ms / 1e3)
    line = {
        "impl": "reference", "metric": "decode-attn tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(case, args.workload, None, "compact (referenced blocks)"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": s.cores(n), "kind": "oracle",
                         "sample": s.describe(n) + ", per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(case, workload, part_tokens, pool="full"):
    return {
        "workload": case.name, "shape": WORKLOAD_DESC.get(workload, workload),
        "batch": case.num_seqs, "q_heads": case.num_q_heads, "kv_heads": case.num_kv_heads,
        "head_dim": case.head_dim, "block_size": case.block_size, "num_blocks": case.num_blocks,
        "context_tokens": int(case.context_lens.sum()), "unique_kv_tokens": case.meta["unique_tokens"],
        "appended_tokens": int(case.slot_mapping.numel()), "partition_tokens": part_tokens,
        "pool": pool,
        "l2": "flushed between timed steps (512 MiB write, outside the timed events)",
    }


# ---------------------------------------------------------------------------
# GPU measurements
# ---------------------------------------------------------------------------

def event_times(fn, reps, flush, stream, warm=3):
    """Mean and median milliseconds of fn over reps timed calls (CUDA events
    on `stream`, L2 flushed before each call, outside the events)."""
    for _ in range(warm):
        flush.zero_()
        fn()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        fn()
        e[1].record(stream)
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    return sum(ms) / len(ms), statistics.median(ms)


def fp8_step(args, case, dev, q, key, value, slots, bt, cl, kc16, vc16, flush, stream, reps):
    """The same step over an fp8 (E4M3) cache: codes drawn from the case's K/V
    (4x the values, read back with scales 1/4), the decode alone and the fused
    step timed like the 16-bit step.  None when the kernel has no fp8 form for
    this shape (fp32 queries, head_dim 64 with 8-token blocks)."""
    import paged_kv_cache_185_gb300 as wllm

    if (case.dtype == torch.float32 or case.head_dim not in (64, 128, 256) or reps <= 0
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
    dec_ms, _ = event_times(lambda: wllm.paged_attention_decode_fp8(out, q, kc, vc, bt, cl, Hkv, case.scale, ks,
                                                                     vs, bs), reps, flush, stream)
    step_ms, step_med = event_times(lambda: wllm.decode_step_fp8(out, q, key, value, kc, vc, slots, bt, cl, Hkv,
                                                                 case.scale, ks, vs, bs), reps, flush, stream)
    kv16 = case.kv_bytes_read()
    # one byte per cached element, for the reads and the appended rows
    alg = case.algorithmic_bytes() - kv16 + kv16 // case.elt
    app = case.append_bytes()
    T = int(case.slot_mapping.numel())
    valid = int((case.slot_mapping >= 0).sum())
    app8 = 2 * valid * case.num_kv_heads * case.head_dim * (case.elt + 1) + 8 * T if T else 0
    peak, peak_kind = measured_peak()
    achieved = (alg + app8) / (step_ms / 1e3) / 1e9
    del pools, kc, vc
    return {"kv_dtype": "e4m3", "decode_us": dec_ms * 1e3, "step_us": step_ms * 1e3, "step_median_us": step_med * 1e3,
            "tokens_per_s": B / (step_ms / 1e3), "algorithmic_bytes": alg + app8,
            "roofline": {"bound": "hbm", "kernel": "paged_decode_persistent<fp8> (fused step)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": recorded_traffic(case_key(case), "fp8_step")},
            "decode_roofline_frac": alg / (dec_ms / 1e3) / 1e9 / peak,
            "reps": reps, "note": "E4M3 caches; the 16-bit append bytes %d become %d" % (app, app8)}


_CASE_KEY = {}


def case_key(case):
    return _CASE_KEY.get(id(case), case.name)


def measure(args, name, rank, world, local, dev, flush, stream, steps, *, cpu_budget=0.0, single_budget=0.0,
            fp8_reps=0, pool="full"):
    """Time the fused step of one workload; returns its record."""
    import paged_kv_cache_185_gb300 as wllm

    case = replica_case(name, rank)
    _CASE_KEY[id(case)] = name
    B, Hq, Hkv, D, bs = case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    if pool == "compact":  # the referenced blocks only, renumbered: the same bytes read (for ncu captures)
        kh, vh, bth, slh = case.compact()
        kc, vc, bt, slots = kh.to(dev), vh.to(dev), bth.to(dev), slh.to(dev)
        del kh, vh
    else:
        kc, vc = case.pool(dev)
        bt, slots = case.block_tables.to(dev), case.slot_mapping.to(dev)
    q = case.q.to(dev)
    key, value = case.key.to(dev), case.value.to(dev)
    cl = case.context_lens.to(dev)
    out = torch.empty_like(q)
    part_tokens = wllm.partition_tokens(B, Hq, Hkv, D, case.max_blocks, bs, case.dtype)

    def step():
        wllm.decode_step(out, q, key, value, kc, vc, slots, bt, cl, Hkv, case.scale, bs)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        n0 = wllm.launch_count()
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        launches = wllm.launch_count() - n0
        torch.cuda.synchronize()
        barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms_mean = sum(step_ms) / steps
    ms_max = all_max(ms_mean, world)

    # the two calls separately (append, then decode), for the breakdown
    sep = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(min(steps, 100))]
    for e in sep:
        flush.zero_()
        e[0].record(stream)
        if slots.numel():
            wllm.reshape_and_cache(key, value, kc, vc, slots)
        e[1].record(stream)
        wllm.paged_attention_decode(out, q, kc, vc, bt, cl, Hkv, case.scale, bs)
        e[2].record(stream)
    torch.cuda.synchronize()
    app_ms = sum(e[0].elapsed_time(e[1]) for e in sep) / len(sep)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in sep) / len(sep)

    # end to end through the public API with host buffers: the step's inputs
    # staged in one pinned host buffer and copied to the device in one H2D
    # transfer (what a serving loop does: one DMA, not one per tensor), the
    # fused step on views of the device copy, D2H of the output, all inside
    # the events
    h_src = {"q": case.q, "key": case.key, "value": case.value, "bt": bt.cpu(), "cl": case.context_lens,
             "slots": slots.cpu()}
    offs, total = {}, 0
    for n, t in h_src.items():
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    d_v = {}
    for n, t in h_src.items():
        nb = t.numel() * t.element_size()
        h_stage[offs[n]:offs[n] + nb].view(t.dtype).copy_(t.contiguous().view(-1))
        d_v[n] = d_stage[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_src.values())
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(1, min(steps, 500))
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    warm = max(3, args.warmup)
    for i in range(e2e_steps + warm):
        j = i - warm
        flush.zero_()
        if j >= 0:
            e2e_ev[j][0].record(stream)
        d_stage.copy_(h_stage, non_blocking=True)
        wllm.decode_step(out, d_v["q"], d_v["key"], d_v["value"], kc, vc, d_v["slots"], d_v["bt"], d_v["cl"], Hkv,
                         case.scale, bs)
        h_out.copy_(out, non_blocking=True)
        if j >= 0:
            e2e_ev[j][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = all_max(sum(e[0].elapsed_time(e[1]) for e in e2e_ev) / e2e_steps, world)

    fp8 = None
    if fp8_reps > 0:  # (over the compact pool too: the same bytes read, for ncu captures)
        fp8 = fp8_step(args, case, dev, q, key, value, slots, bt, cl, kc, vc, flush, stream, fp8_reps)

    peak, peak_kind = measured_peak()
    alg = case.algorithmic_bytes()
    step_bytes = alg + case.append_bytes()
    achieved = step_bytes / (ms_mean / 1e3) / 1e9
    rec = {
        "workload": case.name, "config": config_of(case, name, part_tokens, pool), "dtype": DTYPE_NAME[case.dtype],
        "steps": steps, "step_us": ms_max * 1e3, "step_median_us": statistics.median(step_ms) * 1e3,
        "tokens_per_s": B * world / (ms_max / 1e3), "algorithmic_bytes": step_bytes,
        "achieved_gbs": achieved, "pct_of_8tbs": 100.0 * achieved / 8000.0,
        "kernel_us": {"step_fused": ms_mean * 1e3, "append_separate": app_ms * 1e3,
                      "decode_separate": dec_ms * 1e3},
        "roofline": {"bound": "hbm", "kernel": "paged_decode_persistent (fused step: append + decode + merge)"
                     if case.dtype != torch.float32 else "append_kernel + paged_decode_kernel (fp32 FMA)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(name) if pool == "full" else None,
                     "algorithmic_bytes": step_bytes},
        "e2e": {"value": B * world / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": int(launches), "launches_per_step": launches / steps,
        "clocks": clocks.summary(),
        "fp8": fp8,
    }
    if rank == 0 and world == 1 and cpu_budget > 0:
        rec["cpu_baseline"] = cpu_oracle_rate(case, cpu_budget)
        if single_budget > 0:
            rec["cpu_baseline"]["single_thread"] = cpu_oracle_rate(case, single_budget, threads=1)
    del kc, vc, q, key, value, slots, bt, cl, out
    torch.cuda.empty_cache()
    return rec


def graph_layers(args, name, rank, dev, flush, stream):
    """Several layers' decode steps (each layer its own K/V pools, the same step
    inputs) back to back, issued eagerly and replayed from one CUDA graph; the
    L2 is flushed between repetitions, outside the events.  Returns per-layer
    times, or None when the layers' pools would not fit the budget."""
    import paged_kv_cache_185_gb300 as wllm

    case = replica_case(name, rank)
    L = args.graph_layers
    if L <= 0 or L * 2 * case.pool_bytes() > (8 << 30) or case.dtype == torch.float32:
        return None
    B, Hq, Hkv, D, bs = case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    q = case.q.to(dev)
    key, value, slots = case.key.to(dev), case.value.to(dev), case.slot_mapping.to(dev)
    bt, cl = case.block_tables.to(dev), case.context_lens.to(dev)
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
        eager, _ = event_times(layers, R, flush, stream)
        graph, _ = event_times(g.replay, R, flush, stream)
        return {"workload": case.name, "layers": L, "us_per_layer": graph * 1e3 / L,
                "eager_us_per_layer": eager * 1e3 / L,
                "note": "layers back to back, each on its own K/V pools; one CUDA graph replay vs eager calls"}
    finally:
        wllm.set_workspace(None)
        del pools


def prefill_bench(args, name, dev, flush, stream):
    """Chunked prefill on the named workload's head geometry: 8 sequences, each
    a 512-token chunk after 0..2048 tokens of context (seeded), timed through
    wllm_paged_attention_prefill (and its fp8-cache form).  FLOPs are the
    causal attention's own (4 * D * (P + 1) per query row at position P),
    against the measured bf16 tensor peak."""
    import numpy as np
    import paged_kv_cache_185_gb300 as wllm

    case = workloads.make_case(name)
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
    R = args.prefill_reps
    ms, _ = event_times(lambda: wllm.paged_attention_prefill(out, q, kc, vc, bt, cl, qsl, case.num_kv_heads,
                                                             case.scale, case.block_size), R, flush, stream)
    fp8_ms = None
    if case.head_dim == 128 or case.block_size >= 16:  # the same chunks over E4M3 codes of the same K/V
        k8 = (kc.float() * 4.0).to(torch.float8_e4m3fn).view(torch.uint8)
        v8 = (vc.float() * 4.0).to(torch.float8_e4m3fn).view(torch.uint8)
        fp8_ms, _ = event_times(lambda: wllm.paged_attention_prefill_fp8(
            out, q, k8, v8, bt, cl, qsl, case.num_kv_heads, case.scale, 0.25, 0.25, case.block_size),
            R, flush, stream)
    flops = 0
    for p0 in prior:
        P = np.arange(int(p0), int(p0) + chunk)
        flops += int(4 * case.head_dim * (P + 1).sum()) * case.num_q_heads
    peak, kind = tensor_peak()
    achieved = flops / (ms / 1e3) / 1e12
    return {"workload": f"{nseq} seqs x {chunk}-token chunks after U[0,2048] context, "
                        f"{case.num_q_heads}/{case.num_kv_heads} heads, D {case.head_dim} ({case.name} heads)",
            "us": ms * 1e3, "tokens_per_s": T / (ms / 1e3),
            "roofline": {"bound": "tensor", "kernel": "paged_prefill_kernel",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_kind": kind, "flops": flops},
            "fp8_cache_us": None if fp8_ms is None else fp8_ms * 1e3,
            "fp8_cache_tflops": None if fp8_ms is None else flops / (fp8_ms / 1e3) / 1e12,
            "reps": R}


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
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    K = args.steps
    with_cpu = world == 1 and not args.no_cpu_baseline

    main = measure(args, args.workload, rank, world, local, dev, flush, stream, K,
                   cpu_budget=args.cpu_budget if with_cpu else 0.0,
                   single_budget=min(3.0, args.cpu_budget) if with_cpu else 0.0,
                   fp8_reps=args.fp8_reps, pool=args.pool)
    per = {}
    names = [] if args.per_workload in ("", "none") else args.per_workload.split(",")
    sub_steps = max(1, min(K, args.sub_steps))
    for name in names:
        if name == args.workload:
            continue
        small = name in ("c0", "c1", "c2")
        per[name] = measure(args, name, rank, world, local, dev, flush, stream, sub_steps,
                            cpu_budget=(3.0 if small else 2.0) if with_cpu else 0.0,
                            single_budget=2.0 if (with_cpu and small) else 0.0,
                            fp8_reps=min(args.fp8_reps, sub_steps))
    graph = (graph_layers(args, args.graph_workload, rank, dev, flush, stream)
             if args.graph_workload not in ("", "none") else None)
    prefill = {}
    for name in ([] if args.prefill_workloads in ("", "none") else args.prefill_workloads.split(",")):
        prefill[name] = prefill_bench(args, name, dev, flush, stream)
    if rank != 0:
        return
    line = {
        "metric": "decode-attn tokens/s", "value": main["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": main["step_us"] / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": main["dtype"],
        "data": "synthetic", "config": main["config"],
        "achieved_gbs": main["achieved_gbs"], "pct_of_8tbs": main["pct_of_8tbs"],
        "kernel_us": main["kernel_us"], "step_median_us": main["step_median_us"],
        "roofline": main["roofline"],
        "cpu_baseline": main.get("cpu_baseline"),
        "e2e": main["e2e"],
        "gpu_launches": main["gpu_launches"],
        "clocks": main["clocks"],
        "fp8": main["fp8"],
        "per_workload": per,
        "graph": graph,
        "prefill": prefill,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="c4", choices=list(workloads.CASE_NAMES),
                    help="the headline workload (default: the long-context batch)")
    ap.add_argument("--per-workload", default="c0,c1,c2,c3,gemma_mqa,bs32",
                    help="comma-separated workloads timed in the same run as sub-records ('none': skip)")
    ap.add_argument("--sub-steps", type=int, default=500, help="timed steps of each per-workload record")
    ap.add_argument("--pool", default="full", choices=["full", "compact"],
                    help="compact: only the referenced blocks on the device (the same bytes read; for ncu)")
    ap.add_argument("--graph-workload", default="c1", help="workload of the CUDA-graph measurement ('none' skips)")
    ap.add_argument("--graph-layers", type=int, default=8,
                    help="layers per CUDA-graph replay for the graph measurement (0: skip)")
    ap.add_argument("--fp8-reps", type=int, default=100,
                    help="repetitions of the fp8-cache measurement (0: skip)")
    ap.add_argument("--prefill-workloads", default="c1,c3",
                    help="head geometries of the chunked-prefill measurement ('none': skip)")
    ap.add_argument("--prefill-reps", type=int, default=50,
                    help="repetitions of the chunked-prefill measurement (0: skip)")
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
