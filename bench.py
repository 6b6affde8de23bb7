"""Benchmark of the paged KV-cache hot path on one GB300 (or N replicas under torchrun).

One step = one decode step of the shared-prompt GQA workload ("gqa_pressure": 100 sequences,
32 query / 8 KV heads x 128, bf16, 16-token blocks, contexts U[256, 4096] raised to >= 513,
25 groups of 4 sharing a 512-token prompt): pa_write_kv of the 100 new tokens, pa_copy_blocks of
the 25 copy-on-write blocks, pa_decode (one kernel incl. the split-K combine), one layer. Inputs are
resident in HBM and larger than L2 (0.7 GB of KV per step against a 129 MB L2); the timed steps
run back to back, and each step alone after an L2 flush (outside the events) is reported beside.

The metric is achieved HBM bandwidth: algorithmic bytes of the step (every distinct KV byte the
attention must read once, the query/output, block tables, split partials written and read back,
and the bytes the movers read and write) divided by the step time, plus decode tokens/s
(sequences per second for this one layer). Run ``python bench.py --help`` for options.

``--impl reference`` times the CPU oracle (the only other implementation; there is no runnable
reference code) on a bounded sample of the same workload.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "gqa_pressure"
SEED = 38 + 2  # seed = 38 + index of the configuration
METRIC = "paged-decode attention: achieved HBM GB/s & % of peak; decode tokens/s"
# GB300 HBM3e bandwidth from NVIDIA's public specification, entered by hand: the "nominal" peak
# printed beside the measured copy peak of MEASURED_PEAKS.json.
NOMINAL_HBM_GBS = 7900.0
L2_BYTES = 129e6  # GB300 L2 capacity, public specification
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
DECODE_SOURCES = ["pa_decode.cuh", "pa_device.cuh", "pa_decode_host.cu", "pa_decode_bf16.cu"]


def split_tokens_for(spec: synth.DecodeSpec) -> int:
    """Context split used by the benchmark (and by the full-size parity tests): 512 tokens for
    16-bit KV, 2048 for E4M3 (the library's own default for these shapes)."""
    return 2048 if synth.ELT_BYTES[spec.kv_dtype] == 1 else 512


# ---------------------------------------------------------------------------- byte accounting

def unique_kv_bytes(case: synth.PagedCase) -> int:
    """Distinct K+V bytes the attention must read: every referenced physical block counted once,
    with as many slots as the longest sequence that reads it has filled."""
    spec = case.spec
    B = spec.block_size
    tables = case.block_tables.cpu().numpy()
    lens = case.ctx_lens.cpu().numpy()
    filled = {}
    for s, L in enumerate(lens):
        nb = (int(L) + B - 1) // B
        for j in range(nb):
            n = min(B, int(L) - j * B)
            b = int(tables[s, j])
            filled[b] = max(filled.get(b, 0), n)
    row = spec.num_kv_heads * spec.head_dim * synth.ELT_BYTES[spec.kv_dtype]
    return 2 * row * sum(filled.values())


def logical_kv_bytes(case: synth.PagedCase) -> int:
    spec = case.spec
    row = spec.num_kv_heads * spec.head_dim * synth.ELT_BYTES[spec.kv_dtype]
    return 2 * row * int(case.ctx_lens.sum())


def decode_bytes(case: synth.PagedCase, split_tokens: int) -> dict:
    spec = case.spec
    lens = case.ctx_lens.cpu().numpy().astype(np.int64)
    B = spec.block_size
    qo = 2 * spec.num_seqs * spec.num_q_heads * spec.head_dim * 2
    tables = 4 * int(((lens + B - 1) // B).sum()) + 4 * spec.num_seqs
    nsplit = (lens + split_tokens - 1) // split_tokens
    multi = nsplit[nsplit > 1]
    partials = 2 * int(multi.sum()) * spec.num_q_heads * (spec.head_dim * 4 + 8)
    kv = unique_kv_bytes(case)
    return {"kv_unique": kv, "kv_logical": logical_kv_bytes(case), "q_out": qo,
            "tables": tables, "partials": partials, "total": kv + qo + tables + partials}


def mover_bytes(case: synth.PagedCase) -> dict:
    spec = case.spec
    row = spec.num_kv_heads * spec.head_dim * synth.ELT_BYTES[spec.kv_dtype]
    write = 2 * 2 * spec.num_seqs * row + 8 * spec.num_seqs      # read new K,V + write slots
    copy = 2 * 2 * case.cow_pairs.shape[0] * case.block_bytes + 8 * case.cow_pairs.shape[0]
    return {"write_kv": write, "copy_blocks": copy}


# ---------------------------------------------------------------------------- helpers

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_38_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    want = decode_source_hash()
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == "pa_decode_kernel" \
                    and parts[1] == workload and parts[2] == want:
                return int(parts[3])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
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
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- our arm

class Step:
    """One decode step of the workload through the library's binding."""

    def __init__(self, case: synth.PagedCase, split_tokens: int):
        import paged_kv_cache_38_gb300 as pa

        self.pa = pa
        self.case = case
        self.split = split_tokens
        self.max_ctx = int(case.ctx_lens.max())
        self.out = torch.empty_like(case.q)
        args = pa.make_decode_args(case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.ctx_lens, self.out, scale=case.scale,
                                   max_ctx_len=self.max_ctx, split_tokens=split_tokens)
        need = pa.pa_decode_workspace_size(args)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=case.q.device)
        self.max_splits = (self.max_ctx + split_tokens - 1) // split_tokens
        self.launches = 3  # write-KV, copy-on-write, decode (split-K combine is in-kernel)

    def decode(self, q=None, block_tables=None, ctx_lens=None, out=None):
        c = self.case
        return self.pa.pa_decode(c.q if q is None else q, c.k_pool, c.v_pool,
                                 c.block_tables if block_tables is None else block_tables,
                                 c.ctx_lens if ctx_lens is None else ctx_lens, c.scale,
                                 out=self.out if out is None else out, k_scale=c.k_scale,
                                 v_scale=c.v_scale, max_ctx_len=self.max_ctx,
                                 split_tokens=self.split, workspace=self.ws)

    def run(self):
        c = self.case
        self.pa.pa_write_kv(c.k_new, c.v_new, c.k_pool, c.v_pool, c.slot_mapping)
        if c.cow_pairs.numel():
            self.pa.pa_copy_blocks([c.k_pool], [c.v_pool], c.cow_pairs)
        return self.decode()


def capture_graph(fn) -> "torch.cuda.CUDAGraph":
    """Capture fn's launches (already warmed up) into a CUDA graph on a side stream."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_steps(fn, steps: int, flush: torch.Tensor):
    """Per-step CUDA-event times (ms) on the current stream, L2 flushed before each step."""
    times = []
    stream = torch.cuda.current_stream()
    for _ in range(steps):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


def run_ours(args, world, rank, local) -> None:
    import paged_kv_cache_38_gb300 as pa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pa.lib()
    spec = synth.SPECS[args.workload]
    case = synth.make_case(spec, seed=SEED, device=dev, logical=False, poison=False)
    split = args.split_tokens or split_tokens_for(spec)
    step = Step(case, split)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    dbytes = decode_bytes(case, split)
    mbytes = mover_bytes(case)
    step_bytes = dbytes["total"] + mbytes["write_kv"] + mbytes["copy_blocks"]

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    # The step's four launches are replayed from a CUDA graph so that the GPU does not wait on
    # Python between them; the eager (one binding call per launch) time is reported beside it.
    step_graph = capture_graph(step.run)
    decode_graph = capture_graph(step.decode)
    for _ in range(args.warmup):
        step_graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K steps back to back, barrier + synchronize on both sides. The pool is
    # 5x the L2 and every step streams it from DRAM (ncu without cache control between launches
    # reads 710 MB of DRAM per decode, as much as with L2 flushed), so no flush separates them;
    # each step alone after an L2 flush is reported beside (ms_per_step_after_l2_flush).
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(args.steps):
            step_graph.replay()
        ev1.record()
        ev1.synchronize()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_per_step = total_ms / args.steps
    flush_step_ms = statistics.mean(time_steps(step_graph.replay, args.steps, flush))
    eager_ms = statistics.mean(time_steps(step.run, args.steps, flush))

    # ---- the decode call alone (one kernel launch through the C ABI), same stream.
    # (a) Back to back, no flush in between: the inputs (the pool) are 5x the L2, so each
    # launch streams its bytes from DRAM; a launch's setup overlaps the previous launch, as in a
    # serving loop. This is the kernel's per-launch time (it matches the kernel duration ncu
    # reports) and the roofline's denominator.
    reps = max(args.steps, 10)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step.decode()
    a.record()
    for _ in range(reps):
        step.decode()
    b.record()
    b.synchronize()
    dec_b2b_ms = a.elapsed_time(b) / reps
    # (b) Each launch alone after an L2 flush (eager, and replayed from a CUDA graph): adds the
    # ~5 us an isolated launch takes to start after the flush kernel (an empty kernel of the
    # same grid measures 4.8 us between events there); reported beside.
    dec_ms = statistics.mean(time_steps(step.decode, reps, flush))
    dec_graph_ms = statistics.mean(time_steps(decode_graph.replay, reps, flush))

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, case, args.steps, flush, step_bytes)

    peaks = load_peaks()
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    dec_gbs = dbytes["total"] / (dec_b2b_ms * 1e-3) / 1e9
    dec_flush_gbs = dbytes["total"] / (dec_ms * 1e-3) / 1e9
    extra = {}
    if rank == 0 and not args.quick:
        extra = run_extras(args, dev, flush, peaks)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, split, args.cpu_seconds)

    if rank != 0:
        return
    traffic = recorded_traffic(args.workload)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded block pools shaped like the pages' workloads)",
        "config": workload_config(args.workload, spec, case, split, world),
        "pct_of_peak": round(100 * value / world / peaks["hbm_gbs"], 1),
        "pct_of_nominal": round(100 * value / world / NOMINAL_HBM_GBS, 1),
        "decode_tokens_per_s": round(world * spec.num_seqs / (ms_per_step * 1e-3), 1),
        "ms_per_step_after_l2_flush": round(flush_step_ms, 4),
        "pct_of_peak_after_l2_flush": round(
            100 * step_bytes / (flush_step_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 1),
        "ms_per_step_eager_after_l2_flush": round(eager_ms, 4),
        "bytes_per_step": {**dbytes, **mbytes, "total": step_bytes},
        "roofline": {"bound": "hbm", "kernel": "pa_decode_kernel",
                     "achieved": round(dec_gbs, 1), "peak": peaks["hbm_gbs"],
                     "peak_source": peaks["source"], "unit": "GB/s",
                     "frac": round(dec_gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "nominal": {"peak": NOMINAL_HBM_GBS, "unit": "GB/s",
                                 "frac": round(dec_gbs / NOMINAL_HBM_GBS, 4),
                                 "source": "GB300 HBM3e specification (nominal)"},
                     "algorithmic_bytes": dbytes["total"],
                     "ms_per_launch": round(dec_b2b_ms, 4),
                     "timing": f"{reps} launches back to back, CUDA events on the launch stream; "
                               "pool 5x L2, not flushed between launches",
                     "after_l2_flush": {
                         "ms_per_launch": round(dec_ms, 4),
                         "ms_per_launch_graph": round(dec_graph_ms, 4),
                         "achieved": round(dec_flush_gbs, 1),
                         "frac": round(dec_flush_gbs / peaks["hbm_gbs"], 4),
                         "timing": "each launch alone, L2 flushed before it (outside the events)"}},
        "gpu_launches": step.launches * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if extra:
        line["extra"] = extra
    print(json.dumps(line))


def run_e2e(step: Step, case: synth.PagedCase, steps: int, flush, step_bytes: int) -> dict:
    """Same step with its inputs copied from pinned host memory and its output read back,
    every step. The step's inputs sit in one pinned staging buffer (one host-to-device copy),
    the output returns in one device-to-host copy, and copies and kernels replay from one CUDA
    graph (eagerly if the capture is refused)."""
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "ctx_lens", "cow_pairs")
    srcs = {k: getattr(case, k) for k in names}
    offs, total = {}, 0
    for k, t in srcs.items():
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256

    def view(buf, k):
        t = srcs[k]
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)

    hbuf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device=case.q.device)
    for k in names:
        view(hbuf, k).copy_(srcs[k].cpu())
    dev = {k: view(dbuf, k) for k in names}
    out_dev = torch.empty_like(case.q)
    out_host = torch.empty(case.q.shape, dtype=case.q.dtype).pin_memory()
    pa = step.pa
    c = case

    def one():
        dbuf.copy_(hbuf, non_blocking=True)
        pa.pa_write_kv(dev["k_new"], dev["v_new"], c.k_pool, c.v_pool, dev["slot_mapping"])
        if c.cow_pairs.numel():
            pa.pa_copy_blocks([c.k_pool], [c.v_pool], dev["cow_pairs"])
        step.decode(q=dev["q"], block_tables=dev["block_tables"], ctx_lens=dev["ctx_lens"],
                    out=out_dev)
        out_host.copy_(out_dev, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    fn, graphed = one, False
    try:
        g = capture_graph(one)
        fn, graphed = g.replay, True
    except RuntimeError:
        torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    b.synchronize()
    ms = a.elapsed_time(b) / steps
    ms_flush = statistics.mean(time_steps(fn, steps, flush))
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "ms_per_step_after_l2_flush": round(ms_flush, 4),
            "h2d_bytes_per_step": total,
            "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
            "copies_per_step": 2, "graph": graphed}


# ---------------------------------------------------------------------------- other workloads

def run_extras(args, dev, flush, peaks) -> dict:
    """The other configurations of the pages: MHA fp16, FP8 long contexts, the preemption swap
    and a large copy-on-write batch. Each is timed like the main step; all report GB/s."""
    import paged_kv_cache_38_gb300 as pa

    res = {}
    for name in ("mha7b", "fp8_long"):
        spec = synth.SPECS[name]
        case = synth.make_case(spec, seed=SEED - 2 + (1 if name == "mha7b" else 3), device=dev,
                               logical=False, poison=False)
        split = split_tokens_for(spec)
        st = Step(case, split)
        for _ in range(3):
            st.decode()
        # back to back (pools larger than L2), as the main roofline; after an L2 flush beside
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(20):
            st.decode()
        e.record()
        e.synchronize()
        t = a.elapsed_time(e) / 20
        tf = statistics.mean(time_steps(st.decode, 10, flush))
        b = decode_bytes(case, split)
        res[name] = {"decode_ms": round(t, 4), "gbs": round(b["total"] / (t * 1e-3) / 1e9, 1),
                     "pct_of_peak": round(100 * b["total"] / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 1),
                     "pct_of_nominal": round(100 * b["total"] / (t * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 1),
                     "tokens_per_s": round(spec.num_seqs / (t * 1e-3), 1),
                     "decode_ms_after_l2_flush": round(tf, 4),
                     "pct_of_peak_after_l2_flush":
                         round(100 * b["total"] / (tf * 1e-3) / 1e9 / peaks["hbm_gbs"], 1),
                     "split_tokens": split, "bytes": b["total"]}
        del case, st
        torch.cuda.empty_cache()
    res["preemption_swap"] = run_swap_bench(dev)
    res["copy_blocks_large"] = run_copy_bench(dev, flush, peaks)
    res["write_kv_fp8"] = run_quantise_bench(dev, flush, peaks)
    res["scheduler"] = run_scheduler_bench(dev)
    res["block_size_sweep"] = run_block_sweep(dev, flush, peaks)
    res["prefill"] = run_prefill_bench(dev, flush, peaks)
    return res


def prefill_flops(ctx_lens, q_starts, num_q_heads: int, head_dim: int) -> int:
    """Causal attention work of a prefill: query i of a chunk of n over L positions sees
    L - n + i + 1 keys; each key costs 2 D flops for Q K^T and 2 D for P V, per query head."""
    total = 0
    for s in range(len(ctx_lens)):
        L, n = int(ctx_lens[s]), int(q_starts[s + 1] - q_starts[s])
        first = L - n + 1
        total += n * first + n * (n - 1) // 2
    return 4 * head_dim * num_q_heads * total


def run_prefill_bench(dev, flush, peaks) -> dict:
    """pa_prefill on the GQA geometry (32 q / 8 kv heads x 128, bf16, 16-token blocks):
    16 whole 2,048-token prompts, and 64 chunks of 512 new tokens on 1,536-token histories
    (chunked prefill / recompute); then other head geometries on 8 whole 2,048-token prompts:
    MHA (32 / 32 x 128, f16), a group of 8 (64 / 8 x 128) and head_dim 64 (32 / 8 x 64); and the
    16 prompts over an E4M3 cache with bf16 queries (the FP8 workload's recompute path, f16
    tensor-core operands). Causal flops per second against the measured bf16 GEMM peak (f16
    runs at the same dense rate)."""
    import paged_kv_cache_38_gb300 as pa

    out = {}
    for name, lens, chunk, hq, hkv, d, dt, kvdt in (
            ("prompts_16x2048", [2048] * 16, 2048, 32, 8, 128, "bf16", "bf16"),
            ("chunks_64x512_on_2048", [2048] * 64, 512, 32, 8, 128, "bf16", "bf16"),
            ("mha_prompts_8x2048", [2048] * 8, 2048, 32, 32, 128, "f16", "f16"),
            ("g8_prompts_8x2048", [2048] * 8, 2048, 64, 8, 128, "bf16", "bf16"),
            ("d64_prompts_8x2048", [2048] * 8, 2048, 32, 8, 64, "bf16", "bf16"),
            ("e4m3_prompts_16x2048", [2048] * 16, 2048, 32, 8, 128, "bf16", "e4m3")):
        spec = synth.DecodeSpec(name, len(lens), hq, hkv, d, 16, kvdt, dt, ctx_lens=tuple(lens))
        case = synth.make_case(spec, seed=SEED, device=dev, logical=False, poison=False)
        n = [chunk] * len(lens)
        qs = torch.tensor(np.concatenate([[0], np.cumsum(n)]), dtype=torch.int32, device=dev)
        q = torch.randn(int(qs[-1]), hq, d, device=dev).to(synth.TORCH_DTYPES[dt])
        o = torch.empty_like(q)
        call = lambda: pa.pa_prefill(q, case.k_pool, case.v_pool, case.block_tables,  # noqa: E731
                                     case.ctx_lens, qs, case.scale, out=o, max_q_len=chunk,
                                     k_scale=case.k_scale, v_scale=case.v_scale)
        for _ in range(3):
            call()
        t = statistics.mean(time_steps(call, 10, flush))
        fl = prefill_flops(lens, qs.cpu().numpy(), hq, d)
        tf = fl / (t * 1e-3) / 1e12
        out[name] = {"ms": round(t, 4), "tflops": round(tf, 1),
                     "pct_of_bf16_peak": round(100 * tf / peaks["bf16_tflops"], 1),
                     "tokens_per_s": round(int(qs[-1]) / (t * 1e-3), 1)}
        del case, q, o
        torch.cuda.empty_cache()
    return out


def run_block_sweep(dev, flush, peaks) -> dict:
    """Block sizes 8, 16, 32, 64 (the summary page's ablation: decode cost and swap bandwidth
    against block size). Decode: the GQA workload rebuilt at each block size (same contexts and
    512-token shared prompts). Swap: the preemption victim's 1,500 tokens over 32 layers of
    8 kv heads x 128 bf16, out and back, direct (mapped pinned memory) and staged (one copy)."""
    import paged_kv_cache_38_gb300 as pa

    out = {}
    for B in (8, 16, 32, 64):
        spec = synth.SPECS["gqa_pressure"].scaled(name=f"gqa_pressure_b{B}", block_size=B)
        case = synth.make_case(spec, seed=SEED, device=dev, logical=False, poison=False)
        split = split_tokens_for(spec)
        st = Step(case, split)
        for _ in range(3):
            st.decode()
        t = statistics.mean(time_steps(st.decode, 10, flush))
        byts = decode_bytes(case, split)["total"]
        row = {"decode_us": round(t * 1e3, 1), "decode_gbs": round(byts / (t * 1e-3) / 1e9, 1),
               "decode_pct_of_peak": round(100 * byts / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 1)}
        del case, st
        torch.cuda.empty_cache()
        # swap of one 1,500-token sequence over 32 layers
        layers, hkv, d = 32, 8, 128
        n = -(-1500 // B)
        nblk = 2 * n + 8
        kp = [torch.empty(nblk, hkv, B, d, dtype=torch.bfloat16, device=dev) for _ in range(layers)]
        vp = [torch.empty_like(kp[0]) for _ in range(layers)]
        perm = np.random.default_rng(SEED + B).permutation(nblk).astype(np.int32)
        out_ids, in_ids = perm[:n], perm[n:2 * n]
        bb = hkv * B * d * 2
        total = n * layers * 2 * bb
        host = torch.empty(total, dtype=torch.uint8).pin_memory()
        staging = torch.empty(total, dtype=torch.uint8, device=dev)
        for mode, stg in (("direct", None), ("staged", staging)):
            ts_o, ts_i = [], []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                pa.pa_swap_blocks(kp, vp, host, out_ids, pa.PA_SWAP_OUT, staging=stg)
                b.record()
                b.synchronize()
                ts_o.append(a.elapsed_time(b))
                a.record()
                pa.pa_swap_blocks(kp, vp, host, in_ids, pa.PA_SWAP_IN, staging=stg)
                b.record()
                b.synchronize()
                ts_i.append(a.elapsed_time(b))
            row[f"swap_{mode}_out_gbs"] = round(total / (min(ts_o) * 1e-3) / 1e9, 1)
            row[f"swap_{mode}_in_gbs"] = round(total / (min(ts_i) * 1e-3) / 1e9, 1)
        row["swap_bytes_each_way"] = total
        row["swap_blocks"] = n
        out[f"b{B}"] = row
        del kp, vp, host, staging
        torch.cuda.empty_cache()
    return out


def run_scheduler_bench(dev) -> dict:
    """The C++ scheduler driving the kernels: the GQA workload's geometry (32 q / 8 kv heads x
    128, bf16, 16-token blocks) with 25 groups of 4 samples sharing a 512-token prompt plus 60
    single requests, in a pool of 12,000 blocks. Reports the host time of one scheduling step
    and the served loop (plan, moves, KV writes, decode) over 150 steps, eager."""
    import paged_kv_cache_38_gb300 as pa
    from paged_kv_cache_38_gb300 import scheduler as sch

    hq, hkv, d, b, nblk = 32, 8, 128, 16, 12000
    rng = np.random.default_rng(SEED)

    def requests(s):
        for r in range(25):
            s.add_request(r, 512 + int(rng.integers(1, 64)), 400, 4)
        for r in range(25, 85):
            s.add_request(r, int(rng.integers(256, 2048)), 400, 1)

    s = sch.Scheduler(nblk, b, 512, 256, sch.SWAP, 4 * nblk)
    requests(s)
    host = []
    for _ in range(150):
        t0 = time.perf_counter()
        s.step()
        host.append(time.perf_counter() - t0)
    # the served loop on the GPU
    s = sch.Scheduler(nblk, b, 512, 256, sch.SWAP, 4 * nblk)
    rng = np.random.default_rng(SEED)
    requests(s)
    g = torch.Generator(device=dev).manual_seed(SEED)
    rows = 4096
    k_rows = torch.randn(rows, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    v_rows = torch.randn(rows, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    kp = torch.empty(nblk, hkv, b, d, dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    cpu_pool = torch.empty(1, 1, 2, hkv * b * d * 2, dtype=torch.uint8).pin_memory()
    q_all = torch.randn(512, hq, d, generator=g, device=dev).to(torch.bfloat16)
    ws = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    tokens, writes, steps = 0, 0, 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(150):
        plan = s.step()
        if len(plan.swap_out_np) or len(plan.swap_in_np):
            raise RuntimeError("the served-loop workload is sized to run without swapping")
        sch.execute_moves(plan, [kp], [vp], cpu_pool)
        if len(plan.slots_np):
            idx = torch.from_numpy(plan.slots_np % rows).to(dev, non_blocking=True)
            pa.pa_write_kv(k_rows[idx], v_rows[idx], kp, vp,
                           torch.from_numpy(plan.slots_np).to(dev, non_blocking=True))
        n = len(plan.seq_ids_np)
        if n:
            bt = torch.from_numpy(plan.tables_np).to(dev, non_blocking=True)
            cl = torch.from_numpy(plan.ctx_np).to(dev, non_blocking=True)
            pa.pa_decode(q_all[:n], kp, vp, bt, cl, d ** -0.5, max_ctx_len=int(plan.ctx_np.max()),
                         workspace=ws)
        tokens += n
        writes += len(plan.slots_np)
        steps += 1
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    res = {"requests": 85, "sequences": 160, "pool_blocks": nblk,
           "host_step_us_median": round(1e6 * statistics.median(host), 1),
           "served_steps": steps, "served_ms_per_step": round(1e3 * wall / steps, 3),
           "served_decode_tokens_per_s": round(tokens / wall, 1),
           "kv_positions_written": writes}
    del kp, vp, ws
    torch.cuda.empty_cache()
    return res


def run_quantise_bench(dev, flush, peaks) -> dict:
    """pa_write_kv_fp8 (bf16 in, E4M3 pool) for a prefill-sized batch of 32,768 tokens of the
    FP8 workload's geometry (8 kv heads x 128), plus the 256-token decode step as a latency."""
    import paged_kv_cache_38_gb300 as pa

    hkv, d, b, ntok = 8, 128, 16, 32768
    nblk = ntok // b + 64
    g = torch.Generator(device=dev).manual_seed(SEED)
    k = torch.randn(ntok, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(ntok, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    kp = torch.empty(nblk, hkv, b, d, dtype=torch.uint8, device=dev)
    vp = torch.empty_like(kp)
    slots = torch.from_numpy(np.random.default_rng(SEED).permutation(nblk * b)[:ntok]).to(dev)
    ks, vs = float(k.float().abs().max()) / 448.0, float(v.float().abs().max()) / 448.0
    call = lambda n: pa.pa_write_kv_fp8(k[:n], v[:n], kp, vp, slots[:n], ks, vs)  # noqa: E731
    call(ntok)
    t = statistics.mean(time_steps(lambda: call(ntok), 10, flush))
    t_small = statistics.mean(time_steps(lambda: call(256), 20, flush))
    byts = ntok * (2 * hkv * d * 2 + 2 * hkv * d + 8)  # bf16 read, E4M3 written, slot read
    gbs = byts / (t * 1e-3) / 1e9
    res = {"tokens": ntok, "bytes": byts, "ms": round(t, 4), "gbs": round(gbs, 1),
           "pct_of_peak": round(100 * gbs / peaks["hbm_gbs"], 1),
           "step_256_tokens_us": round(t_small * 1e3, 2)}
    # the same tokens through pa_write_kv into a bf16 pool (what a prefill writes without FP8)
    kp16 = torch.empty(nblk, hkv, b, d, dtype=torch.bfloat16, device=dev)
    vp16 = torch.empty_like(kp16)
    call16 = lambda: pa.pa_write_kv(k, v, kp16, vp16, slots)  # noqa: E731
    call16()
    t16 = statistics.mean(time_steps(call16, 10, flush))
    byts16 = ntok * (2 * hkv * d * 2 * 2 + 8)  # bf16 read and written, slot read
    res["bf16_write_kv"] = {"bytes": byts16, "ms": round(t16, 4),
                            "gbs": round(byts16 / (t16 * 1e-3) / 1e9, 1),
                            "pct_of_peak": round(100 * byts16 / (t16 * 1e-3) / 1e9 / peaks["hbm_gbs"], 1)}
    del k, v, kp, vp, kp16, vp16
    torch.cuda.empty_cache()
    return res


def run_swap_bench(dev) -> dict:
    import paged_kv_cache_38_gb300 as pa

    spec = synth.SPECS["preemption"]
    case = synth.make_case(spec, seed=SEED + 3, device=dev, logical=False, poison=False)
    victim = spec.num_seqs - 1
    out_ids, in_ids = synth.swap_plan(case, victim, seed=SEED)
    n, L, bb = len(out_ids), spec.num_layers, case.block_bytes
    total = n * L * 2 * bb
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    staging = torch.empty(total, dtype=torch.uint8, device=dev)
    res = {"blocks": n, "bytes_each_way": total}

    def timed(fn, reps=5):
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return min(ts), statistics.mean(ts)

    # host link peak: one large pinned copy each way
    big = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    big_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    d2h_ms, _ = timed(lambda: big_h.copy_(big, non_blocking=True))
    h2d_ms, _ = timed(lambda: big.copy_(big_h, non_blocking=True))
    res["link_peak_d2h_gbs"] = round((1 << 30) / (d2h_ms * 1e-3) / 1e9, 1)
    res["link_peak_h2d_gbs"] = round((1 << 30) / (h2d_ms * 1e-3) / 1e9, 1)
    del big, big_h
    ref = None
    for mode, stg in (("direct", None), ("staged", staging)):
        o_ms, _ = timed(lambda: pa.pa_swap_blocks(case.k_pools, case.v_pools, host, out_ids,
                                                  pa.PA_SWAP_OUT, staging=stg))
        i_ms, _ = timed(lambda: pa.pa_swap_blocks(case.k_pools, case.v_pools, host, in_ids,
                                                  pa.PA_SWAP_IN, staging=stg))
        res[f"{mode}_out_ms"] = round(o_ms, 3)
        res[f"{mode}_in_ms"] = round(i_ms, 3)
        res[f"{mode}_out_gbs"] = round(total / (o_ms * 1e-3) / 1e9, 1)
        res[f"{mode}_in_gbs"] = round(total / (i_ms * 1e-3) / 1e9, 1)
    # bit-exact round trip and an identical resumed decode
    bt = case.block_tables.clone()
    split = split_tokens_for(spec)
    st = Step(case, split)
    before = st.decode().clone()
    pa.pa_swap_blocks(case.k_pools, case.v_pools, host, out_ids, pa.PA_SWAP_OUT)
    for p in case.k_pools + case.v_pools:
        p.view(torch.uint8).view(case.num_blocks, -1)[torch.from_numpy(out_ids).long().to(dev)] = 0
    pa.pa_swap_blocks(case.k_pools, case.v_pools, host, in_ids, pa.PA_SWAP_IN)
    bt[victim, :n] = torch.from_numpy(in_ids).to(dev)
    after = st.decode(block_tables=bt).clone()
    res["round_trip_decode_bit_exact"] = bool(torch.equal(before[victim], after[victim]))
    res["vs_pages_context"] = "pages: ~3 ms each way for 188 MiB over PCIe Gen5 x16 (estimate)"
    del case, st, staging, host
    torch.cuda.empty_cache()
    return res


def run_copy_bench(dev, flush, peaks, layers: int = 32) -> dict:
    """pa_copy_blocks at the preemption geometry: 4,096 disjoint pairs x 32 layers, plus the
    25-pair step of the GQA workload as a latency figure."""
    import paged_kv_cache_38_gb300 as pa

    nblk, bb = 8192 + 64, 32 * 1024
    k = [torch.empty(nblk, bb, dtype=torch.uint8, device=dev) for _ in range(layers)]
    v = [torch.empty(nblk, bb, dtype=torch.uint8, device=dev) for _ in range(layers)]
    perm = torch.from_numpy(np.random.default_rng(SEED).permutation(nblk)[:8192].astype(np.int32))
    pairs = torch.stack([perm[:4096], perm[4096:]], 1).contiguous().to(dev)
    moved = 2 * 2 * 4096 * layers * bb
    pa.pa_copy_blocks(k, v, pairs)
    t = statistics.mean(time_steps(lambda: pa.pa_copy_blocks(k, v, pairs), 5, flush))
    small = pairs[:25].contiguous()
    ts = statistics.mean(time_steps(lambda: pa.pa_copy_blocks(k[:1], v[:1], small), 20, flush))
    gbs = moved / (t * 1e-3) / 1e9
    res = {"pairs": 4096, "layers": layers, "bytes_moved": moved, "ms": round(t, 3),
           "gbs": round(gbs, 1), "pct_of_peak": round(100 * gbs / peaks["hbm_gbs"], 1),
           "cow_25_pairs_us": round(ts * 1e3, 2)}
    del k, v
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------- CPU oracle

def cpu_baseline(case: synth.PagedCase, split: int, seconds: float) -> dict:
    """The fp64 oracle as it stands over a seeded sample of the step's sequences (whole step:
    write, copy, decode), scaled to the same GB/s metric: on all host cores (the line's value)
    and on one core, each for about ``seconds``."""
    import oracle

    orc = oracle.load()
    spec = case.spec
    kp = case.k_pool.cpu().view(torch.uint8).numpy().reshape(-1).copy()
    vp = case.v_pool.cpu().view(torch.uint8).numpy().reshape(-1).copy()
    q = case.q.cpu()
    bt, cl = case.block_tables.cpu(), case.ctx_lens.cpu()
    row = spec.num_kv_heads * spec.head_dim * synth.ELT_BYTES[spec.kv_dtype]

    def rate(threads: int, chunk: int) -> dict:
        order = np.random.default_rng(SEED).permutation(spec.num_seqs)
        done, t0, byts = 0, time.perf_counter(), 0
        orc.write_kv(case.k_new.cpu(), case.v_new.cpu(), kp, vp, case.slot_mapping.cpu(),
                     num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                     block_size=spec.block_size, kv_dtype=spec.kv_dtype)
        byts += 2 * 2 * row * spec.num_seqs
        while done < spec.num_seqs and time.perf_counter() - t0 < seconds:
            idx = torch.as_tensor(order[done:done + chunk], dtype=torch.long)
            orc.decode(q[idx], kp, vp, bt[idx], cl[idx], q_dtype=spec.q_dtype,
                       kv_dtype=spec.kv_dtype, num_q_heads=spec.num_q_heads,
                       num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                       block_size=spec.block_size, scale=case.scale, num_threads=threads)
            byts += (2 * row * int(cl[idx].sum())
                     + 2 * len(idx) * spec.num_q_heads * spec.head_dim * 2)
            done += len(idx)
        el = time.perf_counter() - t0
        return {"value": round(byts / el / 1e9, 3), "seconds": round(el, 2), "seqs": done}

    cores = orc.max_threads()
    allc = rate(0, 4)
    one = rate(1, 1)
    sample = ("write_kv of the step + oracle decode of {n} of %d sequences (seeded order), "
              "KV, q and output bytes per second" % spec.num_seqs)
    return {"value": allc["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "seconds": allc["seconds"], "sample": sample.format(n=allc["seqs"]),
            "single_thread": {"value": one["value"], "unit": "GB/s", "cores": 1,
                              "seconds": one["seconds"], "sample": sample.format(n=one["seqs"])}}


def workload_config(name: str, spec: synth.DecodeSpec, case: synth.PagedCase, split: int,
                    world: int) -> dict:
    """The `config` object of both arms' JSON lines."""
    return {
        "workload": (f"{name}: {spec.num_seqs} seqs, {spec.num_q_heads} q / "
                     f"{spec.num_kv_heads} kv heads x {spec.head_dim}, {spec.kv_dtype} KV, "
                     f"block {spec.block_size}, ctx U{list(spec.ctx_range)} (>= "
                     f"{spec.shared_prompt + 1}), {spec.num_seqs // spec.group_size} groups x "
                     f"{spec.group_size} share a {spec.shared_prompt}-token prompt, "
                     f"{case.cow_pairs.shape[0]} CoW copies/step, 1 layer"),
        "step": "pa_write_kv + pa_copy_blocks + pa_decode (split-K combine in-kernel), "
                "replayed from a CUDA graph",
        "split_tokens": split, "num_blocks": case.num_blocks,
        "ctx_tokens": int(case.ctx_lens.sum()),
        "l2": (f"steps back to back, inputs larger than L2: each step reads "
               f"{unique_kv_bytes(case) / 1e6:.0f} MB of KV, {unique_kv_bytes(case) / L2_BYTES:.1f}x "
               f"the L2; the same step after an untimed L2 flush is reported beside"),
        "parallelism": f"replicas x{world}",
    }


def run_reference(args, world, rank) -> None:
    """Reference arm: the CPU oracle timed on a bounded sample of the same workload. The
    sample (sequences per step) is sized from a short calibration so that the whole run of
    warm-up and timed steps takes about --ref-seconds."""
    if rank != 0:
        return
    import oracle

    spec = synth.SPECS[args.workload]
    case = synth.make_case(spec, seed=SEED, device="cpu", logical=False, poison=False)
    split = args.split_tokens or split_tokens_for(spec)
    orc = oracle.load()
    kp = case.k_pool.view(torch.uint8).numpy().reshape(-1).copy()
    vp = case.v_pool.view(torch.uint8).numpy().reshape(-1).copy()
    rng = np.random.default_rng(SEED)
    row = spec.num_kv_heads * spec.head_dim * synth.ELT_BYTES[spec.kv_dtype]

    def one(seqs):
        idx = torch.as_tensor(seqs, dtype=torch.long)
        orc.write_kv(case.k_new[idx], case.v_new[idx], kp, vp, case.slot_mapping[idx],
                     num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                     block_size=spec.block_size, kv_dtype=spec.kv_dtype)
        orc.decode(case.q[idx], kp, vp, case.block_tables[idx], case.ctx_lens[idx],
                   q_dtype=spec.q_dtype, kv_dtype=spec.kv_dtype, num_q_heads=spec.num_q_heads,
                   num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                   block_size=spec.block_size, scale=case.scale)
        return 2 * row * int(case.ctx_lens[idx].sum()) + 4 * len(seqs) * row

    t0 = time.perf_counter()
    one(rng.choice(spec.num_seqs, 2, replace=False))
    per_seq = (time.perf_counter() - t0) / 2
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    sample = int(min(spec.num_seqs, max(1, per_step // max(per_seq, 1e-9))))
    for _ in range(args.warmup):
        one(rng.choice(spec.num_seqs, sample, replace=False))
    t0 = time.perf_counter()
    byts = 0
    for _ in range(args.steps):
        byts += one(rng.choice(spec.num_seqs, sample, replace=False))
    el = time.perf_counter() - t0
    value = byts / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, spec, case, split, world),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": orc.max_threads(),
                         "kind": "oracle",
                         "sample": f"{sample} of {spec.num_seqs} seeded sequences per step "
                                   f"(sized for ~{args.ref_seconds:g} s in all): write_kv + "
                                   f"decode, KV bytes read per second"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.SPECS))
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--quick", action="store_true", help="skip the other configurations")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="time budget of the reference arm's warm-up and timed steps")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill benches and print their result")
    ap.add_argument("--swap-only", action="store_true",
                    help="run only the 188 MiB preemption swap bench and print its result "
                         "(a small case for profiling)")
    ap.add_argument("--quantise-only", action="store_true",
                    help="run only the 32,768-token pa_write_kv_fp8 / pa_write_kv bench and print "
                         "its result (a small case for profiling)")
    ap.add_argument("--copy-only-layers", type=int, default=0,
                    help="run only the 4,096-pair pa_copy_blocks bench with this many layers "
                         "(a small case for profiling) and print its result")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.copy_only_layers > 0 or args.prefill_only or args.quantise_only or args.swap_only:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
        if args.prefill_only:
            print(json.dumps(run_prefill_bench(dev, flush, load_peaks())))
        elif args.quantise_only:
            print(json.dumps(run_quantise_bench(dev, flush, load_peaks())))
        elif args.swap_only:
            print(json.dumps(run_swap_bench(dev)))
        else:
            print(json.dumps(run_copy_bench(dev, flush, load_peaks(), layers=args.copy_only_layers)))
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
