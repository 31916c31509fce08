"""Benchmark of one paged-KV decode step on GB300.

A step is the whole hot path for one decode layer of one batch:
slot-mapping cache write of the batch's new K/V, split-KV decode attention
through the block tables (partition count chosen by the library), and the
log-sum-exp combine.  Inputs are seeded synthetic tensors shaped like the
workload named by --workload (default: the Qwen2.5-7B-shaped layer, B=8,
Hq=28, Hkv=4, D=128, every L=4096, 16-token blocks).

Timing: every graph of the timed region replayed once and W warm-up steps,
then exactly K steps between a barrier and a device synchronise on each side,
timed with CUDA events on the launching stream.  The K steps are replayed
from CUDA graphs that hold exactly those steps, queued while the GPU spins
for a head start, and consecutive steps rotate over enough copies of the KV
pool that the data a step reads was evicted from the 129 MB L2 before it is
read again.  A step that is one launch (the default fused step) has its
kernel duration taken as the timed region over the launches; other steps
sample the decode kernel with events recorded around it in separate graphs
after the timed region.  The line's "configs" object measures every config
of the metric (see measure_configs).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "qwen2.5-7b-bs16"
L2_BYTES = 129 * 1000 * 1000
GPU_HEADSTART_CYCLES = 400_000   # ~0.2 ms of GPU spin before a timed region
METRIC = "paged decode attention: achieved HBM TB/s (% of ~8 TB/s) and us/call"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--splits", type=int, default=0, help="0 = library's automatic choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU work for the oracle baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = min(steps, 500)")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="total oracle time of --impl reference, spread over its steps")
    ap.add_argument("--unfused", action="store_true",
                    help="time pa_cache_write + pa_decode_splitkv instead of pa_decode_step")
    ap.add_argument("--configs", choices=["main", "none"], default="main",
                    help="also measure every config of the metric (per-call latency, steady "
                         "state, cache write, oracle at 1 and all cores) into the line's 'configs'")
    ap.add_argument("--config-oracle-seconds", type=float, default=0.6,
                    help="CPU time per oracle sample in the configs sweep")
    return ap.parse_args()


# ----------------------------------------------------------------- utilities
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source with comments removed and whitespace collapsed.

    String and character literals are kept as written, so a change to code
    (or to an inline-asm string) changes the result and a comment edit does not.
    """
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def csrc_hash() -> str:
    """Fingerprint of the kernels' code (comments and layout ignored)."""
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "paged_kv_decode_cache_gb300", "csrc", "*"))):
        with open(p, encoding="utf-8", errors="replace") as f:
            h.update(os.path.basename(p).encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernels are unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload, {})
    except Exception:
        return None
    if rec.get("kernel") != kernel or rec.get("csrc_hash") != csrc_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        # raw samples (the JSON line carries their summary): PA_BENCH_CLOCKS_DIR, else a temp dir
        out = os.environ.get("PA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def gpu_for_smi(dev) -> str:
    """The nvidia-smi -i selector of a torch device (its UUID when torch exposes it)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        first = vis.split(",")[dev.index or 0] if vis else str(dev.index or 0)
        return first


def algorithmic_bytes(w):
    """(attention KV+Q+O bytes, cache-write bytes) of one step.  The KV bytes
    are the distinct pool rows the step must bring from HBM: a block shared by
    several sequences (a prefix-cache hit) counts once (for every workload
    without shared blocks this equals the logical count, w.kv_bytes())."""
    return w.unique_kv_bytes() + w.qo_bytes(), w.write_bytes()


# ------------------------------------------------------------------- oracle
def time_oracle(w, budget_s: float, max_rows: int | None = None, nthreads: int = 0):
    """Run the fp64 oracle (cache write + attention rows) on a bounded sample.

    Returns (seconds, algorithmic bytes covered, rows, threads, description).
    Rows are taken in (b, h) order; each row is charged its share of its KV
    head's bytes (1/G) plus its q and o rows, so all rows add up to KV+Q+O.
    """
    import oracle
    threads = nthreads if nthreads > 0 else oracle.max_threads()
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    t0 = time.perf_counter()
    if w.slot_mapping.size:
        oracle.cache_write(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    t_write = time.perf_counter() - t0
    if w.fp8:   # e4m3 pools: whole workload per repetition
        kc8, vc8 = w.k_cache8.copy(), w.v_cache8.copy()
        oracle.cache_write_fp8(w.k_new, w.v_new, w.slot_mapping, kc8, vc8, w.k_scale, w.v_scale)
        reps, secs = 0, 0.0
        while reps == 0 or secs < budget_s:
            t0 = time.perf_counter()
            oracle.decode_fp8(w.q, kc8, vc8, w.block_tables, w.seq_lens, w.scale, w.k_scale,
                              w.v_scale, threads)
            secs += time.perf_counter() - t0
            reps += 1
        desc = f"whole workload {w.name} (e4m3 pools, widened) x {reps} reps, fp64, write excluded"
        return secs, float(w.kv_bytes() + w.qo_bytes()) * reps, reps * w.B * w.Hq, threads, desc
    if w.q_len > 1:   # multi-query: whole workload per repetition
        reps, secs = 0, 0.0
        while reps == 0 or secs < budget_s:
            t0 = time.perf_counter()
            oracle.decode_mq(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, threads)
            secs += time.perf_counter() - t0
            reps += 1
        desc = (f"whole workload {w.name} (causal, q_len {w.q_len}) x {reps} reps, fp64, "
                f"write {w.write_bytes()} B in {t_write*1e3:.1f} ms excluded")
        return secs, float(w.kv_bytes() + w.qo_bytes()) * reps, reps * w.B * w.q_len * w.Hq, threads, desc
    total = w.B * w.Hq
    rb = (np.arange(total) // w.Hq).astype(np.int32)
    rh = (np.arange(total) % w.Hq).astype(np.int32)
    row_bytes = (w.seq_lens[rb].astype(np.float64) * w.D * 2 * 2 / w.G + 2 * w.D * 2)
    # calibrate on a few rows
    n0 = min(total, max(threads, 8))
    t0 = time.perf_counter()
    oracle.decode_rows(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, rb[:n0], rh[:n0], threads)
    t_cal = max(time.perf_counter() - t0, 1e-6)
    per_row = t_cal / n0
    n = int(min(total, max(1, budget_s / per_row)))
    if max_rows is not None:
        n = min(n, max_rows)
    reps = 1
    if n == total:
        reps = max(1, int(budget_s / max(per_row * total, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.decode_rows(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, rb[:n], rh[:n],
                           threads)
    secs = time.perf_counter() - t0
    byts = float(row_bytes[:n].sum()) * reps
    desc = (f"{n} of {total} (b,h) rows x {reps} reps of workload {w.name}, fp64, "
            f"write {w.write_bytes()} B in {t_write*1e3:.1f} ms excluded")
    return secs, byts, n * reps, threads, desc


def run_reference(args, world, rank):
    """--impl reference: the oracle as it stands, timed on the host cores."""
    if rank != 0:
        return
    from paged_kv_decode_cache_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]()
    budget_per_step = max(0.005, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(w, budget_per_step)
    secs = byts = 0.0
    rows = 0
    threads = 1
    desc = ""
    for _ in range(args.steps):
        s, b, r, threads, desc = time_oracle(w, budget_per_step)
        secs += s
        byts += b
        rows += r
    value = byts / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "block_size": w.block_size, "seq_lens_total": int(w.seq_lens.sum()),
                   "q_len": w.q_len, "step": "the oracle's cache write and decode, fp64, host cores"},
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours
def run_ours(args, world, rank, local):
    import torch

    from paged_kv_decode_cache_gb300 import build as B
    from paged_kv_decode_cache_gb300 import pa
    from paged_kv_decode_cache_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    B.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.WORKLOADS[args.workload]()
    attn_bytes, write_bytes = algorithmic_bytes(w)
    step_bytes = attn_bytes + write_bytes

    def to_dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.to(dev)

    q = to_dev(w.q)
    bt = to_dev(w.block_tables)
    sl = to_dev(w.seq_lens)
    kn, vn, slots = to_dev(w.k_new), to_dev(w.v_new), to_dev(w.slot_mapping)
    fp8 = w.fp8   # e4m3 pools: write with pa_cache_write_fp8, decode with pa_decode_splitkv_fp8
    k0, v0 = (to_dev(w.k_cache8), to_dev(w.v_cache8)) if fp8 else (to_dev(w.k_cache), to_dev(w.v_cache))
    touched = w.unique_kv_bytes()   # the pool rows a step reads (shared blocks once)
    R = max(1, min(8, math.ceil(2.5 * L2_BYTES / max(touched, 1)) + 1)) if touched < 3 * L2_BYTES else 1
    pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(R - 1)]
    mq = w.q_len > 1   # multi-query step: write the q_len new tokens, then causal decode
    if mq:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        P = args.splits or pa.pa_choose_num_splits_mq(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.max_blocks,
                                                      w.block_size, sms)
    else:
        P = args.splits or pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
    oshape = (w.B, w.q_len, w.Hq, w.D) if mq else (w.B, w.Hq, w.D)
    out = torch.empty(oshape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(oshape[:-1], dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    forced = pa.pa_get_option(pa.PA_OPT_DECODE_KERNEL)
    use_tc = forced == pa.PA_KERNEL_TENSOR_CORE or (forced != pa.PA_KERNEL_CUDA_CORE and w.D == 128)
    # multi-query calls with more than 32 query columns per KV head run the prefill-shaped kernel
    kernel_name = ("prefill_tc_kernel" if use_tc and w.q_len * w.G > 32 else
                   "decode_tc_kernel" if use_tc else "decode_cc_kernel")

    cascade = w.cascade_blocks > 0   # decoded through pa_decode_cascade
    # the cascade proper (prefix once, suffixes, merge) where the library finds it pays,
    # else pa_decode_cascade runs plain split decode
    cascade_runs = cascade and pa.pa_cascade_pays(w.B, w.Hkv, w.D, w.cascade_blocks, w.block_size)
    cascade_kernels = 0   # kernel launches of the cascade proper
    if cascade_runs:
        # prefix pass, suffix pass and, unless the suffix launch merges both passes'
        # partials, the combine: the library's own count
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        cascade_kernels = pa.pa_cascade_launches(w.B, w.Hq, w.Hkv, w.D, w.cascade_blocks, w.max_blocks,
                                                 w.block_size, sms)
    ws_bytes = (pa.pa_cascade_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.cascade_blocks, w.max_blocks,
                                              w.block_size) if cascade
                else pa.pa_splitkv_workspace_bytes(w.B * w.q_len, w.Hq, w.D, P))
    ws = torch.zeros(max(1, ws_bytes), dtype=torch.uint8,
                     device=dev)
    # kernel launches of the decode call (not the cascade proper): 1 unsplit or split with
    # the merge inside the launch, 2 when a combine follows (a grid that takes waves)
    sms_count = torch.cuda.get_device_properties(dev).multi_processor_count
    decode_launches = pa.pa_decode_launches(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.max_blocks,
                                            w.block_size, P, sms_count)
    merged = P > 1 and decode_launches == 1   # the split kernel merges its own partials

    def step(r, ev0=None, ev1=None):
        kc, vc = pools[r]
        if fp8 and args.unfused:
            pa.pa_cache_write_fp8(kn, vn, slots, kc, vc, w.k_scale, w.v_scale, stream=stream)
        elif (args.unfused or mq or cascade) and not fp8:
            pa.pa_cache_write(kn, vn, slots, kc, vc, stream=stream)
        if ev0 is not None:
            ev0.record(stream)
        if cascade:
            pa.pa_decode_cascade(out, lse, q, kc, vc, w.cascade_blocks, bt, sl, w.scale, workspace=ws,
                                 stream=stream)
        elif fp8 and args.unfused:
            pa.pa_decode_splitkv_fp8(out, lse, q, kc, vc, w.k_scale, w.v_scale, bt, sl, w.scale,
                                     num_splits=P, workspace=ws, stream=stream)
        elif fp8:   # one launch: quantise and write this step's K/V, attend, merge the splits
            pa.pa_decode_step_fp8(out, lse, q, kn, vn, slots, kc, vc, w.k_scale, w.v_scale, bt, sl,
                                  w.scale, num_splits=P, workspace=ws, stream=stream)
        elif mq:
            pa.pa_decode_mq(out, lse, q, kc, vc, bt, sl, w.scale, num_splits=P, workspace=ws,
                            stream=stream)
        elif args.unfused:
            pa.pa_decode_splitkv(out, lse, q, kc, vc, bt, sl, w.scale, num_splits=P, workspace=ws,
                                 stream=stream)
        else:   # one launch: write this step's K/V, attend, merge the splits
            pa.pa_decode_step(out, lse, q, kn, vn, slots, kc, vc, bt, sl, w.scale, num_splits=P,
                              workspace=ws, stream=stream)
        if ev1 is not None:
            ev1.record(stream)

    launches_per_step = (1 + cascade_kernels if cascade_runs else
                         (1 if (args.unfused or mq or cascade) else 0) + decode_launches)
    # The timed region replays CUDA graphs that hold exactly the K timed steps
    # (consecutive steps cycle over the pool replicas): one graph when K <= 1024,
    # else K // 1024 replays of a 1024-step graph and one graph of the rest.  A
    # step that is a single launch (the fused step) is timed by the whole
    # region: its average launch duration is the region's time over the
    # launches, gaps included.  Other steps sample the decode kernel's duration
    # after the timed region, from NG graphs of S steps whose first step carries
    # a pair of events around the decode launch (event nodes cost the steps
    # around them several us of launch gaps, so they stay out of the region).
    S = R * max(1, math.ceil(16 / R))
    NG = 8
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
    except TypeError:
        mk = None
    with torch.cuda.stream(stream):
        for r in range(R):  # eager warm-up of every replica before capture
            step(r)
    stream.synchronize()

    def capture(n, events=False):
        evs = [(mk(), mk()) if (events and mk and i == 0) else (None, None) for i in range(n)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k, (e0, e1) in enumerate(evs):
                step(k % R, e0, e1)
        return g, evs

    C = min(args.steps, 1024)
    timed = [capture(C)[0]] * (args.steps // C)
    if args.steps % C:
        timed.append(capture(args.steps % C)[0])
    warm = capture(max(1, min(args.warmup, 1024)))[0]

    # Every graph of the timed region runs once first (its first replay uploads
    # it), then the W warm-up steps: the timed region holds only steady-state
    # steps whatever K and W are.
    with torch.cuda.stream(stream):
        for g in {id(g): g for g in timed}.values():
            g.replay()
        for _ in range(max(1, math.ceil(args.warmup / 1024))):
            warm.replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_for_smi(dev)) as clk:
        with torch.cuda.stream(stream):
            # the GPU idles here while the host queues the timed replays, so the
            # region measures the GPU's steps, not the host's submission latency
            torch.cuda._sleep(GPU_HEADSTART_CYCLES)
            t_start.record(stream)
            for g in timed:
                g.replay()
            t_end.record(stream)
        t_end.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    clocks = clk.summary()
    kern_ms = []
    fused_write = not (args.unfused or mq or cascade)   # pa_decode_step[_fp8] writes the new K/V
    fused = fused_write and decode_launches == 1                  # ... in the step's only launch
    if mk and not fused:
        samples = [capture(S, events=True) for _ in range(NG)]
        with torch.cuda.stream(stream):
            for g, _ in samples:
                g.replay()
            for g, _ in samples:
                g.replay()
        stream.synchronize()
        for g, evs in samples:
            kern_ms += [e0.elapsed_time(e1) for e0, e1 in evs if e0 is not None]
    kern_ms_sampled = statistics.mean(kern_ms) if kern_ms else None

    ms_per_step = elapsed_ms / args.steps
    if fused:   # one launch per step: the timed region over the launches
        kern_ms_avg, kern_method = ms_per_step, "timed region / launches (one launch per step)"
    else:
        kern_ms_avg, kern_method = kern_ms_sampled, "CUDA events around the launch, sampled steps"
    value = step_bytes * world / (ms_per_step * 1e-3) / 1e12

    # ---- end to end through the public API, host buffers, copies inside the region
    e2e_steps = args.e2e_steps or min(args.steps, 500)
    # A step's inputs (q, block tables, lengths, new K/V, slots) are staged in one
    # pinned host buffer with a device twin of the same layout, whose slices are
    # the tensors handed to the API; the result (out, lse) comes back the same
    # way: one host->device and one device->host copy per step.  As a serving
    # loop double-buffers its staging, step k uses device and host twins k % 2
    # and its copies run on their own streams: its inputs go up while step
    # k - 1 decodes, its result comes down while step k + 1 decodes.  Every
    # step's two copies are inside the timed region, which ends once the last
    # result is on the host.  Steps are replayed from CUDA graphs.
    def packed(arrays):
        offs, n = [], 0
        for a in arrays:
            offs.append(n)
            n += (a.nbytes + 255) // 256 * 256
        return offs, n
    ins = [np.ascontiguousarray(a) for a in (w.q, w.block_tables, w.seq_lens, w.k_new, w.v_new,
                                             w.slot_mapping)]
    in_offs, in_bytes = packed(ins)
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    hv = h_in.numpy()
    for a, o in zip(ins, in_offs):
        hv[o:o + a.nbytes] = a.view(np.uint8).ravel()
    def dview(buf, off, a, dtype):
        return buf[off:off + a.nbytes].view(dtype).view(a.shape)
    o_proto = np.zeros(oshape, np.uint16)
    l_proto = np.zeros(oshape[:-1], np.float32)
    out_offs, out_bytes = packed([o_proto, l_proto])
    d_ins = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_outs = [torch.zeros(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_outs = [torch.zeros(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    views = []
    for d_in, d_out in zip(d_ins, d_outs):
        views.append(dict(q=dview(d_in, in_offs[0], ins[0], torch.bfloat16),
                          bt=dview(d_in, in_offs[1], ins[1], torch.int32),
                          sl=dview(d_in, in_offs[2], ins[2], torch.int32),
                          kn=dview(d_in, in_offs[3], ins[3], torch.bfloat16),
                          vn=dview(d_in, in_offs[4], ins[4], torch.bfloat16),
                          slots=dview(d_in, in_offs[5], ins[5], torch.int64),
                          out=dview(d_out, out_offs[0], o_proto, torch.bfloat16),
                          lse=dview(d_out, out_offs[1], l_proto, torch.float32)))
    h2d, d2h = in_bytes, out_bytes
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_ready = [torch.cuda.Event() for _ in range(2)]  # inputs k up, result k - 2 down
    ev_dec = [torch.cuda.Event() for _ in range(2)]    # step k has run
    ev_out = [torch.cuda.Event() for _ in range(2)]    # result k is on the host

    def e2e_decode(v, r):
        kc, vc = pools[r]
        if cascade:
            pa.pa_cache_write(v["kn"], v["vn"], v["slots"], kc, vc, stream=stream)
            pa.pa_decode_cascade(v["out"], v["lse"], v["q"], kc, vc, w.cascade_blocks, v["bt"], v["sl"],
                                 w.scale, workspace=ws, stream=stream)
        elif fp8 and args.unfused:
            pa.pa_cache_write_fp8(v["kn"], v["vn"], v["slots"], kc, vc, w.k_scale, w.v_scale, stream=stream)
            pa.pa_decode_splitkv_fp8(v["out"], v["lse"], v["q"], kc, vc, w.k_scale, w.v_scale, v["bt"],
                                     v["sl"], w.scale, num_splits=P, workspace=ws, stream=stream)
        elif fp8:
            pa.pa_decode_step_fp8(v["out"], v["lse"], v["q"], v["kn"], v["vn"], v["slots"], kc, vc,
                                  w.k_scale, w.v_scale, v["bt"], v["sl"], w.scale, num_splits=P,
                                  workspace=ws, stream=stream)
        elif mq:
            pa.pa_cache_write(v["kn"], v["vn"], v["slots"], kc, vc, stream=stream)
            pa.pa_decode_mq(v["out"], v["lse"], v["q"], kc, vc, v["bt"], v["sl"], w.scale, num_splits=P,
                            workspace=ws, stream=stream)
        else:
            pa.pa_decode_step(v["out"], v["lse"], v["q"], v["kn"], v["vn"], v["slots"], kc, vc, v["bt"],
                              v["sl"], w.scale, num_splits=P, workspace=ws, stream=stream)

    def e2e_steps_on(n, rot0):
        """n pipelined steps issued from `stream`, forked to the two copy streams
        and joined back.  Step k's upload waits for step k - 2 (whose input
        buffer it reuses), and its "ready" event also covers the download of
        step k - 2's result (whose output buffer step k reuses), so a step
        waits on one event; uploads and downloads use separate queues."""
        fork = torch.cuda.Event()
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        for k in range(n):
            i = k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_dec[i])
                d_ins[i].copy_(h_in, non_blocking=True)          # inputs k
                if k >= 2:
                    s_in.wait_event(ev_out[i])
                ev_ready[i].record(s_in)
            stream.wait_event(ev_ready[i])
            e2e_decode(views[i], (rot0 + k) % R)
            ev_dec[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_dec[i])
                h_outs[i].copy_(d_outs[i], non_blocking=True)    # result k
                ev_out[i].record(s_out)
        for i in range(min(2, n)):
            stream.wait_event(ev_out[i])

    with torch.cuda.stream(stream):  # eager warm-up of every replica before capture
        e2e_steps_on(max(R, 2), 0)
    stream.synchronize()
    e2e_graphs = []
    for _ in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_steps_on(S, 0)
        e2e_graphs.append(g)
    n_e2e = max(1, e2e_steps // S)
    with torch.cuda.stream(stream):
        for j in range(min(4, n_e2e)):
            e2e_graphs[j % 2].replay()
    stream.synchronize()
    barrier(world)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(GPU_HEADSTART_CYCLES)
        a0.record(stream)
        for j in range(n_e2e):
            e2e_graphs[j % 2].replay()
        a1.record(stream)
    a1.synchronize()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), world) / (n_e2e * S)
    # the staged results are the library's output
    last = (S - 1) % 2
    assert np.array_equal(h_outs[last].numpy()[out_offs[0]:out_offs[0] + o_proto.nbytes],
                          d_outs[last][out_offs[0]:out_offs[0] + o_proto.nbytes].cpu().numpy())
    e2e_value = step_bytes * world / (e2e_ms * 1e-3) / 1e12

    peak, peak_kind = measured_peak_gbs()
    # the timed launch reads K, V and q, writes the bf16 output and (fused step) moves
    # this step's new K/V into the pool; its split partials and merge are overhead
    kern_bytes = attn_bytes + (write_bytes if fused_write else 0)
    roofline = None
    if kern_ms_avg:
        ach = kern_bytes / (kern_ms_avg * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(ach / peak, 4), "traffic": recorded_traffic(args.workload, kernel_name),
                    "peak_kind": peak_kind,
                    "kernel": kernel_name + ((" (cascade: prefix + suffix with merge)" if cascade_kernels == 2
                                              else " (cascade: prefix + suffix + combine)") if cascade_runs else
                                             " (shared prefix: plain split decode)" if cascade else
                                             " (fp8 pools)" if fp8 else " (multi-query)" if mq else
                                             "" if args.unfused else " (fused write)")
                              + (" + split merge" if merged else
                                 " + combine" if decode_launches == 2 and not cascade_runs else ""),
                    "kernel_us": round(kern_ms_avg * 1e3, 3), "kernel_bytes": kern_bytes,
                    "kernel_timing": kern_method,
                    "kernel_us_event_sample": (round(kern_ms_sampled * 1e3, 3)
                                               if kern_ms_sampled else None)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, byts, rows, threads, desc = time_oracle(w, args.cpu_seconds)
        cpu = {"value": byts / secs / 1e12, "unit": "TB/s", "cores": threads, "kind": "oracle",
               "sample": desc}

    configs = None
    if rank == 0 and world == 1 and args.configs != "none":
        configs = measure_configs(args, dev, peak)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "block_size": w.block_size, "seq_lens_total": int(w.seq_lens.sum()),
                       "splits": P, "q_len": w.q_len,
                       "step": (f"pa_cache_write, then pa_decode_cascade (cascade: {cascade_kernels} launches)"
                                if cascade_runs else
                                "pa_cache_write, then pa_decode_cascade (plain split decode: the "
                                "cascade does not pay)" if cascade else
                                "pa_cache_write_fp8, then pa_decode_splitkv_fp8 (e4m3 pools)"
                                if fp8 and args.unfused else
                                "pa_decode_step_fp8: quantising cache write + split decode + merge "
                                f"(e4m3 pools), {decode_launches} launch{'es' if decode_launches > 1 else ''}"
                                if fp8 else
                                "cache_write of the q_len new tokens, then pa_decode_mq (causal)"
                                if mq else "cache_write, then split decode with merge"
                                if args.unfused else
                                "pa_decode_step: cache write + split decode + merge, one launch"
                                if decode_launches == 1 else
                                "pa_decode_step: cache write + split decode (partials), then the combine"),
                       "parallelism": f"replicas x{world}",
                       "l2": f"{R} pool replicas rotated per step ({touched/1e6:.0f} MB read per step)"},
            "us_per_step": ms_per_step * 1e3,
            "pct_of_8TBps": value / 8.0 * 100,
            "step_bytes": step_bytes,
            "step_bytes_logical": w.kv_bytes() + w.qo_bytes() + write_bytes,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * launches_per_step,
            "kernel_samples": len(kern_ms),
            "clocks": clocks,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------ every config of the metric
# (config number of the metric's list, workload) for the sweep: the tiny parity
# case, the Qwen2.5-1.5B layer at B = 1 and 8, the Qwen2.5-7B layer at 16-token
# blocks and 256-token pages, the four long-context shapes, the Qwen3 batch.
CONFIG_SWEEP = [
    (1, "tiny"), (2, "qwen2.5-1.5b-B1"), (2, "qwen2.5-1.5b-B8"), (3, "qwen2.5-7b-bs16"),
    (3, "qwen2.5-7b-bs256"), (4, "long-B1-L4096"), (4, "long-B2-L4096"), (4, "long-B1-L32768"),
    (4, "long-B2-L32768"), (5, "qwen3-0.6b-B256"),
]
PER_CALL_WARMUP, PER_CALL_CALLS = 10, 50


def _pct(xs, q):
    return float(np.percentile(np.asarray(xs), q))


def measure_configs(args, dev, peak):
    """Each config of the metric on this GPU, the same fused step the headline
    times (pa_decode_step: cache write + split decode + merge, automatic split):

    - per call: 10 warm-up calls, then 50 calls each between a pair of CUDA
      events, the L2 flushed before every call by writing a buffer twice its
      size (outside the events); median, p10 and p90 in us;
    - steady state: back-to-back replays of a CUDA graph over enough pool
      replicas that each step reads its KV from HBM, timed as a region;
    - the cache write alone (pa_cache_write of the step's new tokens), per call
      as above, with its read + write bytes;
    - long-context shapes: the same per-call latency unsplit (P = 1), which
      shows what the split buys;
    - bytes: logical (every token of every sequence, K + V, plus q and out) and
      unique (a pool row shared by several sequences counted once), each with
      its fraction of the measured copy peak at the median per-call time and
      at the steady-state time;
    - the fp64 oracle on the host, 1 core and all cores, on a bounded sample.
    """
    import torch

    from paged_kv_decode_cache_gb300 import pa
    from paged_kv_decode_cache_gb300 import workloads as W
    import oracle

    def bf(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(torch.int16).view(torch.bfloat16) if a.dtype == np.uint16 else t).to(dev)

    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    all_cores = oracle.max_threads()
    out_all = {}
    with ClockSampler(gpu_for_smi(dev)) as clk:
        for cfg, name in CONFIG_SWEEP:
            w = W.WORKLOADS[name]()
            q, bt, sl = bf(w.q), bf(w.block_tables), bf(w.seq_lens)
            kn, vn, slots = bf(w.k_new), bf(w.v_new), bf(w.slot_mapping)
            k0, v0 = bf(w.k_cache), bf(w.v_cache)
            P = pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
            ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)),
                             dtype=torch.uint8, device=dev)
            out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)

            def step(kc, vc, splits=P):
                pa.pa_decode_step(out, lse, q, kn, vn, slots, kc, vc, bt, sl, w.scale,
                                  num_splits=splits, workspace=ws, stream=stream)

            def per_call(fn):
                with torch.cuda.stream(stream):
                    for _ in range(PER_CALL_WARMUP):
                        flush.fill_(1)
                        fn()
                    evs = [(torch.cuda.Event(enable_timing=True),
                            torch.cuda.Event(enable_timing=True)) for _ in range(PER_CALL_CALLS)]
                    for e0, e1 in evs:
                        flush.fill_(1)
                        e0.record(stream)
                        fn()
                        e1.record(stream)
                stream.synchronize()
                us = [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]
                return {"us_p50": round(_pct(us, 50), 3), "us_p10": round(_pct(us, 10), 3),
                        "us_p90": round(_pct(us, 90), 3)}

            lat = per_call(lambda: step(k0, v0))
            unsplit = per_call(lambda: step(k0, v0, 1)) if cfg == 4 else None
            wr = per_call(lambda: pa.pa_cache_write(kn, vn, slots, k0, v0, stream=stream))

            # steady state: one graph of S steps over R pool replicas, replayed back to back
            touched = w.unique_kv_bytes()
            R = (max(1, min(8, math.ceil(2.5 * L2_BYTES / max(touched, 1)) + 1))
                 if touched < 3 * L2_BYTES else 1)
            pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(R - 1)]
            S = R * max(1, math.ceil(16 / R))
            with torch.cuda.stream(stream):
                for kc, vc in pools:
                    step(kc, vc)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in range(S):
                    step(*pools[k % R])
            reps = max(4, int(math.ceil(2000.0 / max(1.0, lat["us_p50"] * S))))
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                torch.cuda._sleep(GPU_HEADSTART_CYCLES)
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for _ in range(reps):
                    g.replay()
                a1.record(stream)
            a1.synchronize()
            graph_us = a0.elapsed_time(a1) * 1e3 / (reps * S)

            logical = w.kv_bytes() + w.qo_bytes() + w.write_bytes()
            unique = w.unique_kv_bytes() + w.qo_bytes() + w.write_bytes()
            frac = lambda b, us: round(b / (us * 1e-6) / 1e9 / peak, 4)   # noqa: E731
            row = {"config": cfg, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "block_size": w.block_size, "seq_lens_total": int(w.seq_lens.sum()),
                   "splits": P, **lat, "calls": PER_CALL_CALLS,
                   "graph_us": round(graph_us, 3), "graph_pool_replicas": R,
                   "bytes_logical": logical, "bytes_unique": unique,
                   "frac_logical_p50": frac(logical, lat["us_p50"]),
                   "frac_unique_p50": frac(unique, lat["us_p50"]),
                   "frac_logical_graph": frac(logical, graph_us),
                   "frac_unique_graph": frac(unique, graph_us),
                   "cache_write": {**wr, "tokens": int((w.slot_mapping >= 0).sum()),
                                   "bytes_read_plus_written": w.write_bytes()}}
            if unsplit:
                row["unsplit"] = unsplit
            for cores in (1, all_cores):
                secs, byts, rows, threads, desc = time_oracle(w, args.config_oracle_seconds,
                                                              nthreads=cores)
                row[f"oracle_{'1core' if cores == 1 else 'allcores'}"] = {
                    "TBps": byts / secs / 1e12, "cores": threads, "sample": desc}
            out_all[name] = row
            del pools, k0, v0, g
            torch.cuda.empty_cache()
    return {"peak_gbs": peak, "l2_between_calls": "flushed (2x L2 written)",
            "step": "pa_decode_step (fused cache write + split decode + merge: in the launch, or by "
                    "the combine kernel after a grid that runs in waves), auto P",
            "clocks": clk.summary(), "workloads": out_all}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
