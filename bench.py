#!/usr/bin/env python
"""Benchmark: effective weight GB/s of the block-quantized mat-vec (qgemv) on GB300.

One step = the two vocabulary-sized LM heads through the fused argmax call
(qgemv_argmax) at ntok = 1, 2, 3 and 4: the Q8_0 head 248320x2560 (675.4 MB) and
the affine 4-bit g64 drafter head 248320x5120 (715.2 MB), 8 launches and 5.56 GB
of weight reads per step, logits and argmax written.  value = weight bytes / time
(scales and biases included, 1e9 B per GB).  The step is one CUDA graph (early
start between launches); the timed region is a block of exactly K steps, and
blocks are repeated until at least 1 s has been timed, so the clock record
covers a real interval.  Also reported, outside the timed region:

* config.per_config: every (head, ntok) launch alone and the 2560->12288
  projection (the largest shapes), with GB/s, the fraction of the measured copy
  peak and, for the 4-bit head, the products per second against the FMA pipe's
  128 products per clock per SM;
* per_workload: every other workload family x ntok, median of 7 graph replays (after 2
  untimed ones) of max(200, copies) launches rotating over weight copies totalling
  >= 4x L2;
* e2e: the same step through the public API with host buffers, per call
  (pinned x uploaded, logits and argmax read back, host synchronized every step);
* roofline of the dominant kernel, cpu_baseline (the fp64 oracle on the host's
  cores, one thread and all of them).

--impl reference times the CPU oracle instead (the only reference there is).
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
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "effective weight GB/s and % of GB300 HBM peak, qgemv at ntok=1..4"
HEADS = ["q8_0_head_248320x2560", "affine4_head_248320x5120"]
WORKLOAD_NAME = ("LM-head qgemv_argmax: Q8_0 248320x2560 and affine4-g64 248320x5120, "
                 "each at ntok=1,2,3,4 (8 launches, 5.56 GB of weights per step)")
LARGEST = HEADS + ["q8_0_12288x2560"]      # the shapes the >= 70% / >= 60% target is stated on
NTOKS = (1, 2, 3, 4)
PEAK_FALLBACK_GBS = 6800.0
MIN_TIMED_S = 1.0                          # timed blocks of K steps are repeated up to this
FMA_LANES_PER_CLK_SM = 128                 # products per clock per SM of the FMA pipe on GB300
                                           # (fma.rn.f32x2 or dp2a: 64 lane-instructions x 2)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-detail", action="store_true", help="skip the per-workload table")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    p.add_argument("--detail-only", default="", help="comma list of workload names for the table")
    p.add_argument("--one-experts", default="", help="ntok: five routed-expert layers on a 64-expert stack "
                   "(the small case an ncu capture profiles)")
    p.add_argument("--one-layer", default="", help="ntok: as --one-experts, with the layer as one launch")
    p.add_argument("--one", default="", help="fmt,n_out,n_in,ntok[,tile spec]: run one shape 3 times "
                                             "(a small case for ncu) and exit")
    p.add_argument("--one-argmax", default="", help="as --one, through qgemv_argmax (the LM-head call)")
    p.add_argument("--profile-step", type=int, default=0, help="run the headline step (8 launches) this many "
                   "times after one warm-up step, eagerly with early start, and exit (for ncu launch lists)")
    p.add_argument("--sweep", default="", help="comma list of workload names: time every tile spec of "
                   "--sweep-specs (';'-separated, qg_set_tile_override grammar; default a grid) at "
                   "--sweep-ntoks, one JSON line per point to --sweep-out, the best per (workload, ntok) "
                   "to stdout")
    p.add_argument("--sweep-specs", default="")
    p.add_argument("--sweep-ntoks", default="1,2,3,4")
    p.add_argument("--sweep-out", default="tile_sweep.jsonl")
    p.add_argument("--sweep-experts", default="", help="';'-separated tile specs: time the routed-expert "
                   "layer (plan + gate/up + down) under each, one JSON line per spec")
    p.add_argument("--phases", default="", help="comma list of workload names: per-CTA phase timestamps "
                   "(qg_set_phase_record) of 20 back-to-back launches in a graph, with and without early "
                   "start, at --sweep-ntoks; one JSON line per (workload, ntok, launch mode)")
    p.add_argument("--cpu-worker", default="", help=argparse.SUPPRESS)
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


KERNEL_FILES = ("qgemv_kernels.cuh", "qgemv_inst.cu", "qg_layout.h", "qgemv_api.cu")


def csrc_hash() -> str:
    """Hash of the kernel sources: a stored ncu traffic figure is used only while it matches."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_quantized_token_format_gb300", "csrc")
    for name in KERNEL_FILES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (all-reduce MAX); every rank gets the same value."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every replica streams step_bytes per step; the job
    takes the slowest rank's time."""
    return step_bytes * steps * world / (max_ms * 1e-3) / 1e9


def timed_blocks(block_s_estimate: float, min_total_s: float = MIN_TIMED_S, min_blocks: int = 3) -> int:
    """How many blocks of K steps to time so that at least min_total_s is timed."""
    if block_s_estimate <= 0:
        return min_blocks
    return max(min_blocks, int(math.ceil(min_total_s / block_s_estimate)))


def algo_bytes(fmt, n_out, n_in, ntok, argmax=False):
    b = workloads_bytes(fmt, n_out, n_in) + 4 * ntok * (n_in + n_out)
    return b + (4 * ntok if argmax else 0)


def workloads_bytes(fmt, n_out, n_in):
    n = n_out * n_in
    return {"q8_0": n // 32 * 34, "q4_0": n // 32 * 18, "affine4_g64": n // 2 + n // 64 * 4, "bf16": 2 * n,
            "q5_0": n // 32 * 22}[fmt]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if t0 - 0.05 <= ts <= t1 + 0.15:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def gen_packed(qg, w: workloads.Workload, threads: int = 16) -> np.ndarray:
    """Device-layout bytes of a whole workload matrix, generated 4096 rows at a time."""
    stride = qg.qg_row_stride(w.fmt, w.n_in)
    out = np.empty(w.n_out * stride, dtype=np.uint8)
    n_chunks = (w.n_out + workloads.ROW_CHUNK - 1) // workloads.ROW_CHUNK

    def one(c):
        Wc = workloads.weight_chunk(w.seed, w.n_out, w.n_in, c)
        r0 = c * workloads.ROW_CHUNK
        qg.qg_pack(w.fmt, Wc, out=out[r0 * stride:(r0 + Wc.shape[0]) * stride])

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(n_chunks)))
    return out


def time_graph(torch, call, n, reps=5, warm=2):
    """Median per-call microseconds of a graph of n calls (call(i), i < n), over reps replays
    after `warm` untimed ones (a replay right after an idle host gap runs 5-10% slower)."""
    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        for i in range(n):
            call(i)
    for _ in range(max(1, warm)):
        g.replay()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / n * 1e3)
    del g
    return statistics.median(times)


# ----------------------------------------------------------------------------- CPU oracle legs

def cpu_worker(spec: str):
    """Run inside a fresh process with BLAS pinned to one thread: time the oracle on a
    slice of each workload's rows (the slice starts at row0_frac of the rows)."""
    import oracle
    cfg = json.loads(spec)
    names, steps, warm, frac = cfg["names"], cfg["steps"], cfg["warmup"], cfg["row_frac"]
    r0f = cfg.get("row0_frac", 0.0)
    data = []
    for name in names:
        w = workloads.WORKLOADS[name]
        rows = max(64, int(math.ceil(w.n_out * frac)))
        r0 = min(int(w.n_out * r0f), w.n_out - rows)
        W = workloads.weight_rows(w.seed, w.n_out, w.n_in, np.arange(r0, r0 + rows))
        data.append((w, rows, oracle.quantize(w.fmt, W), workloads.activations(w.seed, w.n_in, 4)))
    per_step_bytes = sum(workloads_bytes(w.fmt, rows, w.n_in) for w, rows, _, _ in data) * len(NTOKS)

    def step():
        for ntok in NTOKS:
            for w, rows, canon, x in data:
                if w.argmax:
                    oracle.qgemv_argmax(w.fmt, canon, rows, w.n_in, x[:ntok])
                else:
                    oracle.gemv(w.fmt, canon, rows, w.n_in, x[:ntok])

    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "steps": steps, "bytes_per_step": per_step_bytes,
                      "rows": {w.name: rows for w, rows, _, _ in data}}))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_oracle(names, steps, warmup, row_frac, procs=1):
    """The oracle in `procs` concurrent worker processes (one BLAS thread each, disjoint
    row slices of row_frac of the rows).  Returns the bytes all workers processed per
    step, the slowest worker's seconds and the workers' row counts."""
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    ps = []
    for p in range(procs):
        spec = json.dumps({"names": names, "steps": steps, "warmup": warmup, "row_frac": row_frac,
                           "row0_frac": p * row_frac})
        ps.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-worker", spec],
                                   stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    outs = []
    for pr in ps:
        so, se = pr.communicate(timeout=1800)
        if pr.returncode != 0:
            raise RuntimeError(se[-2000:])
        outs.append(json.loads(so.strip().splitlines()[-1]))
    return {"bytes_per_step": sum(o["bytes_per_step"] for o in outs), "seconds": max(o["seconds"] for o in outs),
            "steps": steps, "rows": outs[0]["rows"], "procs": procs}


def cpu_baseline_entry(names, row_frac, steps):
    """cpu_baseline: the oracle on one thread and on every host core (one worker process
    per core, each on its own slice of the rows)."""
    cores = host_cores()
    one = run_cpu_oracle(names, steps=steps, warmup=0, row_frac=row_frac, procs=1)
    allc = run_cpu_oracle(names, steps=steps, warmup=0, row_frac=row_frac / cores, procs=cores)
    v1 = one["bytes_per_step"] * one["steps"] / one["seconds"] / 1e9
    va = allc["bytes_per_step"] * allc["steps"] / allc["seconds"] / 1e9
    return {"value": round(va, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": (f"{steps} passes over a {row_frac:.2%} row slice of each head at ntok 1..4 "
                       f"(qgemv_argmax in numpy fp64); all cores: {cores} worker processes on disjoint "
                       f"slices of it, one BLAS thread each"),
            "one_thread": {"value": round(v1, 4), "cores": 1, "seconds": round(one["seconds"], 3),
                           "rows": one["rows"]},
            "all_cores": {"value": round(va, 4), "cores": cores, "seconds": round(allc["seconds"], 3)}}


# ----------------------------------------------------------------------------- GPU legs

def main_gpu(args, rank, world, local_rank):
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    sms = int(props.multi_processor_count)
    peak, peak_kind = peaks()
    stream = torch.cuda.current_stream()

    heads = [workloads.WORKLOADS[n] for n in HEADS]
    W = {w.name: torch.from_numpy(gen_packed(qg, w)).to(dev) for w in heads}
    X = {w.name: torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev) for w in heads}
    Y = {w.name: torch.empty((4, w.n_out), dtype=torch.float32, device=dev) for w in heads}
    AM = torch.full((len(NTOKS), len(heads), 4), -7, dtype=torch.int32, device=dev)
    WS = {w.name: torch.zeros(qg.qgemv_argmax_workspace_bytes(w.n_out, 4), dtype=torch.uint8, device=dev)
          for w in heads}
    launches_per_step = len(NTOKS) * len(heads)
    step_bytes = sum(workloads_bytes(w.fmt, w.n_out, w.n_in) for w in heads) * len(NTOKS)
    step_algo = sum(algo_bytes(w.fmt, w.n_out, w.n_in, t, True) for w in heads for t in NTOKS)

    def call(w, ntok, stream_handle=None):
        qg.qgemv_argmax(w.fmt, W[w.name], w.n_out, w.n_in, X[w.name], Y[w.name][:ntok],
                        AM[ntok - 1, HEADS.index(w.name)], WS[w.name], ntok, stream=stream_handle)

    def launches():
        for ntok in NTOKS:
            for w in heads:
                call(w, ntok)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def capture(early: bool):
        qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START if early else 0)
        launches()                                 # every kernel and plan warmed before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            launches()
        torch.cuda.synchronize()
        return g

    def run_block(g, K):
        """Exactly K steps between a barrier + synchronize on both sides; CUDA-event ms."""
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(K):
            g.replay()
        end.record()
        torch.cuda.synchronize()
        barrier()
        return start.elapsed_time(end)

    K, Wm = max(1, args.steps), max(3, args.warmup)
    # Secondary: ordinary launches (each kernel waits for the previous one to finish).
    g_plain = capture(False)
    for _ in range(Wm):
        g_plain.replay()
    plain_ms = run_block(g_plain, K)
    plain_value = step_bytes * K / (plain_ms * 1e-3) / 1e9
    del g_plain
    # Headline: early start (programmatic dependent launch): the weights are written
    # once before the run, so a call may stream them while the previous call finishes.
    g = capture(True)
    t_w = time.perf_counter()
    for _ in range(Wm):
        g.replay()
    torch.cuda.synchronize()
    est_step_s = (time.perf_counter() - t_w) / Wm
    blocks = timed_blocks(K * est_step_s)
    if world > 1:
        blocks = int(max_over_ranks(float(blocks), world, dev))
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (str(uuid) if uuid else str(local_rank))
    block_ms = []
    with ClockSampler(gpu_id) as clk:
        t_wall0 = time.time()
        for _ in range(blocks):
            block_ms.append(run_block(g, K))
        t_wall1 = time.time()
    clocks = clk.summary(t_wall0, t_wall1)
    total_ms = max_over_ranks(sum(block_ms), world, dev)
    steps_timed = K * blocks
    ms_per_step = total_ms / steps_timed
    value = job_gbs(step_bytes, steps_timed, world, total_ms)
    sm_mhz = clocks.get("sm_mhz") or 2070.0

    # --- per-config table: each (head, ntok) launch alone, and the 2560->12288 projection
    per_config = {}
    for w in heads:
        row = {}
        for ntok in NTOKS:
            us = time_graph(torch, lambda i, w=w, ntok=ntok: call(w, ntok), n=20)
            gbs = workloads_bytes(w.fmt, w.n_out, w.n_in) / (us * 1e-6) / 1e9
            fma_rate = ntok * w.n_out * w.n_in / (us * 1e-6)
            fma_peak = FMA_LANES_PER_CLK_SM * sms * sm_mhz * 1e6
            row[str(ntok)] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "frac_nominal_7900": round(gbs / 7900.0, 4),
                              "fma_frac": round(fma_rate / fma_peak, 4)}
        per_config[w.name] = row
    proj = workloads.WORKLOADS["q8_0_12288x2560"]
    pbase = torch.from_numpy(gen_packed(qg, proj)).to(dev)
    copies = max(1, math.ceil(4 * l2 / pbase.numel()))
    pool = [pbase] + [pbase.clone() for _ in range(copies - 1)]
    px = torch.from_numpy(workloads.activations(proj.seed, proj.n_in, 4)).to(dev)
    py = torch.empty((4, proj.n_out), dtype=torch.float32, device=dev)
    row = {}
    for ntok in NTOKS:
        us = time_graph(torch, lambda i, ntok=ntok: qg.qgemv(proj.fmt, pool[i % copies], proj.n_out, proj.n_in,
                                                             px, py[:ntok], ntok), n=200, reps=7)
        gbs = workloads_bytes(proj.fmt, proj.n_out, proj.n_in) / (us * 1e-6) / 1e9
        row[str(ntok)] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                          "frac_nominal_7900": round(gbs / 7900.0, 4)}
    per_config[proj.name] = row
    del pool, pbase

    # --- roofline of the dominant kernel: every launch of the step is qgemv_kernel
    # (100% of the step's GPU time); its average launch duration is the step time
    # over the 8 launches (consecutive launches overlap slightly under early start).
    achieved = step_algo * steps_timed / (total_ms * 1e-3) / 1e9 / world
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            td = json.load(f)
        if td.get("csrc_hash") == csrc_hash():
            traffic = td.get("traffic_bytes_per_launch")
    aff = per_config["affine4_head_248320x5120"]
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": "qgemv_kernel (all 8 launches of the step: 2 heads x ntok 1..4)",
                "algorithmic_bytes_per_launch": round(step_algo / launches_per_step),
                "avg_launch_us": round(ms_per_step / launches_per_step * 1e3, 3), "peak_kind": peak_kind,
                "secondary": {"bound": "FMA pipe products (dp2a / fma.rn.f32x2, 128 per clock per SM), "
                                       "4-bit head at ntok 3-4",
                              "peak_fma_per_s": FMA_LANES_PER_CLK_SM * sms * sm_mhz * 1e6,
                              "fma_frac": {t: aff[t]["fma_frac"] for t in ("3", "4")}}}

    result = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
              "warmup": Wm, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
              "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
              "config": {"workload": WORKLOAD_NAME,
                         "formats": "Q8_0 and affine 4-bit g64 weights, fp32 x, logits and accumulation, "
                                    "int32 argmax",
                         "weight_bytes_per_step": step_bytes, "launches_per_step": launches_per_step,
                         "l2": f"inputs larger than L2: every launch reads a {675.4:.0f}-{715.2:.0f} MB head "
                               f"(L2 {l2 / 1e6:.0f} MB)",
                         "timing": f"{blocks} timed blocks of exactly {K} steps (CUDA graph of one step replayed), "
                                   f"each between a barrier and a synchronize, CUDA events on the launch stream; "
                                   f"{steps_timed} steps, {total_ms / 1e3:.2f} s timed",
                         "timed_blocks": blocks, "block_ms": [round(b, 3) for b in block_ms],
                         "launch": "early start (programmatic dependent launch, QG_LAUNCH_EARLY_START)",
                         "value_plain_launches": round(plain_value, 2),
                         "per_config": per_config,
                         "parallelism": "replicas" if world > 1 else "single GPU"},
              "frac_of_peak": round(value / world / peak, 4), "peak_gbs": peak, "peak_kind": peak_kind,
              "frac_of_nominal_7900": round(value / world / 7900.0, 4),
              "clocks": clocks, "gpu_launches": launches_per_step * steps_timed, "roofline": roofline}

    # --- e2e through the public API with host buffers (no graph), rank-local.  A
    # step uploads both heads' x in one copy from pinned memory, makes the 8 calls and
    # reads every call's logits and the argmax ids back to pinned memory, then waits for
    # them.  Each call's logits leave on a copy stream as soon as that call ends, so the
    # read-back overlaps the later calls; the calls run ntok 4 down to 1, leaving the
    # smallest logits (ntok 1) for the one copy that cannot overlap.  The same step with
    # every copy after the last call is reported beside it.
    if not args.no_e2e:
        xs_elems = [4 * w.n_in for w in heads]
        pin_x = torch.empty(sum(xs_elems), dtype=torch.float32).pin_memory()
        dx = torch.empty(pin_x.numel(), dtype=torch.float32, device=dev)
        off, xv = 0, {}
        for w, n in zip(heads, xs_elems):
            pin_x[off:off + n].copy_(torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).reshape(-1))
            xv[w.name] = dx[off:off + n].view(4, w.n_in)
            off += n
        order = [(ntok, w) for ntok in sorted(NTOKS, reverse=True) for w in heads]
        y_all = torch.empty(sum(t * w.n_out for t, w in order), dtype=torch.float32, device=dev)
        pin_y = torch.empty(y_all.numel(), dtype=torch.float32).pin_memory()
        pin_am = torch.empty(AM.numel(), dtype=torch.int32).pin_memory()
        ysl, off = [], 0
        for ntok, w in order:
            ysl.append(slice(off, off + ntok * w.n_out))
            off += ntok * w.n_out
        sh = qg.current_stream_handle()
        copy_stream = torch.cuda.Stream(device=dev)
        done = [torch.cuda.Event() for _ in order]

        # Each call's device addresses, workspace size and stream as plain ints, computed
        # once (the binding takes addresses as well as tensors), so the host's per-call
        # cost is the ctypes call itself.
        call_args = []
        for i, (ntok, w) in enumerate(order):
            am = AM[ntok - 1, HEADS.index(w.name)]
            call_args.append((w.fmt, W[w.name].data_ptr(), w.n_out, w.n_in, xv[w.name].data_ptr(),
                              y_all[ysl[i]].data_ptr(), am.data_ptr(), WS[w.name].data_ptr(),
                              WS[w.name].numel(), ntok))

        def run_call(i):
            fmt, wp, n_out, n_in, xp, yp, ap, wsp, wsb, ntok = call_args[i]
            qg.qgemv_argmax(fmt, wp, n_out, n_in, xp, yp, ap, wsp, ntok, workspace_bytes=wsb, stream=sh)

        def e2e_step():
            dx.copy_(pin_x, non_blocking=True)
            for i in range(len(order)):
                run_call(i)
                done[i].record(stream)
                copy_stream.wait_event(done[i])
                with torch.cuda.stream(copy_stream):
                    pin_y[ysl[i]].copy_(y_all[ysl[i]], non_blocking=True)
            with torch.cuda.stream(copy_stream):
                pin_am.copy_(AM.view(-1), non_blocking=True)
            copy_stream.synchronize()

        def e2e_step_serial():
            dx.copy_(pin_x, non_blocking=True)
            for i in range(len(order)):
                run_call(i)
            pin_y.copy_(y_all, non_blocking=True)
            pin_am.copy_(AM.view(-1), non_blocking=True)
            stream.synchronize()

        n_e2e = max(20, min(400, int(1.0 / max(est_step_s, 1e-4))))

        def e2e_gbs(step_fn):
            for _ in range(3):
                step_fn()
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                step_fn()
            return round(step_bytes * n_e2e / (time.perf_counter() - t0) / 1e9, 2)

        e2e_value = e2e_gbs(e2e_step)
        result["e2e"] = {"value": e2e_value, "unit": "GB/s",
                         "h2d_bytes_per_step": pin_x.numel() * 4,
                         "d2h_bytes_per_step": pin_y.numel() * 4 + pin_am.numel() * 4, "steps": n_e2e,
                         "serial_readback_value": e2e_gbs(e2e_step_serial),
                         "how": "python qgemv_argmax calls (ctypes, device addresses as ints), x of both heads "
                                "uploaded in one copy from "
                                "pinned memory, every call's logits read back to pinned memory on a copy stream "
                                "as soon as the call ends, argmax ids after the last call, host synchronized "
                                "every step; no CUDA graph; early start on (serial_readback_value: all copies "
                                "after the last call)"}

    if rank == 0 and not args.no_detail:
        result["per_workload"] = detail_table(args, qg, torch, dev, l2, peak, have=W)

    if rank == 0 and not args.no_cpu:
        try:
            result["cpu_baseline"] = cpu_baseline_entry(HEADS, row_frac=1.0 / 16, steps=6)
        except Exception as e:  # noqa: BLE001
            result["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
                                      "sample": f"failed: {e}"}
    return result


def detail_table(args, qg, torch, dev, l2, peak, have=None):
    """Every workload x ntok except the headline heads (timed in config.per_config): median of
    7 replays of a graph of max(200, copies) launches over rotating copies (after 2 untimed
    replays).  `have`: packed matrices already on
    the device, by workload name (the drafted-vocabulary variants reuse the full Q8_0 head)."""
    if args.detail_only:
        names = args.detail_only.split(",")
    else:
        names = [n for n in workloads.WORKLOADS if n not in HEADS]
    expert_names = [n for n in names if n in workloads.EXPERT_LAYERS]
    names = [n for n in names if n not in workloads.EXPERT_LAYERS]
    table = {}
    cache = {}
    have = have or {}
    for name in names:
        w = workloads.WORKLOADS[name]
        src = name
        if name == "q8_0_head_106299x2560":
            src = "q8_0_head_248320x2560"
        if src in have:
            base = have[src]
        else:
            if src not in cache:
                ws = workloads.WORKLOADS[src]
                cache.clear()
                torch.cuda.empty_cache()
                cache[src] = torch.from_numpy(gen_packed(qg, ws)).to(dev)
            base = cache[src]
        wbytes = workloads_bytes(w.fmt, w.n_out, w.n_in)
        copies = max(1, math.ceil(4 * l2 / base.numel()))
        pool = [base] + [base.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev)
        y = torch.empty((4, w.n_out), dtype=torch.float32, device=dev)
        am = torch.empty(4, dtype=torch.int32, device=dev)
        wsp = torch.zeros(qg.qgemv_argmax_workspace_bytes(w.n_out, 4), dtype=torch.uint8, device=dev)
        row = {}
        for ntok in NTOKS:
            def call(i):
                if w.argmax:
                    qg.qgemv_argmax(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y, am, wsp, ntok)
                else:
                    qg.qgemv(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y, ntok)
            for i in range(copies + 2):        # every copy touched once before the capture
                call(i)
            us = time_graph(torch, call, n=max(200, copies), reps=7)
            gbs = wbytes / (us * 1e-6) / 1e9
            row[str(ntok)] = {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "tile": qg.qg_describe_tile(w.fmt, w.n_out, w.n_in, ntok)}
        table[name] = {"fmt": w.fmt, "n_out": w.n_out, "n_in": w.n_in, "weight_bytes": wbytes,
                       "call": "qgemv_argmax" if w.argmax else "qgemv", "copies": copies, "ntok": row}
        del pool

    for name in [n for n in workloads.DRAFT_IDS if (n in names or (n in HEADS and not args.detail_only))]:
        w = workloads.WORKLOADS[name]
        base = have[name] if name in have else torch.from_numpy(gen_packed(qg, w)).to(dev)
        table[f"{w.fmt}_draft_ids_{workloads.DRAFT_IDS[name][0]}_of_{w.n_out}x{w.n_in}"] = \
            draft_ids_detail(qg, torch, dev, l2, peak, w, base)
        del base
    cache.clear()
    torch.cuda.empty_cache()
    if not args.detail_only or expert_names:
        for name in (expert_names or workloads.EXPERT_LAYERS):
            table[name] = experts_detail(qg, torch, dev, peak, workloads.EXPERT_LAYERS[name])
            torch.cuda.empty_cache()
    return table


def experts_detail(qg, torch, dev, peak, layer, unique=32, routings=64):
    """Routed experts, one layer: the plan, the gate/up projection (token rows, gate / up
    row pairs written as silu(gate) * up; it also prefetches the same experts' down rows
    into L2) and the down projection of that activation (one row per slot) per
    ntok, each step with its own seeded routing (64 routings in turn), timed as
    64-step graphs; "layer_one_launch" is the same layer as one persistent launch.  Bytes = the active experts' weight
    bytes (each read from HBM once per layer).  The stack holds n_experts experts at
    their own addresses; their contents repeat every `unique` experts (the data does
    not change the timing; the addresses do).  "gate_up" and "down" are timed alone
    ("down" alone reads HBM; in "layer" it reads what gate/up prefetched)."""
    E, dm, ff = layer.n_experts, layer.d_model, layer.d_ff
    shapes = {"gu": (2 * ff, dm, layer.seed), "dn": (dm, ff, layer.seed + 1)}
    stacks = {}
    for key, (n_out, n_in, seed) in shapes.items():
        stride = qg.qg_row_stride(layer.fmt, n_in)
        host = np.empty(unique * n_out * stride, dtype=np.uint8)

        def one(k, n_out=n_out, n_in=n_in, seed=seed, stride=stride, host=host):
            qg.qg_pack(layer.fmt, workloads.expert_matrix(seed, k, n_out, n_in),
                       out=host[k * n_out * stride:(k + 1) * n_out * stride])

        with ThreadPoolExecutor(16) as ex:
            list(ex.map(one, range(unique)))
        stacks[key] = torch.from_numpy(host).to(dev).repeat(E // unique)
    bytes_e = {k: workloads_bytes(layer.fmt, n_out, n_in) for k, (n_out, n_in, _) in shapes.items()}
    out = {"fmt": layer.fmt, "n_experts": E, "gate_up": f"{2 * ff}x{dm} per expert", "down": f"{dm}x{ff} per expert",
           "topk": layer.topk, "share": layer.share, "routings": routings,
           "bytes_per_expert": bytes_e["gu"] + bytes_e["dn"],
           "tile": {k: qg.qg_describe_expert_tile(layer.fmt, n_out, n_in) for k, (n_out, n_in, _) in shapes.items()},
           "ntok": {}}
    for ntok in NTOKS:
        G = ntok * layer.topk
        ids_np = [workloads.routing(layer.seed * 100 + 17 * ntok + r, ntok, layer.topk, E, layer.share)
                  for r in range(routings)]
        unique_e = float(np.mean([len(np.unique(i)) for i in ids_np]))
        ids = [torch.from_numpy(i).to(dev) for i in ids_np]
        plans = [torch.empty(qg.qg_expert_plan_ints(G), dtype=torch.int32, device=dev) for _ in range(routings)]
        x = torch.from_numpy(workloads.activations(layer.seed, dm, ntok)).to(dev)
        act = torch.zeros((G, ff), dtype=torch.float32, device=dev)
        y_dn = torch.empty((G, dm), dtype=torch.float32, device=dev)

        def plan(r):
            qg.qg_expert_plan(ids[r], E, plans[r])

        def gu(r):   # gate/up pairs -> silu(gate) * up; also prefetches the down rows into L2
            qg.qgemv_experts(layer.fmt, stacks["gu"], E, 2 * ff, dm, x, plans[r], G, act, swiglu=True,
                             W_next=stacks["dn"], next_n_out=dm, next_n_in=ff)

        def dn(r):   # reads the activation; the plan was written two launches back
            qg.qgemv_experts(layer.fmt, stacks["dn"], E, dm, ff, act, plans[r], G, y_dn, x_by_slot=True,
                             plan_ready=True)

        def layer_step(r):
            plan(r)
            gu(r)
            dn(r)

        wsl = torch.zeros(qg.qgemv_expert_layer_workspace_bytes(), dtype=torch.uint8, device=dev)

        def layer_one(r):   # the same layer as one persistent launch
            qg.qgemv_expert_layer(layer.fmt, stacks["gu"], stacks["dn"], E, dm, ff, x, ids[r], plans[r], act, y_dn,
                                  wsl)

        for r in range(routings):
            plan(r)
        torch.cuda.synchronize()
        row = {"pairs": G, "unique_experts": round(unique_e, 2),
               "grouping_saves": round(1.0 - unique_e / G, 3)}
        for key, fn in (("plan", plan), ("gate_up", gu), ("down", dn), ("layer", layer_step),
                        ("layer_one_launch", layer_one)):
            for r in range(3):
                fn(r)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                for r in range(routings):
                    fn(r)
            g.replay()
            ts = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) / routings * 1e3)
            us = statistics.median(ts)
            nbytes = unique_e * {"plan": 0, "gate_up": bytes_e["gu"], "down": bytes_e["dn"],
                                 "layer": bytes_e["gu"] + bytes_e["dn"],
                                 "layer_one_launch": bytes_e["gu"] + bytes_e["dn"]}[key]
            row[key] = {"us": round(us, 3)}
            if nbytes:
                gbs = nbytes / (us * 1e-6) / 1e9
                row[key].update({"gbs": round(gbs, 1), "frac": round(gbs / peak, 4)})
            del g
        out["ntok"][str(ntok)] = row
    del stacks
    return out


def draft_ids_detail(qg, torch, dev, l2, peak, w, head):
    """The id-list draft head: gather the listed rows once (timed: bytes read + written),
    then qgemv_argmax_ids on the small head per ntok (timed like every other workload)."""
    k, seed = workloads.DRAFT_IDS[w.name]
    ids = torch.from_numpy(workloads.draft_ids(seed, w.n_out, k)).to(dev)
    small = torch.empty(qg.qg_packed_bytes(w.fmt, k, w.n_in), dtype=torch.uint8, device=dev)
    qg.qg_gather_rows(w.fmt, head, w.n_out, w.n_in, ids, small)
    torch.cuda.synchronize()
    times = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        qg.qg_gather_rows(w.fmt, head, w.n_out, w.n_in, ids, small)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    g_us = statistics.median(times)
    moved = 2 * small.numel()
    wbytes = workloads_bytes(w.fmt, k, w.n_in)
    copies = max(1, math.ceil(4 * l2 / small.numel()))
    pool = [small] + [small.clone() for _ in range(copies - 1)]
    x = torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev)
    y = torch.empty((4, k), dtype=torch.float32, device=dev)
    am = torch.empty(4, dtype=torch.int32, device=dev)
    wsp = torch.zeros(qg.qgemv_argmax_workspace_bytes(k, 4), dtype=torch.uint8, device=dev)
    row = {}
    for ntok in NTOKS:
        n = 50
        for i in range(copies + 2):
            qg.qgemv_argmax_ids(w.fmt, pool[i % copies], k, w.n_in, x, y, am, ids, wsp, ntok)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, capture_error_mode="thread_local"):
            for i in range(n):
                qg.qgemv_argmax_ids(w.fmt, pool[i % copies], k, w.n_in, x, y, am, ids, wsp, ntok)
        gr.replay()
        ts = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gr.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / n * 1e3)
        us = statistics.median(ts)
        gbs = wbytes / (us * 1e-6) / 1e9
        row[str(ntok)] = {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                          "tile": qg.qg_describe_tile(w.fmt, k, w.n_in, ntok)}
        del gr
    return {"fmt": w.fmt, "n_out": k, "n_in": w.n_in, "weight_bytes": wbytes, "call": "qgemv_argmax_ids",
            "ids": f"{k} ids of the {w.n_out}-row head (seeded, sorted)", "copies": copies,
            "gather": {"us": round(g_us, 1), "bytes_moved": moved, "gbs": round(moved / (g_us * 1e-6) / 1e9, 1),
                       "frac": round(moved / (g_us * 1e-6) / 1e9 / peak, 4)},
            "ntok": row}


# ----------------------------------------------------------------------------- reference arm

def reference_arm(args, rank, world):
    """The oracle as it stands on the host's cores (one worker process per core, one BLAS
    thread each, disjoint row slices), on the headline workload; each step is a bounded
    row sample of it, sized so the run ends within a few minutes."""
    if rank != 0:
        return None
    K, Wm = max(1, args.steps), max(3, args.warmup)
    cores = host_cores()
    # One step over every row of both heads takes ~60-80 s of oracle work on one core;
    # sample rows so that K + Wm steps take about two minutes on all cores.
    est_full_step_core_s = 60.0
    frac = min(1.0, 120.0 * cores / ((K + Wm) * est_full_step_core_s))
    r = run_cpu_oracle(HEADS, steps=K, warmup=Wm, row_frac=frac / cores, procs=cores)
    value = r["bytes_per_step"] * r["steps"] / r["seconds"] / 1e9
    sample = (f"each step: the oracle (qgemv_argmax, numpy fp64) on {frac:.3%} of each head's rows at ntok "
              f"1..4, split over {cores} worker processes (one per host core, one BLAS thread each)")
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": round(r["seconds"] / K * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD_NAME, "rows_sampled_per_worker": r["rows"], "workers": cores},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def tile_sweep(args):
    """GB/s per (workload, ntok, tile spec): each point is the median of 3 replays (after 2
    untimed ones) of a graph of at least 100 launches rotating over weight copies
    totalling >= 4x L2 (set
    QGEMV_EARLY_START=1 to sweep with early-start launches).  The table in
    csrc/tile_select.cpp was filled from such sweeps."""
    import itertools
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    specs = args.sweep_specs.split(";") if args.sweep_specs else [
        f"rpw={r},depth={d},warps={w},ctas={c}"
        for r, d, w, c in itertools.product((1, 2, 4), (2, 3, 5, 8), (4, 8, 12, 16), (1, 2, 3))]
    ntoks = [int(v) for v in args.sweep_ntoks.split(",")]
    dev = torch.device("cuda:0")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = open(args.sweep_out, "a")
    for name in args.sweep.split(","):
        w = workloads.WORKLOADS[name]
        base = torch.from_numpy(gen_packed(qg, w)).to(dev)
        copies = max(1, math.ceil(4 * l2 / base.numel()))
        pool = [base] + [base.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev)
        y = torch.empty((4, w.n_out), dtype=torch.float32, device=dev)
        am = torch.empty(4, dtype=torch.int32, device=dev)
        ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(w.n_out, 4), dtype=torch.uint8, device=dev)
        wb = workloads_bytes(w.fmt, w.n_out, w.n_in)
        for ntok in ntoks:
            best = None
            for spec in specs:
                try:
                    qg.qg_set_tile_override(spec)
                    desc = qg.qg_describe_tile(w.fmt, w.n_out, w.n_in, ntok)
                except qg.QGError:
                    continue

                def call(i, ntok=ntok):
                    if w.argmax:
                        qg.qgemv_argmax(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y[:ntok], am, ws, ntok)
                    else:
                        qg.qgemv(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y[:ntok], ntok)
                us = time_graph(torch, call, n=max(100, copies), reps=3)
                rec = {"name": name, "ntok": ntok, "spec": spec, "desc": desc, "us": round(us, 3),
                       "gbs": round(wb / us / 1e3, 1)}
                out.write(json.dumps(rec) + "\n")
                out.flush()
                if best is None or rec["gbs"] > best["gbs"]:
                    best = rec
            print(json.dumps({"best": best}), flush=True)
        del pool, base
        torch.cuda.empty_cache()
    qg.qg_set_tile_override(None)


PHASE_KEYS = ["copies_issued", "wait_done", "x_staged", "first_stage", "warp0_done", "cta_done"] + \
    [f"stage{k}_landed" for k in range(7)]


def summarize_phases(rec) -> dict:
    """Summary of the phase stamps of n launches x grid CTAs (rec: int64 [n, grid, 16], the
    qg_set_phase_record layout: [0] entry and [1] exit globaltimer ns, [2] SM id, [6] the
    entry SM clock, [3..5, 7..15] the SM clock at each phase, 32 bits, 0 = not reached).
    Global times are taken relative to the first entry in integers (as float64, raw
    globaltimer values would keep only ~256 ns).  Per CTA the SM clock rate is its cycles
    from entry to its end over its global duration; phases are converted with it.  Medians
    over launches of per-launch medians (and of per-launch maxima for *_max)."""
    med = statistics.median
    rec = np.asarray(rec, dtype=np.int64)
    n = rec.shape[0]
    base = int(rec[:, :, 0].min())
    t_in = (rec[:, :, 0] - base).astype(np.float64)
    t_out = (rec[:, :, 1] - base).astype(np.float64)
    sm = rec[:, :, 2]
    raw = rec[:, :, 3:16] & 0xFFFFFFFF
    # SM clock (32 bits) at each phase, relative to the entry clock in word 6 (index 3 here)
    cyc = np.where(raw != 0, (raw - raw[:, :, 3:4]) % (1 << 32), 0).astype(np.float64)
    cyc[:, :, 3] = 0.0
    mhz = cyc[:, :, 5] / np.maximum(t_out - t_in, 1.0) * 1e3
    ns = cyc / np.maximum(mhz[:, :, None], 1.0) * 1e3
    start, end = t_in.min(axis=1), t_out.max(axis=1)
    out = {"sm_mhz": round(float(np.median(mhz)), 1)}
    out["span_ns"] = round(float(med(list(end - start))), 1)
    if n > 1:
        out["overlap_prev_ns"] = round(float(med(list(end[:-1] - start[1:]))), 1)
        out["period_ns"] = round(float(med(list(end[1:] - end[:-1]))), 1)
    out["cta_entry_spread_ns"] = round(float(med(list(t_in.max(axis=1) - start))), 1)
    out["cta_exit_spread_ns"] = round(float(med(list(end - t_out.min(axis=1)))), 1)
    # per SM: first entry of launch i minus last exit of launch i-1 on the same SM
    # (negative: the two launches' CTAs were resident on that SM together)
    hand = []
    for i in range(1, n):
        for smv in np.unique(sm[i]):
            prev = t_out[i - 1][sm[i - 1] == smv]
            if prev.size:
                hand.append(float(t_in[i][sm[i] == smv].min() - prev.max()))
    out["sm_handoff_ns"] = round(float(med(hand)), 1) if hand else None
    for j, key in enumerate(PHASE_KEYS):
        if not np.any(cyc[:, :, j]):
            continue
        out[key + "_ns"] = round(float(med([med(list(ns[i, :, j])) for i in range(n)])), 1)
        out[key + "_ns_max"] = round(float(med([float(ns[i, :, j].max()) for i in range(n)])), 1)
    return out


def phase_times(args):
    """Where a launch's time goes: each launch of a 20-launch graph (rotating over weight
    copies totalling >= 4x L2) records per CTA the global time at entry and exit and the SM
    cycles to warp 0's first copies issued, to the end of the wait for the previous kernel,
    to x staged, to warp 0's last row group, to the CTA's end, and to the landing of each
    of warp 0's first ring stages, polled before the wait (recording only).  Reported per (workload,
    ntok, launch mode): medians over the launches of the per-launch medians over CTAs (in
    ns, cycles converted with the clock each CTA saw), the launch span (first entry to last
    exit), the overlap with the previous launch and the period (exit to exit)."""
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    ntoks = [int(v) for v in args.sweep_ntoks.split(",")]
    dev = torch.device("cuda:0")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for name in args.phases.split(","):
        w = workloads.WORKLOADS[name]
        base = torch.from_numpy(gen_packed(qg, w)).to(dev)
        copies = max(1, math.ceil(4 * l2 / base.numel()))
        pool = [base] + [base.clone() for _ in range(copies - 1)]
        n = max(20, copies)                 # one replay reads >= 4x L2 of weights
        buf = torch.zeros(n * qg.QG_PHASE_SLOT_WORDS, dtype=torch.int64, device=dev)
        x = torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev)
        y = torch.empty((4, w.n_out), dtype=torch.float32, device=dev)
        am = torch.empty(4, dtype=torch.int32, device=dev)
        ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(w.n_out, 4), dtype=torch.uint8, device=dev)
        wb = workloads_bytes(w.fmt, w.n_out, w.n_in)
        for ntok in ntoks:
            desc = qg.qg_describe_tile(w.fmt, w.n_out, w.n_in, ntok)
            grid = int(desc.split("grid=")[1])

            def call(i, ntok=ntok):
                if w.argmax:
                    qg.qgemv_argmax(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y[:ntok], am, ws, ntok)
                else:
                    qg.qgemv(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y[:ntok], ntok)
            for mode, flags in (("early_start", qg.QG_LAUNCH_EARLY_START), ("plain", 0)):
                qg.qg_set_launch_options(flags)
                us = time_graph(torch, call, n=n, reps=3)
                # the captured launches take slots 0..n-1 in launch order
                buf.zero_()
                qg.qg_set_phase_record(buf, n)
                try:
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, capture_error_mode="thread_local"):
                        for i in range(n):
                            call(i)
                finally:
                    qg.qg_set_phase_record(None)
                g.replay()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                ev[0].record()
                g.replay()
                ev[1].record()
                torch.cuda.synchronize()
                us_rec = ev[0].elapsed_time(ev[1]) / n * 1e3
                del g
                rec = buf.view(n, -1)[:, :grid * qg.QG_PHASE_WORDS].reshape(n, grid, qg.QG_PHASE_WORDS).cpu().numpy()
                out = {"name": name, "ntok": ntok, "mode": mode, "tile": desc, "us_per_launch": round(us, 3),
                       "us_per_launch_recording": round(us_rec, 3), "gbs": round(wb / us / 1e3, 1)}
                out.update(summarize_phases(rec))
                print(json.dumps(out), flush=True)
        del pool, base, buf
        torch.cuda.empty_cache()
    qg.qg_set_launch_options(0)


def sweep_experts(args):
    """The routed-expert layer (the bench's 512-expert Q8_0 layer, share 0.65) under each
    tile override spec: plan, gate/up and down times per ntok."""
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    peak, _ = peaks()
    qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
    layer = workloads.EXPERT_LAYERS["q8_0_experts_512x2560x640_top10"]
    for spec in args.sweep_experts.split(";"):
        qg.qg_set_tile_override(spec or None)
        r = experts_detail(qg, torch, dev, peak, layer, routings=32)
        print(json.dumps({"spec": spec, "tile": r["tile"],
                          "ntok": {t: {k: v[k]["us"] for k in ("gate_up", "down", "layer")}
                                   for t, v in r["ntok"].items()}}), flush=True)
        torch.cuda.empty_cache()
    qg.qg_set_tile_override(None)


# ----------------------------------------------------------------------------- entry

def one_shape(spec: str, argmax: bool = False):
    """Run one synthetic shape three times (the small case an ncu capture profiles), through
    qgemv or, with argmax, qgemv_argmax."""
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    parts = spec.split(",", 4)
    fmt, n_out, n_in, ntok = parts[0], int(parts[1]), int(parts[2]), int(parts[3])
    if len(parts) > 4 and parts[4]:
        qg.qg_set_tile_override(parts[4])
    w = workloads.Workload("one", fmt, n_out, n_in, 130)
    packed = torch.from_numpy(gen_packed(qg, w)).cuda()
    x = torch.from_numpy(workloads.activations(w.seed, n_in, 4)).cuda()
    y = torch.empty((4, n_out), device="cuda")
    am = torch.empty(4, dtype=torch.int32, device="cuda")
    ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, 4), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        if argmax:
            qg.qgemv_argmax(fmt, packed, n_out, n_in, x, y[:ntok], am, ws, ntok)
        else:
            qg.qgemv(fmt, packed, n_out, n_in, x, y[:ntok], ntok)
    torch.cuda.synchronize()
    assert qg.qg_device_status() == 0
    print("ok", qg.qg_describe_tile(fmt, n_out, n_in, ntok))


def profile_step(n: int):
    """The headline step's 8 qgemv_argmax launches (both heads, ntok 1..4), one warm-up
    step then n steps, eagerly with early start: a bounded case for ncu launch lists
    and DRAM-traffic captures of the step's kernels."""
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    heads = [workloads.WORKLOADS[n_] for n_ in HEADS]
    W = {w.name: torch.from_numpy(gen_packed(qg, w)).cuda() for w in heads}
    X = {w.name: torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).cuda() for w in heads}
    Y = {w.name: torch.empty((4, w.n_out), device="cuda") for w in heads}
    am = torch.empty(4, dtype=torch.int32, device="cuda")
    ws = {w.name: torch.zeros(qg.qgemv_argmax_workspace_bytes(w.n_out, 4), dtype=torch.uint8, device="cuda")
          for w in heads}
    qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
    for _ in range(1 + n):
        for ntok in NTOKS:
            for w in heads:
                qg.qgemv_argmax(w.fmt, W[w.name], w.n_out, w.n_in, X[w.name], Y[w.name][:ntok], am, ws[w.name], ntok)
    torch.cuda.synchronize()
    assert qg.qg_device_status() == 0
    print("ok", 8 * (1 + n), "launches")


def one_experts(spec: str, one_launch: bool = False):
    """Five routed-expert layers (plan, gate/up with the activation and the down
    prefetch, down; or, with one_launch, qgemv_expert_layer) at `ntok` on a 64-expert
    Q8_0 stack of the expert table's shapes (the small case an ncu capture profiles)."""
    import torch
    import block_quantized_token_format_gb300 as qg
    import __graft_entry__
    __graft_entry__.build()
    ntok = int(spec)
    layer = workloads.EXPERT_LAYERS["q8_0_experts_512x2560x640_top10"]
    E, dm, ff, U = 64, layer.d_model, layer.d_ff, 32
    stk = {}
    for key, (n_out, n_in, seed) in {"gu": (2 * ff, dm, layer.seed), "dn": (dm, ff, layer.seed + 1)}.items():
        stride = qg.qg_row_stride(layer.fmt, n_in)
        host = np.empty(U * n_out * stride, dtype=np.uint8)
        for k in range(U):
            qg.qg_pack(layer.fmt, workloads.expert_matrix(seed, k, n_out, n_in),
                       out=host[k * n_out * stride:(k + 1) * n_out * stride])
        stk[key] = torch.from_numpy(host).cuda().repeat(E // U)
    G = ntok * layer.topk
    x = torch.from_numpy(workloads.activations(layer.seed, dm, ntok)).cuda()
    act = torch.zeros((G, ff), device="cuda")
    y = torch.empty((G, dm), device="cuda")
    plan = torch.empty(qg.qg_expert_plan_ints(G), dtype=torch.int32, device="cuda")
    qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
    ws = torch.zeros(qg.qgemv_expert_layer_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for r in range(5):
        ids = torch.from_numpy(workloads.routing(1000 + r, ntok, layer.topk, E, layer.share)).cuda()
        if one_launch:
            qg.qgemv_expert_layer(layer.fmt, stk["gu"], stk["dn"], E, dm, ff, x, ids, plan, act, y, ws)
            continue
        qg.qg_expert_plan(ids, E, plan)
        qg.qgemv_experts(layer.fmt, stk["gu"], E, 2 * ff, dm, x, plan, G, act, swiglu=True, W_next=stk["dn"],
                         next_n_out=dm, next_n_in=ff)
        qg.qgemv_experts(layer.fmt, stk["dn"], E, dm, ff, act, plan, G, y, x_by_slot=True, plan_ready=True)
    torch.cuda.synchronize()
    assert qg.qg_device_status() == 0
    print("ok", qg.qg_describe_expert_tile(layer.fmt, 2 * ff, dm))


def main():
    args = parse_args()
    if args.one_experts:
        one_experts(args.one_experts)
        return
    if args.one_layer:
        one_experts(args.one_layer, one_launch=True)
        return
    if args.cpu_worker:
        cpu_worker(args.cpu_worker)
        return
    if args.sweep:
        tile_sweep(args)
        return
    if args.sweep_experts:
        sweep_experts(args)
        return
    if args.phases:
        phase_times(args)
        return
    if args.one:
        one_shape(args.one.replace(";", ","))
        return
    if args.one_argmax:
        one_shape(args.one_argmax.replace(";", ","), argmax=True)
        return
    if args.profile_step:
        profile_step(args.profile_step)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.impl == "reference":
        res = reference_arm(args, rank, world)
    else:
        res = main_gpu(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
