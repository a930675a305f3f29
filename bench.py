#!/usr/bin/env python
"""Benchmark: effective weight GB/s of the block-quantized mat-vec (qgemv) on GB300.

One step = one pass of the Q8_0 dense projection set (n_in -> n_out: 2560->6144,
2560->10240, 2560->12288, 6144->2560) at ntok = 1, 2, 3 and 4: 16 kernel launches
over 379 MB of distinct weights.  value = weight bytes / time (scales included,
1e9 B per GB).  The steps are replayed from CUDA graphs of 10 steps (160
launches; the kernels are 3-12 us long, launching them one by one from Python
would time the host).  Also reported, outside the timed region:

* per_workload: every workload family x ntok (including the fused LM-head
  argmax heads), median of 5 graph replays of 50 launches rotating over weight
  copies totalling >= 4x L2;
* e2e: the same step through the public API with host buffers, per call
  (pinned x uploaded, y read back, host synchronized every step, no graph);
* roofline of the dominant kernel, cpu_baseline (the fp64 oracle on the host).

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
WORKLOAD_NAME = ("Q8_0 dense projection set (n_in->n_out 2560->6144, 2560->10240, "
                 "2560->12288, 6144->2560) at ntok=1,2,3,4")
NTOKS = (1, 2, 3, 4)
PEAK_FALLBACK_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-detail", action="store_true", help="skip the per-workload table")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--detail-only", default="", help="comma list of workload names for the table")
    p.add_argument("--one-experts", default="", help="ntok: five routed-expert layers on a 64-expert stack "
                   "(the small case an ncu capture profiles)")
    p.add_argument("--one-layer", default="", help="ntok: as --one-experts, with the layer as one launch")
    p.add_argument("--one", default="", help="fmt,n_out,n_in,ntok[,tile spec]: run one shape 3 times "
                                             "(a small case for ncu) and exit")
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

    def mark(self):
        return time.time()

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


# ----------------------------------------------------------------------------- CPU oracle legs

def cpu_worker(spec: str):
    """Run inside a fresh process with BLAS pinned to one thread: time the oracle."""
    import oracle
    cfg = json.loads(spec)
    names, steps, warm, frac = cfg["names"], cfg["steps"], cfg["warmup"], cfg["row_frac"]
    data = []
    for name in names:
        w = workloads.WORKLOADS[name]
        rows = max(64, int(math.ceil(w.n_out * frac)))
        W = workloads.weight_rows(w.seed, w.n_out, w.n_in, np.arange(rows))
        data.append((w, rows, oracle.quantize(w.fmt, W), workloads.activations(w.seed, w.n_in, 4)))
    per_step_bytes = sum(workloads_bytes(w.fmt, rows, w.n_in) for w, rows, _, _ in data) * len(NTOKS)

    def step():
        for ntok in NTOKS:
            for w, rows, canon, x in data:
                oracle.gemv(w.fmt, canon, rows, w.n_in, x[:ntok])

    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "steps": steps, "bytes_per_step": per_step_bytes,
                      "rows": {w.name: rows for w, rows, _, _ in data}}))


def run_cpu_oracle(names, steps, warmup, row_frac):
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    spec = json.dumps({"names": names, "steps": steps, "warmup": warmup, "row_frac": row_frac})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", spec],
                       capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


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
    peak, peak_kind = peaks()
    stream = torch.cuda.current_stream()

    # --- the dense set: two sets of 16 distinct weight buffers (one per shape x ntok)
    dense = [workloads.WORKLOADS[n] for n in workloads.DENSE_SET]
    host = {w.name: gen_packed(qg, w) for w in dense}
    bufs = {}
    for s in range(2):
        for w in dense:
            base = torch.from_numpy(host[w.name]).to(dev)
            for ntok in NTOKS:
                bufs[(s, w.name, ntok)] = base if ntok == 1 else base.clone()
    xs = {w.name: torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev) for w in dense}
    ys = {(w.name, ntok): torch.empty((ntok, w.n_out), dtype=torch.float32, device=dev)
          for w in dense for ntok in NTOKS}
    step_bytes = sum(workloads_bytes(w.fmt, w.n_out, w.n_in) for w in dense) * len(NTOKS)
    distinct = sum(b.numel() for b in bufs.values())

    def launches(s, ntoks):
        for ntok in ntoks:
            for w in dense:
                qg.qgemv(w.fmt, bufs[(s, w.name, ntok)], w.n_out, w.n_in, xs[w.name], ys[(w.name, ntok)], ntok)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    G = 10   # steps per chunk graph (even: the two buffer sets alternate inside it)

    def capture(early: bool):
        """One graph per step (per buffer set) and one graph of G consecutive steps."""
        qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START if early else 0)
        for s in range(2):                              # warm every kernel / cache occupancy before capture
            launches(s, NTOKS)
        torch.cuda.synchronize()
        single = []
        for s in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                launches(s, NTOKS)
            single.append(g)
        chunk = torch.cuda.CUDAGraph()
        with torch.cuda.graph(chunk, capture_error_mode="thread_local"):
            for i in range(G):
                launches(i % 2, NTOKS)
        torch.cuda.synchronize()
        return single, chunk

    def run(graphs, K, Wm):
        single, chunk = graphs
        for i in range(Wm):
            single[i % 2].replay()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        start.record()
        i = 0
        while i + G <= K:
            chunk.replay()
            i += G
        while i < K:
            single[i % 2].replay()
            i += 1
        end.record()
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
        return start.elapsed_time(end), t0, t1

    K, Wm = args.steps, max(3, args.warmup)
    # Secondary: ordinary launches (each kernel waits for the previous one to finish).
    plain_graphs = capture(False)
    plain_ms, _, _ = run(plain_graphs, max(10, K // 4), Wm)
    plain_value = step_bytes * max(10, K // 4) / (plain_ms * 1e-3) / 1e9
    del plain_graphs
    # Headline: early start (programmatic dependent launch): the weights are written
    # once before the run, so a call may stream them while the previous call finishes.
    graphs = capture(True)
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (str(uuid) if uuid else str(local_rank))
    with ClockSampler(gpu_id) as clk:
        total_ms, t_wall0, t_wall1 = run(graphs, K, Wm)
    clocks = clk.summary(t_wall0, t_wall1)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / K
    value = job_gbs(step_bytes, K, world, total_ms)

    # --- roofline of the dominant kernel.  Every launch of the step is qgemv_kernel
    # (100% of the step's GPU time), so its average launch duration is the step time
    # over the 16 launches (consecutive launches overlap slightly under early start).
    step_algo = sum(algo_bytes(w.fmt, w.n_out, w.n_in, t) for w in dense for t in NTOKS)
    achieved = step_algo * K / (total_ms * 1e-3) / 1e9
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            td = json.load(f)
        if td.get("csrc_hash") == csrc_hash():
            traffic = td.get("traffic_bytes_per_launch")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": "qgemv_kernel (all 16 launches of the step: 4 shapes x ntok 1..4)",
                "algorithmic_bytes_per_launch": round(step_algo / 16),
                "avg_launch_us": round(ms_per_step / 16 * 1e3, 3), "peak_kind": peak_kind}

    result = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
              "warmup": Wm, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
              "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
              "config": {"workload": WORKLOAD_NAME, "formats": "Q8_0 weights, fp32 x and y, fp32 accumulation",
                         "weight_bytes_per_step": step_bytes, "launches_per_step": 16,
                         "l2": f"inputs larger than L2: each step reads {step_bytes / 1e6:.0f} MB of distinct "
                               f"weights; two alternating sets ({distinct / 1e6:.0f} MB) vs L2 {l2 / 1e6:.0f} MB",
                         "timing": f"CUDA graph replay ({G} steps = {16 * G} launches per graph), "
                                   "CUDA events on the launch stream",
                         "launch": "early start (programmatic dependent launch, QG_LAUNCH_EARLY_START)",
                         "value_plain_launches": round(plain_value, 2),
                         "parallelism": "replicas" if world > 1 else "single GPU"},
              "frac_of_peak": round(value / world / peak, 4), "peak_gbs": peak, "peak_kind": peak_kind,
              "frac_of_nominal_7900": round(value / world / 7900.0, 4),
              "clocks": clocks, "gpu_launches": 16 * K, "roofline": roofline}

    # --- e2e through the public API with host buffers (no graph), rank-local.  A
    # step uploads every shape's x in one copy from pinned memory, makes the 16 calls
    # and reads every y back in one copy (x and y are views of one buffer each, as a
    # caller would lay them out), then waits for the host copy.
    x_elems = {w.name: 4 * w.n_in for w in dense}
    y_elems = {(w.name, ntok): ntok * w.n_out for w in dense for ntok in NTOKS}
    pin_x_all = torch.empty(sum(x_elems.values()), dtype=torch.float32).pin_memory()
    dx_all = torch.empty(pin_x_all.numel(), dtype=torch.float32, device=dev)
    pin_y_all = torch.empty(sum(y_elems.values()), dtype=torch.float32).pin_memory()
    dy_all = torch.empty(pin_y_all.numel(), dtype=torch.float32, device=dev)
    dx, dy, off = {}, {}, 0
    for w in dense:
        n = x_elems[w.name]
        pin_x_all[off:off + n].copy_(torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).reshape(-1))
        dx[w.name] = dx_all[off:off + n].view(4, w.n_in)
        off += n
    off = 0
    for k, n in y_elems.items():
        dy[k] = dy_all[off:off + n]
        off += n
    h2d = pin_x_all.numel() * 4
    d2h = pin_y_all.numel() * 4
    sh = qg.current_stream_handle()

    def e2e_step(s):
        dx_all.copy_(pin_x_all, non_blocking=True)
        for ntok in NTOKS:
            for w in dense:
                qg.qgemv(w.fmt, bufs[(s, w.name, ntok)], w.n_out, w.n_in, dx[w.name], dy[(w.name, ntok)], ntok,
                         stream=sh)
        pin_y_all.copy_(dy_all, non_blocking=True)
        stream.synchronize()

    for i in range(5):
        e2e_step(i % 2)
    n_e2e = max(50, min(2000, K // 10))
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i % 2)
    e2e_s = time.perf_counter() - t0
    result["e2e"] = {"value": round(step_bytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                     "how": "python qgemv calls per launch (ctypes), all x uploaded in one copy from pinned "
                            "memory and all y read back in one copy, host synchronized every step; no CUDA "
                            "graph; early start on"}

    if rank == 0 and not args.no_detail:
        result["per_workload"] = detail_table(args, qg, torch, dev, l2, peak)

    if rank == 0 and not args.no_cpu:
        try:
            cores = 1
            r = run_cpu_oracle(workloads.DENSE_SET, steps=1, warmup=0, row_frac=1.0)
            result["cpu_baseline"] = {"value": round(r["bytes_per_step"] * r["steps"] / r["seconds"] / 1e9, 4),
                                      "unit": "GB/s", "cores": cores, "kind": "oracle",
                                      "sample": "one full step of the workload (16 oracle calls: 4 shapes x ntok "
                                                "1..4, all rows), numpy fp64, BLAS pinned to 1 thread",
                                      "seconds": round(r["seconds"], 3),
                                      "host_cores_available": len(os.sched_getaffinity(0))}
        except Exception as e:  # noqa: BLE001
            result["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                      "sample": f"failed: {e}"}
    return result


def detail_table(args, qg, torch, dev, l2, peak):
    """Every workload x ntok: median of 5 replays of a 50-launch graph over rotating copies."""
    names = [n for n in workloads.WORKLOADS] if not args.detail_only else args.detail_only.split(",")
    table = {}
    cache = {}
    for name in names:
        w = workloads.WORKLOADS[name]
        src = name
        if name == "q8_0_head_106299x2560":
            src = "q8_0_head_248320x2560"
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
            n = 50
            for i in range(copies + 2):
                call(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                for i in range(n):
                    call(i)
            g.replay()
            times = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                times.append(a.elapsed_time(b) / n * 1e3)
            us = statistics.median(times)
            gbs = wbytes / (us * 1e-6) / 1e9
            row[str(ntok)] = {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "tile": qg.qg_describe_tile(w.fmt, w.n_out, w.n_in, ntok)}
            del g
        table[name] = {"fmt": w.fmt, "n_out": w.n_out, "n_in": w.n_in, "weight_bytes": wbytes,
                       "call": "qgemv_argmax" if w.argmax else "qgemv", "copies": copies, "ntok": row}
        del pool
        if name in workloads.DRAFT_IDS:
            table[f"{w.fmt}_draft_ids_{workloads.DRAFT_IDS[name][0]}_of_{w.n_out}x{w.n_in}"] = \
                draft_ids_detail(qg, torch, dev, l2, peak, w, base)
    cache.clear()
    torch.cuda.empty_cache()
    if not args.detail_only or any(n in workloads.EXPERT_LAYERS for n in names):
        for name in workloads.EXPERT_LAYERS:
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
    if rank != 0:
        return None
    K, Wm = args.steps, max(3, args.warmup)
    full_rows = sum(workloads.WORKLOADS[n].n_out for n in workloads.DENSE_SET)
    # a full step of the oracle takes seconds; sample rows so the run ends within ~2 minutes
    est_full_step_s = 6.0
    frac = min(1.0, 120.0 / ((K + Wm) * est_full_step_s))
    r = run_cpu_oracle(workloads.DENSE_SET, steps=K, warmup=Wm, row_frac=frac)
    value = r["bytes_per_step"] * r["steps"] / r["seconds"] / 1e9
    sample = (f"each step: the oracle on the first {frac:.4%} of each shape's rows (>= 64 rows), "
              f"4 shapes x ntok 1..4, numpy fp64, BLAS pinned to 1 thread")
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": round(r["seconds"] / K * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD_NAME, "rows_sampled": r["rows"]},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- entry

def one_shape(spec: str):
    """Run one synthetic shape three times (the small case an ncu capture profiles)."""
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
    for _ in range(3):
        qg.qgemv(fmt, packed, n_out, n_in, x, y, ntok)
    torch.cuda.synchronize()
    print("ok", qg.qg_describe_tile(fmt, n_out, n_in, ntok))


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
    if args.one:
        one_shape(args.one.replace(";", ","))
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
