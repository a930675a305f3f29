"""Tile sweep: measure GB/s per (workload, ntok, tile spec) on the current GPU.

    python -m block_quantized_token_format_gb300.tile_sweep NAMES [SPECS] [NTOKS] [--out FILE]

NAMES: comma list of workload names (workloads.WORKLOADS); SPECS: ';'-separated
tile specs (qg_set_tile_override grammar; default: a grid over rows per warp,
ring depth, warps per CTA and CTAs per SM); NTOKS: comma list (default 1,2,3,4).
Each point is the median of 3 CUDA-graph replays of 20 launches that rotate over
weight copies totalling >= 4x L2.  One JSON line per point goes to FILE
(default tile_sweep.jsonl in the working directory) and the best spec per (workload, ntok) is
printed.  Set QGEMV_EARLY_START=1 to sweep with early-start launches.  The
table in csrc/tile_select.cpp was filled from such sweeps.
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import os
import statistics
import sys

import numpy as np


def _gen_packed(qg, workloads, w, threads=16):
    from concurrent.futures import ThreadPoolExecutor
    stride = qg.qg_row_stride(w.fmt, w.n_in)
    out = np.empty(w.n_out * stride, dtype=np.uint8)

    def one(c):
        Wc = workloads.weight_chunk(w.seed, w.n_out, w.n_in, c)
        r0 = c * workloads.ROW_CHUNK
        qg.qg_pack(w.fmt, Wc, out=out[r0 * stride:(r0 + Wc.shape[0]) * stride])

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range((w.n_out + workloads.ROW_CHUNK - 1) // workloads.ROW_CHUNK)))
    return out


def main(argv=None):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch
    import workloads
    import block_quantized_token_format_gb300 as qg

    ap = argparse.ArgumentParser()
    ap.add_argument("names")
    ap.add_argument("specs", nargs="?", default="")
    ap.add_argument("ntoks", nargs="?", default="1,2,3,4")
    ap.add_argument("--out", default="tile_sweep.jsonl")
    a = ap.parse_args(argv)
    specs = a.specs.split(";") if a.specs else [
        f"rpw={r},depth={d},warps={w},ctas={c}"
        for r, d, w, c in itertools.product((1, 2, 4), (2, 3, 5, 8), (4, 8, 12, 16), (1, 2, 3))]
    ntoks = [int(v) for v in a.ntoks.split(",")]
    dev = torch.device("cuda:0")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    os.makedirs(os.path.dirname(os.path.abspath(a.out)), exist_ok=True)
    out = open(a.out, "a")
    for name in a.names.split(","):
        w = workloads.WORKLOADS[name]
        base = torch.from_numpy(_gen_packed(qg, workloads, w)).to(dev)
        copies = max(1, math.ceil(4 * l2 / base.numel()))
        pool = [base] + [base.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(workloads.activations(w.seed, w.n_in, 4)).to(dev)
        y = torch.empty((4, w.n_out), dtype=torch.float32, device=dev)
        wb = qg.qg_canonical_bytes(w.fmt, w.n_out, w.n_in)
        for ntok in ntoks:
            best = None
            for spec in specs:
                try:
                    qg.qg_set_tile_override(spec)
                    desc = qg.qg_describe_tile(w.fmt, w.n_out, w.n_in, ntok)
                except qg.QGError:
                    continue
                n = 20
                for i in range(copies):
                    qg.qgemv(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y, ntok)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, capture_error_mode="thread_local"):
                    for i in range(n):
                        qg.qgemv(w.fmt, pool[i % copies], w.n_out, w.n_in, x, y, ntok)
                g.replay()
                torch.cuda.synchronize()
                ts = []
                for _ in range(3):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    g.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) / n * 1e3)
                us = statistics.median(ts)
                rec = {"name": name, "ntok": ntok, "spec": spec, "desc": desc, "us": round(us, 3),
                       "gbs": round(wb / us / 1e3, 1)}
                out.write(json.dumps(rec) + "\n")
                out.flush()
                if best is None or rec["gbs"] > best["gbs"]:
                    best = rec
                del g
            print(json.dumps({"best": best}), flush=True)
        del pool, base
        torch.cuda.empty_cache()
    qg.qg_set_tile_override(None)


if __name__ == "__main__":
    main()
