"""Seeded synthetic inputs for the block-quantized mat-vec workloads.

This module holds shape tables and random-number generation only: no
quantization, no dequantization and none of the mat-vec's arithmetic.  The
oracle-side tests, the CUDA-side tests and ``bench.py`` all draw their fp32
weights and activations here, so both sides see the same numbers.

Recipe (model weights are not needed and not available; these stand in):

* W is fp32, drawn as ``standard_normal(float32) * float32(0.02)`` in blocks of
  4096 rows; block ``i`` of a matrix with seed ``s`` uses
  ``Generator(PCG64(SeedSequence(s, spawn_key=(i,))))``, so any row can be
  regenerated without drawing the whole matrix.
* x is fp32 N(0, 1): one ``[4, n_in]`` draw from seed ``s + 1``; a call with
  ``ntok = k`` uses rows ``0..k-1``, so token 0 of every ntok is the same vector.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

ROW_CHUNK = 4096
W_STD = np.float32(0.02)
MAX_NTOK = 4


@dataclass(frozen=True)
class Workload:
    name: str
    fmt: str          # "q8_0" | "q4_0" | "affine4_g64" | "bf16"
    n_out: int
    n_in: int
    seed: int
    argmax: bool = False
    note: str = ""


# The five workload families of the mat-vec at ntok = 1..4 (shapes are n_out x n_in).
WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    # config 0: the small square projection.
    Workload("q8_0_2560x2560", "q8_0", 2560, 2560, 100, note="small case"),
    # config 1: the dense projection set, n_in -> n_out = 2560->6144/10240/12288 and 6144->2560.
    Workload("q8_0_6144x2560", "q8_0", 6144, 2560, 110),
    Workload("q8_0_10240x2560", "q8_0", 10240, 2560, 111),
    Workload("q8_0_12288x2560", "q8_0", 12288, 2560, 112),
    Workload("q8_0_2560x6144", "q8_0", 2560, 6144, 113),
    # config 2: the 8192x2560 format comparison, Q4_0 and BF16 from the same fp32 W.
    Workload("q4_0_8192x2560", "q4_0", 8192, 2560, 120),
    Workload("bf16_8192x2560", "bf16", 8192, 2560, 120),
    # Q5_0 (the Track 1 report's 5-bit draft format) on the same 8192x2560 matrix.
    Workload("q5_0_8192x2560", "q5_0", 8192, 2560, 120),
    # config 3: Q8_0 LM head with fused argmax; the drafted-vocab variant is a row prefix.
    Workload("q8_0_head_248320x2560", "q8_0", 248320, 2560, 130, argmax=True),
    Workload("q8_0_head_106299x2560", "q8_0", 106299, 2560, 130, argmax=True,
             note="first 106299 rows of the 248320-row head"),
    # config 4: affine 4-bit (group 64) drafter LM head with fused argmax.
    Workload("affine4_head_248320x5120", "affine4_g64", 248320, 5120, 140, argmax=True),
]}

# A draft vocabulary given as an id list (not a row prefix): 106,299 ids of the
# 248,320-row Q8_0 head, drawn without replacement and sorted, from this seed.
DRAFT_IDS = {"q8_0_head_248320x2560": (106299, 131)}

# The dense projection set timed as one step by bench.py.
DENSE_SET = ["q8_0_6144x2560", "q8_0_10240x2560", "q8_0_12288x2560", "q8_0_2560x6144"]


@dataclass(frozen=True)
class ExpertLayer:
    """Routed experts of one mixture-of-experts layer: n_experts experts, each a gate
    and an up projection d_model -> d_ff (stacked as 2 * d_ff rows: gate, then up)
    and a down projection d_ff -> d_model; top-k routing with inter-token share."""
    name: str
    fmt: str
    n_experts: int
    d_model: int
    d_ff: int
    topk: int
    share: float
    seed: int


# Routed experts at the size the routed-expert table implies (~1.46 MB per expert at
# about 2.5 bits per weight: 2 x 2560 x 640 gate/up + 640 x 2560 down), 512 experts,
# top-10 routing, 65% inter-token share; stored here in Q8_0.
EXPERT_LAYERS: dict[str, ExpertLayer] = {e.name: e for e in [
    ExpertLayer("q8_0_experts_512x2560x640_top10", "q8_0", 512, 2560, 640, 10, 0.65, 150),
    # The M2 Max page's routing dumps: no two consecutive tokens picked a common expert.
    ExpertLayer("q8_0_experts_512x2560x640_top10_share0", "q8_0", 512, 2560, 640, 10, 0.0, 150),
]}


def expert_matrix(seed: int, e: int, n_out: int, n_in: int) -> np.ndarray:
    """Expert e's fp32 matrix of a stack drawn from ``seed`` (its own weight seed)."""
    return weights(seed * 65536 + e, n_out, n_in)


def _chunk_rng(seed: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(chunk,))))


def weight_chunk(seed: int, n_out: int, n_in: int, chunk: int) -> np.ndarray:
    """Rows ``[chunk*4096, min(n_out, (chunk+1)*4096))`` of the fp32 weight matrix."""
    r0 = chunk * ROW_CHUNK
    if r0 >= n_out or chunk < 0:
        raise IndexError(f"chunk {chunk} outside a {n_out}-row matrix")
    rows = min(ROW_CHUNK, n_out - r0)
    z = _chunk_rng(seed, chunk).standard_normal((rows, n_in), dtype=np.float32)
    return z * W_STD


def iter_weight_chunks(seed: int, n_out: int, n_in: int):
    """Yield ``(row0, W_chunk)`` over the whole matrix, 4096 rows at a time."""
    for c in range((n_out + ROW_CHUNK - 1) // ROW_CHUNK):
        yield c * ROW_CHUNK, weight_chunk(seed, n_out, n_in, c)


def weights(seed: int, n_out: int, n_in: int) -> np.ndarray:
    """The whole fp32 matrix (small shapes only)."""
    return np.concatenate([w for _, w in iter_weight_chunks(seed, n_out, n_in)], axis=0)


def weight_rows(seed: int, n_out: int, n_in: int, rows) -> np.ndarray:
    """Selected rows of the fp32 matrix, regenerating only the 4096-row blocks they live in."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, n_in), dtype=np.float32)
    for c in np.unique(rows // ROW_CHUNK):
        blk = weight_chunk(seed, n_out, n_in, int(c))
        sel = np.nonzero(rows // ROW_CHUNK == c)[0]
        out[sel] = blk[rows[sel] - c * ROW_CHUNK]
    return out


def activations(seed: int, n_in: int, ntok: int) -> np.ndarray:
    """x as fp32 ``[ntok, n_in]``: rows 0..ntok-1 of one ``[4, n_in]`` N(0,1) draw from ``seed + 1``."""
    if not 1 <= ntok <= MAX_NTOK:
        raise ValueError("ntok must be in 1..4")
    g = np.random.Generator(np.random.PCG64(seed + 1))
    return np.ascontiguousarray(g.standard_normal((MAX_NTOK, n_in), dtype=np.float32)[:ntok])


def activations_with_outliers(seed: int, n_in: int, ntok: int, n_massive: int = 3, massive=(300.0, 3000.0),
                              n_moderate: int = 8, moderate=(10.0, 40.0)) -> np.ndarray:
    """x as fp32 ``[ntok, n_in]`` shaped like a transformer's hidden state: N(0,1) per token
    with a per-token scale in [0.5, 2], plus a few fixed "massive" channels (magnitude drawn
    log-uniformly in `massive`, random sign per token) and some moderate outlier channels
    (`moderate`), the channel indices shared by all tokens."""
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.standard_normal((ntok, n_in)).astype(np.float64) * g.uniform(0.5, 2.0, (ntok, 1))
    ch = g.choice(n_in, n_massive + n_moderate, replace=False)
    for j, c in enumerate(ch):
        lo, hi = massive if j < n_massive else moderate
        mag = np.exp(g.uniform(np.log(lo), np.log(hi), ntok))
        x[:, c] = mag * np.where(g.random(ntok) < 0.5, -1.0, 1.0)
    return np.ascontiguousarray(x.astype(np.float32))


def gaussian(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """A generic seeded fp32 normal array for small test cases."""
    g = np.random.Generator(np.random.PCG64(seed))
    return g.standard_normal(shape, dtype=np.float32) * np.float32(scale)


def draft_ids(seed: int, n_full: int, k: int) -> np.ndarray:
    """k distinct row ids of an n_full-row head, drawn without replacement and sorted (int32)."""
    g = np.random.Generator(np.random.PCG64(seed))
    return np.sort(g.choice(n_full, size=k, replace=False)).astype(np.int32)


def routing(seed: int, ntok: int, topk: int, n_experts: int, share: float) -> np.ndarray:
    """Synthetic top-k routing ``ids[ntok, topk]`` (int32), distinct experts per token.

    Token 0 draws topk experts uniformly.  Each later token's choice j repeats, with
    probability ``share``, an expert that an earlier token chose (uniform among those
    this token has not taken yet), otherwise draws one that no token has chosen yet;
    so about ``topk + (ntok - 1) * topk * (1 - share)`` experts are active in a step.
    (When one of the two pools is empty the choice comes from the other.)
    """
    if not 1 <= topk <= n_experts:
        raise ValueError("need 1 <= topk <= n_experts")
    g = np.random.Generator(np.random.PCG64(seed))
    ids = np.zeros((ntok, topk), dtype=np.int32)
    used: list[int] = []
    for t in range(ntok):
        mine: list[int] = []
        for _ in range(topk):
            old = [e for e in used if e not in mine]
            free = np.setdiff1d(np.arange(n_experts), np.array(used + mine, dtype=np.int64))
            if old and (len(free) == 0 or (t > 0 and g.random() < share)):
                e = old[int(g.integers(len(old)))]
            else:
                e = int(free[int(g.integers(len(free)))])
            mine.append(e)
        for e in mine:
            if e not in used:
                used.append(e)
        ids[t] = mine
    return ids

