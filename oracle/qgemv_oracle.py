"""CPU oracle for the block-quantized weight mat-vec (qgemv) -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  It shares no code with the CUDA library: it has its
own quantizers, its own byte layouts and its own fp64 arithmetic, written from
the sources below in plain numpy.

Sources (the web pages this library is built from; short tags used below):

* [Track2]  "Track 2 Audit & Optimization Report: M5 Metal Kernels for
  Multi-Token Speculative Decode", section 1 item 1 (the multi-token
  ``gemv.metal`` operator: per lane ``acc[NR][8]`` over ``ntok`` activation rows,
  Q8_0 with UNIT = 32) and table 2.1 (Q8_0 / BF16 shapes and GB/s).
* [M2Max]   "Where the time goes on an M2 Max", section "Dense K-quants are
  integer-ALU bound at small batches" (effective bandwidth = weight bytes /
  time for an 8192x2560 mat-vec by format: Q4_0, Q8_0, BF16).
* [Issue]   "perf(speculative): cut the MTP drafter's per-step cost", section
  "The cost model" (the affine 4-bit LM head: weight 635.7 + scales 39.7 +
  biases 39.7 MB) and "Phase 2" item 2a (fuse the LM-head projection and its
  argmax) and 2b (reduced draft vocabulary).
* [Track2] also section 1 item 2 (``moe_plan`` groups a step's (token, expert)
  pairs by expert; ``moe_gu`` / ``moe_down`` run each group with its own token
  count ne = 1..4, reading each unique expert once) and table 2.2 (routed
  experts at ntok 1, 3, 4: 10.0, 18.1 and 21.3 unique groups at share 0.65).
* [Track1]  "opus-mtp-turbo: Track 1 report", item 3 (Q4_0 / Q8_0 draft weights;
  one row's sum is independent of the token count).

What is computed (the plain definition; the fast path must equal it up to
rounding):

    y[t, o]   = sum_i deq(W)[o, i] * x[t, i]          (fp64, from the stored bytes)
    argmax[t] = min { o : y[t, o] == max_o' y[t, o'] }  (first index)

fp16 / bf16 scales, integer codes and fp32 activations are exact in fp64, so
``deq`` is exact and the only rounding is numpy's fp64 product and sum.

Quantizer rules (the pages name the formats but never spell the encoders out;
these are the workload definitions, with the readings listed where they are
silent):

* Q8_0, blocks of 32 along n_in: ``d = max|w| / 127`` in fp32, stored as fp16
  (round to nearest even); ``q = round(w / d)`` in fp32 with the unrounded d,
  rounding half away from zero, clamped to [-127, 127]; a block with
  ``max|w| == 0`` has ``d = 0, q = 0``.  Block bytes: fp16 d, then 32 int8 =
  34 B.  Dequant ``q * d``.
* Q4_0, blocks of 32: ``m`` = the signed value of largest magnitude (first on
  ties), ``d = m / -8`` in fp32, stored fp16; ``q = clamp(round(w / d) + 8, 0, 15)``
  (unrounded d, half away from zero); ``m == 0`` gives ``d = 0, q = 8``.
  Block bytes: fp16 d, then 16 bytes where byte j holds element j in its low
  nibble and element j + 16 in its high nibble (the GGUF order) = 18 B.
  Dequant ``(q - 8) * d``.
* Affine 4-bit, groups of 64: ``s = fp16((max - min) / 15)``, ``b = fp16(min)``,
  ``q = clamp(round((w - b) / s), 0, 15)`` in fp32 with the stored fp16 s and b
  (q = 0 when s == 0).  Three planes: uint32 words ``[n_out][n_in/8]`` holding 8
  codes, element k at bits [4k, 4k+4); fp16 scales ``[n_out][n_in/64]``; fp16
  biases ``[n_out][n_in/64]``.  Dequant ``q * s + b``.
* BF16: fp32 rounded to nearest even, row-major ``[n_out][n_in]``.
* Q5_0, blocks of 32 (named on the opus-mtp-turbo Track 1 report, item 3, with its
  quantization-error table; the pages give no layout): the 5-bit analogue of Q4_0.
  ``m`` = the signed value of largest magnitude (first on ties), ``d = m / -16`` in
  fp32, stored fp16; ``q = clamp(round(w / d) + 16, 0, 31)`` (unrounded d, half away
  from zero); ``m == 0`` gives ``d = 0, q = 16``.  Block bytes: fp16 d, a uint32
  whose bit j is bit 4 of element j's code, then 16 bytes where byte j holds the low
  nibbles of elements j and j + 16 (the Q4_0 order) = 22 B.  Dequant ``(q - 16) * d``.

"Parity unpinned": none.  Every function here is pinned by ``tests/`` against
exact rational brute force, hand-built golden blocks under ``tests/golden/``,
byte counts the pages print, round trips and algebraic identities.
"""
from __future__ import annotations

import numpy as np

Q8_0, Q4_0, AFFINE4_G64, BF16, Q5_0 = 0, 1, 2, 3, 4
FMT_NAMES = {"q8_0": Q8_0, "q4_0": Q4_0, "affine4_g64": AFFINE4_G64, "bf16": BF16, "q5_0": Q5_0}

# Weights per scale block / group.
BLOCK = {Q8_0: 32, Q4_0: 32, AFFINE4_G64: 64, BF16: 1, Q5_0: 32}

_Q8_BLOCK = np.dtype([("d", "<f2"), ("q", "i1", (32,))])
_Q4_BLOCK = np.dtype([("d", "<f2"), ("qs", "u1", (16,))])
_Q5_BLOCK = np.dtype([("d", "<f2"), ("qh", "<u4"), ("qs", "u1", (16,))])

ROW_CHUNK = 4096
GEMV_CHUNK = 1024


def fmt_id(fmt) -> int:
    return FMT_NAMES[fmt] if isinstance(fmt, str) else int(fmt)


# ----------------------------------------------------------------------------- sizes

def weight_bytes(fmt, n_out: int, n_in: int) -> int:
    """Bytes of the stored weights, scales and biases included (the numerator of
    the effective-bandwidth metric, [M2Max] "weight bytes / time").

    Q8_0 34 B per 32 weights, Q4_0 18 B per 32, affine4 0.5 B per weight plus
    2 + 2 B per 64, BF16 2 B per weight.
    """
    f = fmt_id(fmt)
    n = n_out * n_in
    if f == Q8_0:
        return n // 32 * 34
    if f == Q4_0:
        return n // 32 * 18
    if f == AFFINE4_G64:
        return n // 2 + (n // 64) * 4
    if f == BF16:
        return n * 2
    if f == Q5_0:
        return n // 32 * 22
    raise ValueError(fmt)


# ----------------------------------------------------------------------------- scalar helpers

def round_half_away(v: np.ndarray) -> np.ndarray:
    """Round an fp32 array to integers, ties away from zero (C ``roundf``)."""
    v = np.asarray(v, dtype=np.float32)
    t = np.trunc(v)
    frac = v - t                      # exact: the fractional bits of v
    return t + np.where(np.abs(frac) >= np.float32(0.5), np.sign(v), np.float32(0))


def f32_to_bf16_bits(w: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(w, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- quantizers

def quantize(fmt, W: np.ndarray) -> np.ndarray:
    """fp32 ``[n_out, n_in]`` -> the format's canonical bytes (uint8, 1-D)."""
    f = fmt_id(fmt)
    W = np.ascontiguousarray(W, dtype=np.float32)
    if f == Q8_0:
        return _quantize_q8_0(W)
    if f == Q4_0:
        return _quantize_q4_0(W)
    if f == AFFINE4_G64:
        return _quantize_affine4(W)
    if f == BF16:
        return f32_to_bf16_bits(W).reshape(-1).view(np.uint8).copy()
    if f == Q5_0:
        return _quantize_q5_0(W)
    raise ValueError(fmt)


def _quantize_q8_0(W: np.ndarray) -> np.ndarray:
    n_out, n_in = W.shape
    assert n_in % 32 == 0
    B = W.reshape(n_out, n_in // 32, 32)
    amax = np.max(np.abs(B), axis=2)
    d32 = amax / np.float32(127)
    safe = np.where(d32 > 0, d32, np.float32(1))
    q = round_half_away(B / safe[..., None])
    q = np.where(d32[..., None] > 0, q, np.float32(0))
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty((n_out, n_in // 32), dtype=_Q8_BLOCK)
    out["d"] = d32.astype(np.float16)
    out["q"] = q
    return out.reshape(-1).view(np.uint8).copy()


def _quantize_q4_0(W: np.ndarray) -> np.ndarray:
    n_out, n_in = W.shape
    assert n_in % 32 == 0
    B = W.reshape(n_out, n_in // 32, 32)
    idx = np.argmax(np.abs(B), axis=2)                      # first index on ties
    m = np.take_along_axis(B, idx[..., None], axis=2)[..., 0]
    d32 = m / np.float32(-8)
    safe = np.where(d32 != 0, d32, np.float32(1))
    q = round_half_away(B / safe[..., None]) + np.float32(8)
    q = np.where(d32[..., None] != 0, q, np.float32(8))
    q = np.clip(q, 0, 15).astype(np.uint8)
    out = np.empty((n_out, n_in // 32), dtype=_Q4_BLOCK)
    out["d"] = d32.astype(np.float16)
    out["qs"] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(-1).view(np.uint8).copy()


def _quantize_q5_0(W: np.ndarray) -> np.ndarray:
    n_out, n_in = W.shape
    assert n_in % 32 == 0
    B = W.reshape(n_out, n_in // 32, 32)
    first = np.argmax(np.abs(B), axis=2)                    # first index on ties
    m5 = np.take_along_axis(B, first[..., None], axis=2)[..., 0]
    d32 = m5 / np.float32(-16)
    safe = np.where(d32 != 0, d32, np.float32(1))
    q = round_half_away(B / safe[..., None]) + np.float32(16)
    q = np.where(d32[..., None] != 0, q, np.float32(16))
    q = np.clip(q, 0, 31).astype(np.uint32)
    out = np.empty((n_out, n_in // 32), dtype=_Q5_BLOCK)
    out["d"] = d32.astype(np.float16)
    out["qh"] = np.sum(((q >> np.uint32(4)) & np.uint32(1)) << np.arange(32, dtype=np.uint32), axis=2,
                       dtype=np.uint32)
    lo = (q & np.uint32(0xF)).astype(np.uint8)
    out["qs"] = lo[..., :16] | (lo[..., 16:] << 4)
    return out.reshape(-1).view(np.uint8).copy()


def _quantize_affine4(W: np.ndarray) -> np.ndarray:
    n_out, n_in = W.shape
    assert n_in % 64 == 0
    G = W.reshape(n_out, n_in // 64, 64)
    mn = G.min(axis=2)
    mx = G.max(axis=2)
    s16 = ((mx - mn) / np.float32(15)).astype(np.float16)
    b16 = mn.astype(np.float16)
    s32 = s16.astype(np.float32)
    b32 = b16.astype(np.float32)
    safe = np.where(s32 != 0, s32, np.float32(1))
    q = round_half_away((G - b32[..., None]) / safe[..., None])
    q = np.where(s32[..., None] != 0, q, np.float32(0))
    q = np.clip(q, 0, 15).astype(np.uint32).reshape(n_out, n_in // 8, 8)
    words = np.zeros((n_out, n_in // 8), dtype=np.uint32)
    for k in range(8):
        words |= q[..., k] << np.uint32(4 * k)
    return np.concatenate([
        words.astype("<u4").reshape(-1).view(np.uint8),
        s16.astype("<f2").reshape(-1).view(np.uint8),
        b16.astype("<f2").reshape(-1).view(np.uint8),
    ])


# ----------------------------------------------------------------------------- dequantizers

def dequantize(fmt, packed: np.ndarray, n_out: int, n_in: int) -> np.ndarray:
    """Canonical bytes -> fp64 ``[n_out, n_in]`` (exact)."""
    f = fmt_id(fmt)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size != weight_bytes(f, n_out, n_in):
        raise ValueError(f"expected {weight_bytes(f, n_out, n_in)} bytes, got {packed.size}")
    if f == Q8_0:
        blk = packed.view(_Q8_BLOCK).reshape(n_out, n_in // 32)
        d = blk["d"].astype(np.float64)
        q = blk["q"].astype(np.float64)
        return (q * d[..., None]).reshape(n_out, n_in)
    if f == Q4_0:
        blk = packed.view(_Q4_BLOCK).reshape(n_out, n_in // 32)
        d = blk["d"].astype(np.float64)
        lo = (blk["qs"] & 0x0F).astype(np.float64)
        hi = (blk["qs"] >> 4).astype(np.float64)
        q = np.concatenate([lo, hi], axis=2)                # elements 0..15, then 16..31
        return ((q - 8.0) * d[..., None]).reshape(n_out, n_in)
    if f == AFFINE4_G64:
        nw = n_out * n_in // 8
        ng = n_out * n_in // 64
        words = packed[: nw * 4].view("<u4").reshape(n_out, n_in // 8)
        s = packed[nw * 4: nw * 4 + ng * 2].view("<f2").astype(np.float64).reshape(n_out, n_in // 64)
        b = packed[nw * 4 + ng * 2:].view("<f2").astype(np.float64).reshape(n_out, n_in // 64)
        q = np.stack([(words >> np.uint32(4 * k)) & np.uint32(0xF) for k in range(8)], axis=2)
        q = q.reshape(n_out, n_in // 64, 64).astype(np.float64)
        return (q * s[..., None] + b[..., None]).reshape(n_out, n_in)
    if f == BF16:
        return bf16_bits_to_f64(packed.view("<u2")).reshape(n_out, n_in)
    if f == Q5_0:
        blk = packed.view(_Q5_BLOCK).reshape(n_out, n_in // 32)
        d = blk["d"].astype(np.float64)
        lo = np.concatenate([blk["qs"] & 0x0F, blk["qs"] >> 4], axis=2).astype(np.uint32)   # elements 0..31
        hb = (blk["qh"][..., None] >> np.arange(32, dtype=np.uint32)) & np.uint32(1)
        q = (lo | (hb << np.uint32(4))).astype(np.float64)
        return ((q - 16.0) * d[..., None]).reshape(n_out, n_in)
    raise ValueError(fmt)


def row_slice(fmt, packed: np.ndarray, n_out: int, n_in: int, r0: int, r1: int) -> np.ndarray:
    """Canonical bytes of rows [r0, r1) as a stand-alone ``(r1 - r0) x n_in`` matrix."""
    f = fmt_id(fmt)
    if f == AFFINE4_G64:
        nw = n_out * n_in // 8
        ng = n_out * n_in // 64
        w = packed[: nw * 4].reshape(n_out, n_in // 2)[r0:r1]
        s = packed[nw * 4: nw * 4 + ng * 2].reshape(n_out, n_in // 32)[r0:r1]
        b = packed[nw * 4 + ng * 2:].reshape(n_out, n_in // 32)[r0:r1]
        return np.concatenate([w.reshape(-1), s.reshape(-1), b.reshape(-1)])
    per_row = weight_bytes(f, 1, n_in)
    return packed.reshape(n_out, per_row)[r0:r1].reshape(-1)


# ----------------------------------------------------------------------------- the mat-vec

def gemv(fmt, packed: np.ndarray, n_out: int, n_in: int, x: np.ndarray, rows=None) -> np.ndarray:
    """fp64 ``y[t, o] = sum_i deq(W)[o, i] * x[t, i]`` ([Track2] section 1, item 1).

    Works 1024 rows at a time: dequantize the rows to fp64, then, token by
    token, one fp64 matrix-vector product with that token's fp32 activations
    promoted to fp64.  Each token is its own product, so a token's outputs do
    not depend on how many tokens share the call ([Track1] item 3: one row's
    sum is independent of the token count).  ``rows`` (an index array)
    restricts the output to those rows.  Returns ``[ntok, n_out]`` (or
    ``[ntok, len(rows)]``).
    """
    f = fmt_id(fmt)
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    if x64.ndim == 1:
        x64 = x64[None, :]
    assert x64.shape[1] == n_in
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        out = np.empty((x64.shape[0], rows.size), dtype=np.float64)
        for r in np.unique(rows // ROW_CHUNK):
            r0 = int(r) * ROW_CHUNK
            r1 = min(n_out, r0 + ROW_CHUNK)
            sel = np.nonzero(rows // ROW_CHUNK == r)[0]
            deq = dequantize(f, row_slice(f, packed, n_out, n_in, r0, r1), r1 - r0, n_in)
            sub = np.ascontiguousarray(deq[rows[sel] - r0])
            for t in range(x64.shape[0]):
                out[t, sel] = sub @ x64[t]
        return out
    y = np.empty((x64.shape[0], n_out), dtype=np.float64)
    for r0 in range(0, n_out, GEMV_CHUNK):
        r1 = min(n_out, r0 + GEMV_CHUNK)
        deq = dequantize(f, row_slice(f, packed, n_out, n_in, r0, r1), r1 - r0, n_in)
        for t in range(x64.shape[0]):
            y[t, r0:r1] = deq @ x64[t]
    return y


def gemv_abs(fmt, packed: np.ndarray, n_out: int, n_in: int, x: np.ndarray, rows=None) -> np.ndarray:
    """fp64 ``sum_i |deq(W)[o, i] * x[t, i]|``: the per-output error normaliser."""
    f = fmt_id(fmt)
    x64 = np.abs(np.asarray(x, dtype=np.float32).astype(np.float64))
    if x64.ndim == 1:
        x64 = x64[None, :]
    sel_rows = np.arange(n_out) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((x64.shape[0], sel_rows.size), dtype=np.float64)
    for r in np.unique(sel_rows // ROW_CHUNK):
        r0 = int(r) * ROW_CHUNK
        r1 = min(n_out, r0 + ROW_CHUNK)
        sel = np.nonzero(sel_rows // ROW_CHUNK == r)[0]
        deq = np.abs(dequantize(f, row_slice(f, packed, n_out, n_in, r0, r1), r1 - r0, n_in))
        out[:, sel] = x64 @ deq[sel_rows[sel] - r0].T
    return out


def argmax_first(y: np.ndarray) -> np.ndarray:
    """Per token, the lowest index of the largest logit ([Issue] Phase 2a).  NaN never wins."""
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    yy = np.where(np.isnan(y), -np.inf, y)
    return np.argmax(yy, axis=1).astype(np.int32)


def top2_gap(y: np.ndarray) -> np.ndarray:
    """Per token, largest minus second-largest logit (absolute, logit units)."""
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    if y.shape[1] < 2:
        return np.full(y.shape[0], np.inf)          # a single output: no runner-up
    part = -np.partition(-y, 1, axis=1)[:, :2]
    return part[:, 0] - part[:, 1]


def qgemv_argmax(fmt, packed, n_out, n_in, x):
    """The fused LM-head call: fp64 logits plus first-index argmax per token."""
    y = gemv(fmt, packed, n_out, n_in, x)
    return y, argmax_first(y)


# ----------------------------------------------------------------------------- draft vocabulary by id list

def gather_rows(fmt, packed: np.ndarray, n_out: int, n_in: int, ids) -> np.ndarray:
    """Canonical bytes of the small head made of rows ``ids`` (in that order).

    [M2Max] "MTP draft vocabulary subset": the draft head scores only the listed
    rows of the LM head, copied once into a small head.  Ids repeat freely; every
    id must lie in ``[0, n_out)``.
    """
    f = fmt_id(fmt)
    ids = np.asarray(ids, dtype=np.int64)
    if ids.size and (ids.min() < 0 or ids.max() >= n_out):
        raise IndexError("row id outside the head")
    if f == AFFINE4_G64:
        nw = n_out * n_in // 8
        ng = n_out * n_in // 64
        w = packed[: nw * 4].reshape(n_out, n_in // 2)[ids]
        s = packed[nw * 4: nw * 4 + ng * 2].reshape(n_out, n_in // 32)[ids]
        b = packed[nw * 4 + ng * 2:].reshape(n_out, n_in // 32)[ids]
        return np.concatenate([w.reshape(-1), s.reshape(-1), b.reshape(-1)])
    per_row = weight_bytes(f, 1, n_in)
    return np.ascontiguousarray(packed.reshape(n_out, per_row)[ids]).reshape(-1)


def qgemv_argmax_ids(fmt, packed, n_out, n_in, x, ids):
    """The draft head over an id list: fp64 logits of the small head (``[ntok, len(ids)]``,
    column j = row ``ids[j]``) and, per token, the full-vocabulary id of its first-index
    argmax, ``ids[j*]`` ([Issue] Phase 2b: a reduced draft vocabulary plus a d2t index
    mapping back to target ids).  Ties go to the lowest position j in the list."""
    ids = np.asarray(ids, dtype=np.int64)
    small = gather_rows(fmt, packed, n_out, n_in, ids)
    y = gemv(fmt, small, ids.size, n_in, x)
    j = argmax_first(y)
    return y, ids[j].astype(np.int32)


# ----------------------------------------------------------------------------- routed experts

MAX_GROUP_SLOTS = 4     # tokens per expert group: ne = 1..4


def expert_plan(ids, n_experts: int):
    """Group a step's routed (token, choice) pairs by expert ([Track2] section 1 item 2).

    ``ids[t, j]`` is the expert of token t's j-th choice; pair ``i = t * topk + j``.
    Reading of the plan: groups in increasing expert id; within a group the pairs in
    increasing i; an expert with more than four pairs (a token listing it twice, or
    more than four tokens) continues in the next group, four pairs at a time.  The
    pairs laid out group after group are the *slots*.

    Returns a dict of int arrays: ``group_start`` (n_groups + 1 entries, last =
    n_slots), ``group_expert``, ``slot_pair`` (the pair i held by each slot),
    ``slot_token`` (= slot_pair // topk) and ``pair_slot`` (the inverse of slot_pair).
    """
    ids = np.asarray(ids)
    if ids.ndim != 2 or ids.size == 0:
        raise ValueError("ids must be [ntok, topk]")
    topk = ids.shape[1]
    flat = [int(v) for v in ids.reshape(-1)]
    if any(not 0 <= e < n_experts for e in flat):
        raise ValueError("expert id out of range")
    group_start, group_expert, slot_pair = [], [], []
    for e in range(n_experts):
        pairs = [i for i, v in enumerate(flat) if v == e]
        for c in range(0, len(pairs), MAX_GROUP_SLOTS):
            group_start.append(len(slot_pair))
            group_expert.append(e)
            slot_pair.extend(pairs[c:c + MAX_GROUP_SLOTS])
    group_start.append(len(slot_pair))
    pair_slot = [0] * len(flat)
    for s, i in enumerate(slot_pair):
        pair_slot[i] = s
    return {"group_start": np.array(group_start, dtype=np.int64),
            "group_expert": np.array(group_expert, dtype=np.int64),
            "slot_pair": np.array(slot_pair, dtype=np.int64),
            "slot_token": np.array(slot_pair, dtype=np.int64) // topk,
            "pair_slot": np.array(pair_slot, dtype=np.int64)}


def experts_gemv_slots(fmt, packed, n_experts: int, n_out: int, n_in: int, x, plan, x_by_slot: bool):
    """The expert-grouped mat-vec over a plan's slots: fp64 ``y[s, o]`` for slot s of
    group g = ``deq(W_e)[o] . x_row(s)`` with e = group_expert[g] and x_row(s) =
    ``x[slot_token[s]]`` (the gate / up projection reads the step's token rows) or
    ``x[s]`` (the down projection reads one activation row per slot).  [Track2]
    section 1 item 2."""
    starts = [int(v) for v in plan["group_start"]]
    n_slots = starts[-1]
    y = np.empty((n_slots, n_out))
    for g, e in enumerate(plan["group_expert"]):
        slots = list(range(starts[g], starts[g + 1]))
        rows = slots if x_by_slot else [int(plan["slot_token"][s]) for s in slots]
        y[slots] = experts_gemv(fmt, packed, n_experts, n_out, n_in, x, [e], [rows])[0, :len(slots)]
    return y


def silu(v):
    """v * sigmoid(v) = v / (1 + exp(-v)), fp64."""
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def swiglu_rows(y):
    """The gated activation of an interleaved gate / up projection: for rows
    ``y[..., 2j]`` (gate j) and ``y[..., 2j + 1]`` (up j), ``silu(gate) * up`` ([Track2]
    section 1 item 2: ``moe_gu`` computes a group's gate and up projections together;
    reading: the activation is SiLU-gated, the form of a gate / up pair)."""
    y = np.asarray(y, dtype=np.float64)
    return silu(y[..., 0::2]) * y[..., 1::2]


def experts_gemv(fmt, packed, n_experts: int, n_out: int, n_in: int, x, group_expert, group_tokens):
    """Expert-grouped multi-token mat-vec.

    [Track2] section 1 item 2 (``moe_plan`` groups the tokens by expert id; ``moe_gu`` /
    ``moe_down`` then run each group with its own token count ne = 1..4, reading each
    unique expert's weights once).  ``packed`` holds the experts' matrices stacked
    (expert e = rows ``[e * n_out, (e + 1) * n_out)``); group g multiplies expert
    ``group_expert[g]`` by the tokens ``group_tokens[g]`` (1..4 indices into x).
    Returns fp64 ``y[g, k, o]`` for the k-th token of group g (``[n_groups, 4, n_out]``;
    slots k >= ne are NaN).
    """
    f = fmt_id(fmt)
    x = np.asarray(x, dtype=np.float32)
    ng = len(group_expert)
    y = np.full((ng, 4, n_out), np.nan)
    for g in range(ng):
        e = int(group_expert[g])
        toks = [int(t) for t in group_tokens[g]]
        if not 0 <= e < n_experts or not 1 <= len(toks) <= 4:
            raise ValueError("bad group")
        sub = row_slice(f, packed, n_experts * n_out, n_in, e * n_out, (e + 1) * n_out)
        y[g, :len(toks)] = gemv(f, sub, n_out, n_in, x[toks])
    return y

