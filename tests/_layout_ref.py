"""Test-side reader of the library's device layout, written from the layout
description in include/qgemv.h (not from the library's code): decodes packed
bytes back to fp64 weights so tests can check the packer's device layout.

Device layout: rows one after the other; a row is a run of steps, each step
512 bytes of codes followed by the scales of those codes, padded to 16 bytes.
Codes: Q8_0 q+128; Q4_0 / Q5_0 (low nibbles) / affine uint32 words of 8
consecutive elements (element k at bits 4k); BF16 raw.  Scales: Q8_0 / Q4_0 fp16 d
per 32 weights; affine (fp16 s, fp16 b) per 64 weights; Q5_0 (uint32 fifth bits,
fp16 d) per 32 weights, the fifth bit of element e at bit 8b + g with
g = 2 (e // 8) + e % 2 and b = (e % 8) // 2.
"""
from __future__ import annotations

import numpy as np

STEP = 512


def codes_bytes(fmt, n_in):
    return {"q8_0": n_in, "q4_0": n_in // 2, "affine4_g64": n_in // 2, "bf16": 2 * n_in, "q5_0": n_in // 2}[fmt]


def scale_bytes_for(fmt, codes):
    return {"q8_0": codes // 16, "q4_0": codes // 8, "affine4_g64": codes // 8, "bf16": 0,
            "q5_0": codes // 16 * 6}[fmt]


def r16(b):
    return (b + 15) // 16 * 16


def row_stride(fmt, n_in):
    c = codes_bytes(fmt, n_in)
    steps = (c + STEP - 1) // STEP
    last = c - STEP * (steps - 1)
    return (steps - 1) * (STEP + scale_bytes_for(fmt, STEP)) + r16(last + scale_bytes_for(fmt, last))


def split_row(fmt, row, n_in):
    """(codes, scales) of one packed row."""
    c = codes_bytes(fmt, n_in)
    full = STEP + scale_bytes_for(fmt, STEP)
    codes, scales = [], []
    k = 0
    while k * STEP < c:
        ck = min(STEP, c - k * STEP)
        base = k * full
        codes.append(row[base: base + ck])
        scales.append(row[base + ck: base + ck + scale_bytes_for(fmt, ck)])
        k += 1
    return np.concatenate(codes), np.concatenate(scales)


def decode_device(fmt: str, packed: np.ndarray, n_out: int, n_in: int) -> np.ndarray:
    st = row_stride(fmt, n_in)
    rows = np.asarray(packed, dtype=np.uint8)[: n_out * st].reshape(n_out, st)
    out = np.empty((n_out, n_in), dtype=np.float64)
    for r in range(n_out):
        codes, scales = split_row(fmt, rows[r], n_in)
        if fmt == "q8_0":
            q = codes.astype(np.int64) - 128
            d = scales.copy().view("<f2").astype(np.float64)
            out[r] = (q.reshape(-1, 32) * d[:, None]).reshape(-1)
        elif fmt in ("q4_0", "affine4_g64", "q5_0"):
            words = codes.copy().view("<u4")
            q = np.stack([(words >> np.uint32(4 * k)) & np.uint32(15) for k in range(8)], axis=1).reshape(-1)
            if fmt == "q5_0":
                rec = scales.reshape(-1, 6)
                qh = rec[:, :4].copy().view("<u4").reshape(-1)
                d = rec[:, 4:].copy().view("<f2").astype(np.float64).reshape(-1)
                # fifth bit of element e at bit 8b + g, g = 2 (e // 8) + e % 2, b = (e % 8) // 2
                e = np.arange(32)
                pos = 8 * ((e & 7) >> 1) + 2 * (e >> 3) + (e & 1)
                hb = (qh[:, None] >> pos.astype(np.uint32)) & np.uint32(1)
                q5 = (q.reshape(-1, 32) | (hb << np.uint32(4))).astype(np.float64)
                out[r] = ((q5 - 16) * d[:, None]).reshape(-1)
                continue
            q = q.astype(np.float64)
            if fmt == "q4_0":
                d = scales.copy().view("<f2").astype(np.float64)
                out[r] = ((q.reshape(-1, 32) - 8) * d[:, None]).reshape(-1)
            else:
                sb = scales.copy().view("<f2").astype(np.float64).reshape(-1, 2)
                out[r] = (q.reshape(-1, 64) * sb[:, 0:1] + sb[:, 1:2]).reshape(-1)
        elif fmt == "bf16":
            b = codes.copy().view("<u2").astype(np.uint32) << 16
            out[r] = b.view(np.float32).astype(np.float64)
    return out
