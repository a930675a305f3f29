"""Test-side reader of the library's device layout, written from the layout
description in include/qgemv.h (not from the library's code): decodes packed
bytes back to fp64 weights so tests can check the packer's device layout."""
from __future__ import annotations

import numpy as np


def row_stride(fmt: str, n_in: int) -> int:
    raw = {"q8_0": n_in + n_in // 32 * 2, "q4_0": n_in // 2 + n_in // 32 * 2,
           "affine4_g64": n_in // 2 + n_in // 64 * 4, "bf16": 2 * n_in}[fmt]
    return (raw + 15) // 16 * 16


def decode_device(fmt: str, packed: np.ndarray, n_out: int, n_in: int) -> np.ndarray:
    st = row_stride(fmt, n_in)
    rows = np.asarray(packed, dtype=np.uint8)[: n_out * st].reshape(n_out, st)
    f16 = lambda b: b.copy().view("<f2").astype(np.float64)
    if fmt == "q8_0":
        q = rows[:, :n_in].astype(np.int64) - 128
        d = f16(rows[:, n_in:n_in + n_in // 16])
        return (q.reshape(n_out, -1, 32) * d[..., None]).reshape(n_out, n_in)
    if fmt in ("q4_0", "affine4_g64"):
        words = rows[:, : n_in // 2].copy().view("<u4")
        q = np.stack([(words >> np.uint32(4 * k)) & np.uint32(15) for k in range(8)], axis=2).reshape(n_out, n_in)
        q = q.astype(np.float64)
        if fmt == "q4_0":
            d = f16(rows[:, n_in // 2: n_in // 2 + n_in // 16])
            return ((q.reshape(n_out, -1, 32) - 8) * d[..., None]).reshape(n_out, n_in)
        sb = rows[:, n_in // 2: n_in // 2 + n_in // 16].copy().view("<f2").astype(np.float64).reshape(n_out, -1, 2)
        return (q.reshape(n_out, -1, 64) * sb[..., 0:1] + sb[..., 1:2]).reshape(n_out, n_in)
    if fmt == "bf16":
        b = rows[:, : 2 * n_in].copy().view("<u2").astype(np.uint32) << 16
        return b.view(np.float32).astype(np.float64)
    raise ValueError(fmt)
