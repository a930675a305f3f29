"""The kernels' in-register decode, emulated bit for bit on the CPU (no GPU): for every
format, the packer's device bytes are turned into values the way the kernels do it —
BF16 widened by a shift; for the integer chunk dot, Q8_0's bytes q + 128 as they are
(the offset removed through the chunk's starting sum) and a Q4_0 / Q5_0 / affine word's
even and odd codes taken as bytes (one mask, one shift and mask, Q5_0's fifth bits
merged from its record) — and scaled by the block scale.  Every value must equal the oracle's fp64
dequantization exactly: this pins the claim that the decode is exact and that the
kernels' view of the device layout matches the packer's, before any GPU run.  The
rule is restated here from the layout description, not taken from the kernel sources.

The integer chunk dot also rounds x: per 32-column chunk and token, X = rn(x * 2^(15-k))
capped at 32767, with 2^(k-1) <= max|x| < 2^k.  test_x_rounding_bound pins the stated bound
of that rounding (X fits int16, |x - X * 2^(k-15)| <= 2^-14 max|x|, the chunk sums of X
against 4-bit codes exact in int32 and in their I2F) on random and adversarial chunks,
written from the rule."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as ORC
import workloads
import block_quantized_token_format_gb300 as qg
from _layout_ref import split_row, row_stride

def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def emulate_row(fmt, codes, scales, n_in):
    """fp64 weights of one row from its device codes and scales, kernel-style."""
    if fmt == "bf16":
        w = codes.copy().view("<u4")
        lo = (w << np.uint32(16)).astype(np.uint32)            # element 2k
        hi = (w & np.uint32(0xFFFF0000)).astype(np.uint32)     # element 2k + 1
        return np.stack([_f32(lo), _f32(hi)], axis=1).reshape(-1).astype(np.float64)
    if fmt == "q8_0":
        # integer chunk dot: the byte u = q + 128 enters dp2a as it is; the chunk's
        # starting sum -128 * sum(X) removes the offset, so the code is u - 128, exact
        q = codes.astype(np.int64) - 128
        d = scales.copy().view("<f2").astype(np.float64)
        return (q.reshape(-1, 32) * d[:, None]).reshape(-1).astype(np.float64)
    words = codes.copy().view("<u4").reshape(-1, 4)            # one 16-byte lane chunk per row
    if fmt in ("q4_0", "affine4_g64", "q5_0"):
        return emulate_bytes(fmt, words, scales)
    raise ValueError(fmt)


def _shift(v, s):
    """v << s for s >= 0, v >> -s otherwise (uint32)."""
    v = v.astype(np.uint64)
    r = (v << np.uint64(s)) if s >= 0 else (v >> np.uint64(-s))
    return (r & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def emulate_bytes(fmt, words, scales):
    """Q4_0 / Q5_0 / affine: word w of a lane chunk gives its even codes as the 4 bytes of
    w & 0x0F0F0F0F and its odd codes as those of (w >> 4) & 0x0F0F0F0F; Q5_0 ORs in the
    fifth bits of group g = 2j (even) or 2j + 1 (odd) as (record << (4 - g)) & 0x10101010;
    byte b of the even word is element 2b, of the odd word element 2b + 1."""
    q = np.empty((words.shape[0], 32), dtype=np.float64)
    if fmt == "q5_0":
        rec = scales.reshape(-1, 6)
        qh = rec[:, :4].copy().view("<u4").reshape(-1)
    for j in range(4):
        w = words[:, j]
        ev = w & np.uint32(0x0F0F0F0F)
        od = (w >> np.uint32(4)) & np.uint32(0x0F0F0F0F)
        if fmt == "q5_0":
            ev = ev | (_shift(qh, 4 - 2 * j) & np.uint32(0x10101010))
            od = od | (_shift(qh, 4 - (2 * j + 1)) & np.uint32(0x10101010))
        for b in range(4):
            q[:, 8 * j + 2 * b] = ((ev >> np.uint32(8 * b)) & np.uint32(0xFF)).astype(np.float64)
            q[:, 8 * j + 2 * b + 1] = ((od >> np.uint32(8 * b)) & np.uint32(0xFF)).astype(np.float64)
    q = q.reshape(-1)
    if fmt == "q4_0":
        d = scales.copy().view("<f2").astype(np.float64)
        return ((q.reshape(-1, 32) - 8) * d[:, None]).reshape(-1)
    if fmt == "q5_0":
        d5 = scales.reshape(-1, 6)[:, 4:].copy().view("<f2").astype(np.float64).reshape(-1)
        return ((q.reshape(-1, 32) - 16) * d5[:, None]).reshape(-1)
    sb = scales.copy().view("<f2").astype(np.float64).reshape(-1, 2)
    return (q.reshape(-1, 64) * sb[:, 0:1] + sb[:, 1:2]).reshape(-1)


def _round_chunk(x):
    """The staging rule for one chunk of fp32 x: (X, 2^(k-15)), or zeros for a chunk whose
    largest |x| is below 2^-112."""
    x = np.asarray(x, dtype=np.float32)
    m = np.float32(np.max(np.abs(x)))
    e = int(m.view(np.uint32) >> 23)
    if e < 15:
        return np.zeros(x.shape, dtype=np.int64), 0.0
    k = e - 126
    X = np.rint(x.astype(np.float64) * 2.0 ** (15 - k)).astype(np.int64)     # round half even
    return np.minimum(X, 32767), 2.0 ** (k - 15)


def test_x_rounding_bound():
    rng = np.random.default_rng(5)
    chunks = [rng.standard_normal(32).astype(np.float32) for _ in range(2000)]
    chunks += [np.float32(2.0) ** rng.integers(-60, 60) * rng.standard_normal(32).astype(np.float32)
               for _ in range(500)]
    ch = rng.standard_normal(32).astype(np.float32) * np.float32(1e-3)
    ch[7] = np.float32(1000.0)                                  # one outlier per chunk
    chunks.append(ch)
    chunks.append(np.full(32, np.float32(np.nextafter(np.float32(4.0), np.float32(0)))))   # max just below 2^k
    chunks.append(np.full(32, np.float32(-4.0)))                                             # max exactly 2^(k-1)
    chunks.append(np.zeros(32, dtype=np.float32))
    chunks.append(np.full(32, np.float32(1e-35)))                                            # below 2^-112: zero
    chunks.append(np.full(32, np.float32(2.0 ** -112)))                                       # the smallest live max
    top = np.float32(np.nextafter(np.float32(8.0), np.float32(0)))
    chunks.append(np.array([top, -top] * 16, dtype=np.float32))                              # rounds to +-2^15: capped
    for x in chunks:
        X, scale = _round_chunk(x)
        m = float(np.max(np.abs(x.astype(np.float64))))
        assert np.all(X >= -2 ** 15) and np.all(X <= 2 ** 15 - 1)
        err = np.abs(x.astype(np.float64) - X * scale)
        assert np.all(err <= 2.0 ** -14 * m + (m if scale == 0.0 else 0.0)), (float(err.max()), m)
        if scale == 0.0:
            assert m < 2.0 ** -112
        # chunk sums against 4-bit codes are exact in int32 and in the I2F to fp32
        s = int(np.sum(15 * np.abs(X)))
        assert s < 2 ** 24 and float(np.float32(s)) == s


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"])
@pytest.mark.parametrize("n_in", [64, 1088, 2560 + 320])
def test_kernel_decode_is_exact(fmt, n_in):
    n_out = 6
    W = workloads.gaussian(404 + n_in, (n_out, n_in), 0.02)
    W[0] = 0.0
    W[1, ::3] = np.float32(0.7)                 # large codes and ties of magnitude
    W[2] = -np.abs(W[2])                        # one-signed rows: Q4_0 / Q5_0 extremes
    canon = ORC.quantize(fmt, W)
    ref = ORC.dequantize(fmt, canon, n_out, n_in)
    packed = qg.qg_to_device_layout(fmt, canon, n_out, n_in)
    st = row_stride(fmt, n_in)
    for r in range(n_out):
        codes, scales = split_row(fmt, packed[r * st:(r + 1) * st], n_in)
        got = emulate_row(fmt, codes, scales, n_in)
        assert np.array_equal(got, ref[r]), (fmt, n_in, r, int(np.argmax(got != ref[r])))


def test_q5_0_record_order_covers_every_bit_once():
    """The record places the 32 fifth bits at 32 distinct positions, and group g's bits
    land at bit 4 of its 4 code bytes after the shift by 4 - g."""
    e = np.arange(32)
    g = 2 * (e >> 3) + (e & 1)
    b = (e & 7) >> 1
    pos = 8 * b + g
    assert sorted(pos.tolist()) == list(range(32))
    assert np.all(pos + (4 - g) == 8 * b + 4)
