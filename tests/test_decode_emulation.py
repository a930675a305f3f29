"""The kernels' in-register decode, emulated bit for bit on the CPU (no GPU): for every
format, the packer's device bytes are turned into fp32 values the way the kernels do
it — a code placed in the mantissa of the magic float 2^23 (byte permute or nibble
mask), the offset removed by one fp32 subtraction, Q5_0's fifth bit merged from the
rotated record word, BF16 widened by a shift — and scaled by the block scale.  Every
value must equal the oracle's fp64 dequantization exactly: this pins the claim that
the decode is exact and that the kernels' view of the device layout matches the
packer's, before any GPU run.  The magic constants are restated here from the
decode's arithmetic (2^23 = 8388608), not taken from the kernel sources."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as ORC
import workloads
import block_quantized_token_format_gb300 as qg
from _layout_ref import split_row, row_stride

MAGIC = np.uint32(0x4B000000)          # bits of 2^23
TWO23 = np.float32(8388608.0)


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def _rotr(v, s):
    v = v.astype(np.uint64)
    return (((v >> np.uint64(s)) | (v << np.uint64(32 - s))) & np.uint64(0xFFFFFFFF)).astype(np.uint32) if s else \
        v.astype(np.uint32)


def emulate_row(fmt, codes, scales, n_in):
    """fp64 weights of one row from its device codes and scales, kernel-style."""
    if fmt == "bf16":
        w = codes.copy().view("<u4")
        lo = (w << np.uint32(16)).astype(np.uint32)            # element 2k
        hi = (w & np.uint32(0xFFFF0000)).astype(np.uint32)     # element 2k + 1
        return np.stack([_f32(lo), _f32(hi)], axis=1).reshape(-1).astype(np.float64)
    if fmt == "q8_0":
        f = _f32(MAGIC | codes.astype(np.uint32)) - (TWO23 + np.float32(128))   # q, exact
        d = scales.copy().view("<f2").astype(np.float32)
        return (f.reshape(-1, 32) * d[:, None]).reshape(-1).astype(np.float64)
    words = codes.copy().view("<u4").reshape(-1, 4)            # one 16-byte lane chunk per row
    out = np.empty((words.shape[0], 32), dtype=np.float64)
    if fmt == "q5_0":
        rec = scales.reshape(-1, 6)
        qh = rec[:, :4].copy().view("<u4").reshape(-1)
        d5 = rec[:, 4:].copy().view("<f2").astype(np.float64).reshape(-1)
    for i in range(8):                                         # 4 columns per step of i
        w = words[:, i >> 1]
        h = (w >> np.uint32(16)) if (i & 1) else w
        rot = _rotr(qh, i if i < 4 else i + 12) if fmt == "q5_0" else None
        for m in range(4):
            bits = (h & np.uint32(0xF << (4 * m))) | MAGIC     # 2^23 + nibble * 16^m
            if fmt == "q5_0":
                bits = bits | (rot & np.uint32(0x10 << (4 * m)))
            off = {"q4_0": 8, "q5_0": 16, "affine4_g64": 0}[fmt]
            f = _f32(bits) - np.float32(8388608.0 + off * 16.0 ** m)   # (q - off) * 16^m, exact
            out[:, 4 * i + m] = f.astype(np.float64) / 16.0 ** m       # the kernel pre-scales x by 16^-m
    q = out.reshape(-1)
    if fmt == "q4_0":
        d = scales.copy().view("<f2").astype(np.float64)
        return (q.reshape(-1, 32) * d[:, None]).reshape(-1)
    if fmt == "q5_0":
        return (q.reshape(-1, 32) * d5[:, None]).reshape(-1)
    sb = scales.copy().view("<f2").astype(np.float64).reshape(-1, 2)
    return (q.reshape(-1, 64) * sb[:, 0:1] + sb[:, 1:2]).reshape(-1)


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


def test_q5_0_rotation_covers_every_bit_once():
    """The rotated record places the 32 fifth bits at 32 distinct positions."""
    e = np.arange(32)
    i, m = e >> 2, e & 3
    pos = (4 * m + 4 + np.where(i < 4, i, i + 12)) % 32
    assert sorted(pos.tolist()) == list(range(32))
