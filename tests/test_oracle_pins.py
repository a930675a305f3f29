"""Pins of the CPU oracle to facts outside itself (no GPU).

Each check is written as a plain function ``check_*(orc)`` taking the oracle
module, so ``test_oracle_mutations.py`` can run the same checks against an
oracle with a planted mistake and show that they fail.

What pins what:
* byte counts          <- times and GB/s printed on the pages (golden rows)
* dequantizers         <- hand-built blocks with exact values (golden blocks)
* quantizers           <- the same blocks round-tripped, half-away rounding blocks,
                          idempotence on random blocks, error band on Gaussian W
* the mat-vec          <- exact rational brute force from the raw bytes through an
                          independent decoder; linearity; token independence;
                          cross-format identities
* argmax               <- planted maxima and ties
"""
from __future__ import annotations

import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle as ORC
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- independent decoder
# A second decoder in pure Python with exact rationals, reading the raw bytes with
# struct and decoding fp16 / bf16 from their IEEE bit fields.  It shares nothing
# with the numpy oracle.

def _f16(bits: int) -> Fraction:
    s, e, m = (bits >> 15) & 1, (bits >> 10) & 0x1F, bits & 0x3FF
    assert e != 31
    v = Fraction(m, 1 << 24) if e == 0 else Fraction(1024 + m, 1024) * Fraction(2) ** (e - 15)
    return -v if s else v


def _bf16(bits: int) -> Fraction:
    s, e, m = (bits >> 15) & 1, (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 255
    v = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else Fraction(128 + m, 128) * Fraction(2) ** (e - 127)
    return -v if s else v


def brute_decode(fmt: int, raw: bytes, n_out: int, n_in: int):
    """Exact dequantized matrix as nested lists of Fractions."""
    W = [[Fraction(0)] * n_in for _ in range(n_out)]
    if fmt == ORC.Q8_0:
        nb = n_in // 32
        for r in range(n_out):
            for b in range(nb):
                off = (r * nb + b) * 34
                d = _f16(struct.unpack_from("<H", raw, off)[0])
                qs = struct.unpack_from("<32b", raw, off + 2)
                for j in range(32):
                    W[r][32 * b + j] = qs[j] * d
    elif fmt == ORC.Q4_0:
        nb = n_in // 32
        for r in range(n_out):
            for b in range(nb):
                off = (r * nb + b) * 18
                d = _f16(struct.unpack_from("<H", raw, off)[0])
                qs = struct.unpack_from("<16B", raw, off + 2)
                for j in range(16):
                    W[r][32 * b + j] = ((qs[j] & 15) - 8) * d
                    W[r][32 * b + j + 16] = ((qs[j] >> 4) - 8) * d
    elif fmt == ORC.AFFINE4_G64:
        nw, ng = n_out * n_in // 8, n_out * n_in // 64
        words = struct.unpack_from(f"<{nw}I", raw, 0)
        sc = struct.unpack_from(f"<{ng}H", raw, 4 * nw)
        bi = struct.unpack_from(f"<{ng}H", raw, 4 * nw + 2 * ng)
        for r in range(n_out):
            for i in range(n_in):
                w = words[r * (n_in // 8) + i // 8]
                q = (w >> (4 * (i % 8))) & 15
                g = r * (n_in // 64) + i // 64
                W[r][i] = q * _f16(sc[g]) + _f16(bi[g])
    elif fmt == ORC.Q5_0:
        nb = n_in // 32
        for r in range(n_out):
            for b in range(nb):
                off = (r * nb + b) * 22
                d = _f16(struct.unpack_from("<H", raw, off)[0])
                qh = struct.unpack_from("<I", raw, off + 2)[0]
                qs = struct.unpack_from("<16B", raw, off + 6)
                for j in range(16):
                    lo0, lo1 = qs[j] & 15, qs[j] >> 4
                    W[r][32 * b + j] = ((lo0 | (((qh >> j) & 1) << 4)) - 16) * d
                    W[r][32 * b + j + 16] = ((lo1 | (((qh >> (j + 16)) & 1) << 4)) - 16) * d
    elif fmt == ORC.BF16:
        vals = struct.unpack_from(f"<{n_out * n_in}H", raw, 0)
        for r in range(n_out):
            for i in range(n_in):
                W[r][i] = _bf16(vals[r * n_in + i])
    else:
        raise ValueError(fmt)
    return W


def brute_gemv(Wq, x):
    xs = [[Fraction(float(v)) for v in row] for row in np.atleast_2d(x)]
    return [[sum(w * xv for w, xv in zip(row, xt)) for row in Wq] for xt in xs]


# ----------------------------------------------------------------------------- checks

def check_page_byte_counts(orc):
    g = _load("page_bandwidth_rows.json")
    for row in g["rows"]:
        nbytes = orc.weight_bytes(row["fmt"], row["n_out"], row["n_in"])
        gbs = nbytes / (row["us"] * 1e-6) / 1e9
        assert abs(gbs - row["gbs"]) <= 0.12, (row, gbs)
    h = g["affine4_head"]
    total = orc.weight_bytes(h["fmt"], h["n_out"], h["n_in"])
    assert round(total / 1e6, 1) == h["total_mb"]
    # plane sizes of the canonical layout, measured on a small matrix and scaled
    n_out, n_in = 4, 5120
    raw = orc.quantize(h["fmt"], workloads.gaussian(5, (n_out, n_in), 0.02))
    assert raw.size == orc.weight_bytes(h["fmt"], n_out, n_in)
    scale = h["n_out"] / n_out
    assert round(n_out * n_in / 2 * scale / 1e6, 1) == h["weight_mb"]
    assert round(n_out * n_in / 64 * 2 * scale / 1e6, 1) == h["scales_mb"] == h["biases_mb"]


def check_golden_q8_0(orc):
    g = _load("q8_0_block.json")
    raw = np.array(g["bytes"], dtype=np.uint8)
    assert raw.size == 34 and len(g["q"]) == 32
    deq = orc.dequantize("q8_0", raw, 1, 32)
    assert np.array_equal(deq[0], np.array(g["values"], dtype=np.float64))
    back = orc.quantize("q8_0", np.array([g["values"]], dtype=np.float32))
    assert np.array_equal(back, raw)
    y = orc.gemv("q8_0", raw, 1, 32, np.ones((1, 32), np.float32))
    assert y[0, 0] == g["dot_with_ones"]


def check_golden_q4_0(orc):
    g = _load("q4_0_block.json")
    raw = np.array(g["bytes"], dtype=np.uint8)
    assert raw.size == 18
    deq = orc.dequantize("q4_0", raw, 1, 32)
    assert np.array_equal(deq[0], np.array(g["values"], dtype=np.float64))
    back = orc.quantize("q4_0", np.array([g["values"]], dtype=np.float32))
    assert np.array_equal(back, raw)


def check_golden_q5_0(orc):
    g = _load("q5_0_block.json")
    raw = np.array(g["bytes"], dtype=np.uint8)
    assert raw.size == 22
    deq = orc.dequantize("q5_0", raw, 1, 32)
    assert np.array_equal(deq[0], np.array(g["values"], dtype=np.float64))
    back = orc.quantize("q5_0", np.array([g["values"]], dtype=np.float32))
    assert np.array_equal(back, raw)
    # half away from zero: m = -4 gives d = 0.25; w = 0.625 is 2.5 d -> q = 3 + 16 = 19
    w = np.zeros((1, 32), np.float32)
    w[0, 0], w[0, 5] = -4.0, 0.625
    deq = orc.dequantize("q5_0", orc.quantize("q5_0", w), 1, 32)
    assert deq[0, 5] == 0.75 and deq[0, 0] == -4.0
    # an all-zero block: d = 0 / -16 = -0 (fp16 0x8000), every code 16 (bit 4 set, low nibble 0)
    z = orc.quantize("q5_0", np.zeros((1, 32), np.float32))
    assert list(z[:6]) == [0x00, 0x80, 0xFF, 0xFF, 0xFF, 0xFF] and all(b == 0 for b in z[6:])
    assert not orc.dequantize("q5_0", z, 1, 32).any()


def check_golden_affine4(orc):
    g = _load("affine4_group.json")
    words = np.array([int(w, 16) for w in g["words"]], dtype="<u4")
    raw = np.concatenate([words.view(np.uint8),
                          np.array([int(g["scale_bits"], 16)], "<u2").view(np.uint8),
                          np.array([int(g["bias_bits"], 16)], "<u2").view(np.uint8)])
    expect = np.array(g["q"], dtype=np.float64) * g["s"] + g["b"]
    deq = orc.dequantize("affine4_g64", raw, 1, 64)
    assert np.array_equal(deq[0], expect)
    back = orc.quantize("affine4_g64", expect[None, :].astype(np.float32))
    assert np.array_equal(back, raw)


def check_golden_bf16(orc):
    g = _load("bf16_values.json")
    bits = np.array([int(b, 16) for b in g["bits"]], dtype="<u2")
    deq = orc.dequantize("bf16", bits.view(np.uint8), 1, bits.size)
    assert np.array_equal(deq[0], np.array(g["values"], dtype=np.float64))
    assert np.array_equal(np.signbit(deq[0]), np.signbit(np.array(g["values"])))
    back = orc.quantize("bf16", np.array([g["values"]], dtype=np.float32))
    assert np.array_equal(back, bits.view(np.uint8))
    row = np.array([int(b, 16) for b in g["dot_row_bits"]], dtype="<u2").view(np.uint8)
    y = orc.gemv("bf16", row, 1, 8, np.array([g["dot_x"]], np.float32))
    assert y[0, 0] == g["dot_value"]


def check_rounding(orc):
    g = _load("rounding_blocks.json")
    # Q8_0
    w = np.zeros((1, 32), np.float32)
    w[0, :len(g["q8_0"]["w_first"])] = g["q8_0"]["w_first"]
    raw = orc.quantize("q8_0", w)
    q = raw[2:34].view(np.int8)[: len(g["q8_0"]["q_first"])]
    assert list(q) == g["q8_0"]["q_first"]
    assert raw[0:2].view("<f2")[0] == g["q8_0"]["d"]
    # Q4_0
    w = np.zeros((1, 32), np.float32)
    w[0, :len(g["q4_0"]["w_first"])] = g["q4_0"]["w_first"]
    raw = orc.quantize("q4_0", w)
    codes = list(raw[2:18] & 15) + list(raw[2:18] >> 4)
    assert codes[: len(g["q4_0"]["q_first"])] == g["q4_0"]["q_first"]
    assert raw[0:2].view("<f2")[0] == g["q4_0"]["d"]
    # affine4
    w = np.zeros((1, 64), np.float32)
    w[0, :len(g["affine4_g64"]["w_first"])] = g["affine4_g64"]["w_first"]
    raw = orc.quantize("affine4_g64", w)
    words = raw[:32].view("<u4")
    codes = [int((words[i // 8] >> (4 * (i % 8))) & 15) for i in range(64)]
    assert codes[: len(g["affine4_g64"]["q_first"])] == g["affine4_g64"]["q_first"]
    assert raw[32:34].view("<f2")[0] == g["affine4_g64"]["s"]
    assert raw[34:36].view("<f2")[0] == g["affine4_g64"]["b"]


def check_brute_force(orc):
    """The fp64 mat-vec equals exact rational arithmetic from the raw bytes."""
    for fmt in ("q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"):
        f = orc.fmt_id(fmt)
        for n_out, n_in in ((1, 64), (3, 64), (7, 128)):
            W = workloads.gaussian(1000 + n_out + n_in + f, (n_out, n_in), 0.02)
            x = workloads.gaussian(2000 + n_out + n_in + f, (3, n_in))
            raw = orc.quantize(fmt, W)
            exact = brute_gemv(brute_decode(f, raw.tobytes(), n_out, n_in), x)
            y = orc.gemv(fmt, raw, n_out, n_in, x)
            for t in range(3):
                for o in range(n_out):
                    e = exact[t][o]
                    scale = max(abs(float(e)), 1e-30)
                    assert abs(y[t, o] - float(e)) <= 1e-15 * max(scale, 1e-3), (fmt, n_out, n_in, t, o)
            # and the oracle's dequantizer equals the exact decode, element by element
            deq = orc.dequantize(fmt, raw, n_out, n_in)
            ex = brute_decode(f, raw.tobytes(), n_out, n_in)
            assert all(deq[r, i] == float(ex[r][i]) for r in range(n_out) for i in range(n_in))


def check_idempotence(orc):
    """quantize(dequantize(B)) == B on random blocks (Q8_0, Q4_0, Q5_0)."""
    for fmt in ("q8_0", "q4_0", "q5_0"):
        W = workloads.gaussian(77, (64, 256), 0.02)
        raw = orc.quantize(fmt, W)
        deq = orc.dequantize(fmt, raw, 64, 256).astype(np.float32)
        assert np.array_equal(orc.quantize(fmt, deq), raw), fmt


def check_affine_constructed_roundtrip(orc):
    """Affine groups with power-of-two scale and bias = k * scale round-trip exactly."""
    rng = np.random.Generator(np.random.PCG64(5))
    n_out, n_in = 8, 256
    q = rng.integers(0, 16, (n_out, n_in // 64, 64))
    q[..., 0], q[..., 1] = 0, 15
    s = 2.0 ** -rng.integers(3, 9, (n_out, n_in // 64))
    b = -rng.integers(0, 9, (n_out, n_in // 64)) * s
    W = (q * s[..., None] + b[..., None]).reshape(n_out, n_in).astype(np.float32)
    raw = orc.quantize("affine4_g64", W)
    assert np.array_equal(orc.dequantize("affine4_g64", raw, n_out, n_in), W.astype(np.float64))


def check_linearity(orc):
    n_out, n_in = 16, 256
    # x1, x2 on a 2^-12 grid with |x| < 4: their sum is exact in fp32.
    rng = np.random.Generator(np.random.PCG64(9))
    x1 = (rng.integers(-16384, 16384, (2, n_in)) / 4096.0).astype(np.float32)
    x2 = (rng.integers(-16384, 16384, (2, n_in)) / 4096.0).astype(np.float32)
    for fmt in ("q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"):
        raw = orc.quantize(fmt, workloads.gaussian(11, (n_out, n_in), 0.02))
        y1 = orc.gemv(fmt, raw, n_out, n_in, x1)
        y2 = orc.gemv(fmt, raw, n_out, n_in, x2)
        y12 = orc.gemv(fmt, raw, n_out, n_in, (x1 + x2) * np.float32(0.5))
        den = orc.gemv_abs(fmt, raw, n_out, n_in, np.abs(x1) + np.abs(x2))
        assert np.all(np.abs(y12 - 0.5 * (y1 + y2)) <= 1e-13 * den + 1e-300), fmt


def check_token_independence(orc):
    n_out, n_in = 33, 512
    for fmt in ("q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"):
        raw = orc.quantize(fmt, workloads.gaussian(21, (n_out, n_in), 0.02))
        x4 = workloads.activations(21, n_in, 4)
        y4 = orc.gemv(fmt, raw, n_out, n_in, x4)
        for t in range(4):
            y1 = orc.gemv(fmt, raw, n_out, n_in, x4[t:t + 1])
            assert np.array_equal(y1[0], y4[t]), (fmt, t)
        same = orc.gemv(fmt, raw, n_out, n_in, np.repeat(x4[:1], 4, axis=0))
        assert all(np.array_equal(same[0], same[t]) for t in range(4))


def check_cross_format(orc):
    rng = np.random.Generator(np.random.PCG64(31))
    n_out, n_in = 12, 256
    x = workloads.gaussian(32, (4, n_in))
    # Q8_0 with d = 2^-k equals BF16 holding q * 2^-k.
    q = rng.integers(-127, 128, (n_out, n_in // 32, 32))
    q[..., 5] = 127
    k = rng.integers(4, 12, (n_out, n_in // 32))
    W = (q * 2.0 ** -k[..., None]).reshape(n_out, n_in).astype(np.float32)
    y8 = orc.gemv("q8_0", orc.quantize("q8_0", W), n_out, n_in, x)
    yb = orc.gemv("bf16", orc.quantize("bf16", W), n_out, n_in, x)
    assert np.array_equal(y8, yb)
    # Q4_0 with d = 2^-k equals affine4 with s = 2^-k, b = -8 * 2^-k on 64-groups.
    q = rng.integers(0, 16, (n_out, n_in // 64, 64))
    q[..., 0], q[..., 33], q[..., 40] = 0, 0, 15
    k = rng.integers(4, 10, (n_out, n_in // 64))
    W = ((q - 8) * 2.0 ** -k[..., None]).reshape(n_out, n_in).astype(np.float32)
    r4 = orc.quantize("q4_0", W)
    ra = orc.quantize("affine4_g64", W)
    assert np.array_equal(orc.dequantize("q4_0", r4, n_out, n_in), W.astype(np.float64))
    assert np.array_equal(orc.dequantize("affine4_g64", ra, n_out, n_in), W.astype(np.float64))
    assert np.array_equal(orc.gemv("q4_0", r4, n_out, n_in, x), orc.gemv("affine4_g64", ra, n_out, n_in, x))
    # Q4_0 code q with scale d equals Q5_0 code q + 8 with the same d: rebuild every Q4_0
    # block as a Q5_0 block by hand (fifth bit = bit 4 of q + 8) and compare.
    blocks = r4.reshape(-1, 18)
    q5 = bytearray()
    for blk in blocks:
        lo = [int(b) & 15 for b in blk[2:]] + [int(b) >> 4 for b in blk[2:]]      # elements 0..31
        c = [v + 8 for v in lo]
        qh = sum(((v >> 4) & 1) << j for j, v in enumerate(c))
        q5 += bytes(blk[:2]) + struct.pack("<I", qh) + bytes((c[j] & 15) | ((c[j + 16] & 15) << 4) for j in range(16))
    r5 = np.frombuffer(bytes(q5), dtype=np.uint8)
    assert np.array_equal(orc.dequantize("q5_0", r5, n_out, n_in), orc.dequantize("q4_0", r4, n_out, n_in))


def check_argmax(orc):
    n_out, n_in = 40, 256
    x = workloads.gaussian(41, (2, n_in))
    W = workloads.gaussian(42, (n_out, n_in), 0.02)
    W[17] = np.float32(0.05) * np.sign(x[0])        # planted unique max for token 0
    W[23] = np.float32(0.05) * np.sign(x[1])        # planted unique max for token 1
    raw = orc.quantize("q8_0", W)
    y, am = orc.qgemv_argmax("q8_0", raw, n_out, n_in, x)
    assert list(am) == [17, 23]
    # exact tie: two identical maximal rows -> the lower index
    W[30] = W[17]
    W[9] = W[17]
    raw = orc.quantize("q8_0", W)
    y, am = orc.qgemv_argmax("q8_0", raw, n_out, n_in, x)
    assert y[0, 9] == y[0, 17] == y[0, 30]
    assert am[0] == 9
    assert orc.argmax_first(np.array([[1.0, np.nan, 3.0, 3.0]]))[0] == 2
    assert orc.top2_gap(np.array([[1.0, 5.0, 4.5]]))[0] == 0.5
    assert orc.top2_gap(np.array([[2.0], [3.0]]))[1] == np.inf


def check_quant_error_band(orc):
    """GEMV rel-RMSE vs the fp32 weights on N(0, 0.02) W, N(0,1) x: same order as the
    0.58-1.18% (Q8_0), 4.4-5.6% (Q5_0) and 5.8-10.7% (Q4_0) that the opus-mtp-turbo
    report's item 3 table measures on real tensors, and Q5_0 between Q8_0 and Q4_0.
    A sanity band, not a parity check."""
    n_out, n_in = 256, 2560
    W = workloads.gaussian(51, (n_out, n_in), 0.02)
    x = workloads.gaussian(52, (8, n_in))
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    bands = {"q8_0": (0.003, 0.012), "q4_0": (0.04, 0.12), "affine4_g64": (0.04, 0.12), "bf16": (0.0005, 0.004),
             "q5_0": (0.02, 0.06)}
    rels = {}
    for fmt, (lo, hi) in bands.items():
        y = orc.gemv(fmt, orc.quantize(fmt, W), n_out, n_in, x)
        rel = np.sqrt(np.mean((y - ref) ** 2) / np.mean(ref ** 2))
        rels[fmt] = rel
        assert lo <= rel <= hi, (fmt, rel)
    assert rels["q8_0"] < rels["q5_0"] < rels["q4_0"]
    assert 1.6 < rels["q4_0"] / rels["q5_0"] < 2.4          # one more bit: about half the error


def check_fp16_bf16_rounding(orc):
    """The fp16 / bf16 conversions the quantizers use round to nearest even (IEEE values)."""
    cases = {0.1: 0x2E66, 1 / 3: 0x3555, 65504.0: 0x7BFF, 65519.0: 0x7BFF, 65520.0: 0x7C00,
             2.0 ** -24: 0x0001, 1.5 * 2.0 ** -25: 0x0001, 2.0 ** -25: 0x0000, 2.0 ** -14: 0x0400}
    with np.errstate(over="ignore"):
        for v, bits in cases.items():
            assert int(np.array([v], np.float32).astype(np.float16).view(np.uint16)[0]) == bits, v
    b = orc.f32_to_bf16_bits(np.array([1.00390625, 1.01171875, -1.00390625, 3.0], np.float32))
    assert list(b) == [0x3F80, 0x3F82, 0xBF80, 0x4040]
    r = orc.round_half_away(np.array([0.5, 1.5, 2.5, -0.5, -2.5, np.nextafter(np.float32(0.5), 0),
                                       8388607.5, -3.2], np.float32))
    assert list(r) == [1, 2, 3, -1, -3, 0, 8388608, -3]


def check_draft_ids(orc):
    """The draft head over an id list ([M2Max] "MTP draft vocabulary subset": the listed
    rows copied once into a small head; [Issue] Phase 2b: the d2t map back to full ids)."""
    n_out, n_in = 50, 128
    x = workloads.gaussian(71, (2, n_in))
    W = workloads.gaussian(72, (n_out, n_in), 0.02)
    W[31] = np.float32(0.05) * np.sign(x[0])        # token 0's maximum, in the list
    W[44] = np.float32(0.06) * np.sign(x[1])        # token 1's overall maximum, NOT in the list
    W[12] = np.float32(0.04) * np.sign(x[1])        # token 1's maximum within the list
    ids = np.array([40, 31, 3, 12, 7, 31, 0], dtype=np.int32)   # unsorted, with a repeat
    for fmt in ("q8_0", "q4_0", "affine4_g64", "bf16"):
        raw = orc.quantize(fmt, W)
        full = orc.gemv(fmt, raw, n_out, n_in, x)
        y, am = orc.qgemv_argmax_ids(fmt, raw, n_out, n_in, x, ids)
        assert y.shape == (2, ids.size)
        assert np.allclose(y, full[:, ids], rtol=1e-13, atol=1e-15), fmt    # column j is row ids[j]
        assert list(am) == [31, 12], (fmt, list(am))                        # mapped back to full ids
        # the gathered bytes decode to exactly the listed rows, in list order
        deq = orc.dequantize(fmt, orc.gather_rows(fmt, raw, n_out, n_in, ids), ids.size, n_in)
        assert np.array_equal(deq, orc.dequantize(fmt, raw, n_out, n_in)[ids]), fmt
    raw = orc.quantize("q8_0", W)
    y0, a0 = orc.qgemv_argmax("q8_0", raw, n_out, n_in, x)           # the identity list is the full head
    y1, a1 = orc.qgemv_argmax_ids("q8_0", raw, n_out, n_in, x, np.arange(n_out, dtype=np.int32))
    assert np.allclose(y0, y1, rtol=1e-13, atol=1e-15) and list(a0) == list(a1)
    try:
        orc.gather_rows("q8_0", raw, n_out, n_in, [n_out])
        raise AssertionError("an id past the head was accepted")
    except IndexError:
        pass


def check_experts(orc):
    """Expert-grouped mat-vec ([Track2] section 1 item 2: tokens grouped by expert,
    each group run with its own token count): every group equals the plain mat-vec
    of its expert's rows on its tokens, and grouping all tokens under one expert
    equals the stacked matrix's rows of that expert."""
    n_experts, n_out, n_in = 5, 24, 128
    W = workloads.gaussian(81, (n_experts * n_out, n_in), 0.02)
    x = workloads.gaussian(82, (4, n_in))
    for fmt in ("q8_0", "q4_0", "affine4_g64", "bf16"):
        raw = orc.quantize(fmt, W)
        ge = [3, 0, 4, 3]
        gt = [[2], [0, 1, 3], [3, 2, 1, 0], [1, 0]]
        y = orc.experts_gemv(fmt, raw, n_experts, n_out, n_in, x, ge, gt)
        full = orc.gemv(fmt, raw, n_experts * n_out, n_in, x)          # every token x every stacked row
        for g, (e, toks) in enumerate(zip(ge, gt)):
            for k, t in enumerate(toks):
                assert np.allclose(y[g, k], full[t, e * n_out:(e + 1) * n_out], rtol=1e-13, atol=1e-15), (fmt, g, k)
            assert np.all(np.isnan(y[g, len(toks):]))
        # hand check of one output: expert 4, token 1 (slot 2 of group 2), row 5
        deq = orc.dequantize(fmt, raw, n_experts * n_out, n_in)
        assert np.isclose(y[2, 2, 5], float(deq[4 * n_out + 5] @ x[1].astype(np.float64)), rtol=1e-13, atol=1e-15)
    try:
        orc.experts_gemv("q8_0", orc.quantize("q8_0", W), n_experts, n_out, n_in, x, [n_experts], [[0]])
        raise AssertionError("an expert past the stack was accepted")
    except ValueError:
        pass


def check_expert_plan(orc):
    """The routed-expert plan ([Track2] section 1 item 2: moe_plan groups the pairs by
    expert).  A hand-worked case, the invariants of the grouping on random routing,
    the four-pair chunking, and the unique-expert count."""
    # ids[t][j]: pairs i = 0..5 -> experts 3,1 | 1,0 | 3,2.  By expert, then i:
    # e0: [3]   e1: [1, 2]   e2: [5]   e3: [0, 4]
    p = orc.expert_plan([[3, 1], [1, 0], [3, 2]], 4)
    assert p["group_start"].tolist() == [0, 1, 3, 4, 6]
    assert p["group_expert"].tolist() == [0, 1, 2, 3]
    assert p["slot_pair"].tolist() == [3, 1, 2, 5, 0, 4]
    assert p["slot_token"].tolist() == [1, 0, 1, 2, 0, 2]
    assert p["pair_slot"].tolist() == [4, 1, 2, 0, 5, 3]
    # one expert taken by six pairs: groups of 4 then 2, both for that expert
    p = orc.expert_plan([[7, 7, 7], [7, 7, 7]], 8)
    assert p["group_start"].tolist() == [0, 4, 6] and p["group_expert"].tolist() == [7, 7]
    assert p["slot_pair"].tolist() == [0, 1, 2, 3, 4, 5]
    rng = np.random.default_rng(5)
    for trial in range(60):
        ntok, topk, n_exp = int(rng.integers(1, 6)), int(rng.integers(1, 11)), int(rng.integers(1, 40))
        ids = rng.integers(0, n_exp, size=(ntok, topk))
        p = orc.expert_plan(ids, n_exp)
        gs, ge, sp = p["group_start"], p["group_expert"], p["slot_pair"]
        n = ntok * topk
        assert gs[0] == 0 and gs[-1] == n and np.all(np.diff(gs) >= 1) and np.all(np.diff(gs) <= 4)
        assert sorted(sp.tolist()) == list(range(n))                       # every pair exactly once
        assert np.all(p["pair_slot"][sp] == np.arange(n))
        assert np.all(p["slot_token"] == sp // topk)
        flat = ids.reshape(-1)
        for g in range(len(ge)):
            sl = sp[gs[g]:gs[g + 1]]
            assert np.all(flat[sl] == ge[g]) and np.all(np.diff(sl) > 0)
        assert np.all(np.diff(ge) >= 0)
        for g in range(1, len(ge)):             # a repeated expert only after a full group
            if ge[g] == ge[g - 1]:
                assert gs[g] - gs[g - 1] == 4
        counts = np.bincount(flat, minlength=n_exp)
        assert len(ge) == int(np.sum((counts + 3) // 4))
    for bad in ([[0, 4]], [[-1, 0]]):
        try:
            orc.expert_plan(bad, 4)
            raise AssertionError("an expert id outside the stack was accepted")
        except ValueError:
            pass
    # the slot form of the mat-vec is the group form laid out by slot
    n_experts, n_out, n_in = 6, 16, 64
    W = workloads.gaussian(83, (n_experts * n_out, n_in), 0.02)
    raw = orc.quantize("q8_0", W)
    ids = [[5, 2, 0], [2, 1, 5]]
    p = orc.expert_plan(ids, n_experts)
    xt = workloads.gaussian(84, (2, n_in))
    y = orc.experts_gemv_slots("q8_0", raw, n_experts, n_out, n_in, xt, p, False)
    full = orc.gemv("q8_0", raw, n_experts * n_out, n_in, xt)
    for i in range(6):
        t, e, s = i // 3, ids[i // 3][i % 3], int(p["pair_slot"][i])
        assert np.allclose(y[s], full[t, e * n_out:(e + 1) * n_out], rtol=1e-13, atol=1e-15)
    xs = workloads.gaussian(85, (6, n_in))
    y = orc.experts_gemv_slots("q8_0", raw, n_experts, n_out, n_in, xs, p, True)
    full = orc.gemv("q8_0", raw, n_experts * n_out, n_in, xs)
    for s in range(6):
        e = int(p["group_expert"][np.searchsorted(p["group_start"], s, side="right") - 1])
        assert np.allclose(y[s], full[s, e * n_out:(e + 1) * n_out], rtol=1e-13, atol=1e-15)


def check_swiglu(orc):
    """SiLU and the interleaved gate / up activation, by closed forms: silu(0) = 0,
    silu(v) - silu(-v) = v (sigmoid(v) + sigmoid(-v) = 1), silu(ln 3) = 0.75 ln 3
    (sigmoid(ln 3) = 3/4), silu(v) -> v for large v and -> 0 for very negative v; the
    activation pairs row 2j (gate) with row 2j + 1 (up)."""
    assert orc.silu(0.0) == 0.0
    v = np.linspace(-9, 9, 37)
    assert np.allclose(orc.silu(v) - orc.silu(-v), v, rtol=0, atol=1e-14)
    assert abs(float(orc.silu(np.log(3.0))) - 0.75 * np.log(3.0)) < 1e-15
    assert abs(float(orc.silu(40.0)) - 40.0) < 1e-12 and abs(float(orc.silu(-40.0))) < 1e-15
    y = np.array([[np.log(3.0), 2.0, 0.0, 5.0, -np.log(3.0), 4.0]])
    a = orc.swiglu_rows(y)
    want = [0.75 * np.log(3.0) * 2.0, 0.0, -0.25 * np.log(3.0) * 4.0]
    assert a.shape == (1, 3) and np.allclose(a[0], want, rtol=1e-15, atol=1e-15)


ALL_CHECKS = [check_page_byte_counts, check_golden_q8_0, check_golden_q4_0, check_golden_q5_0, check_golden_affine4,
              check_golden_bf16, check_rounding, check_brute_force, check_idempotence,
              check_affine_constructed_roundtrip, check_linearity, check_token_independence,
              check_cross_format, check_argmax, check_quant_error_band, check_fp16_bf16_rounding,
              check_draft_ids, check_experts, check_expert_plan,
              check_swiglu]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(ORC)


def test_row_subset_and_chunking():
    """The row-subset path and the 4096-row chunking agree with the whole-matrix path."""
    n_out, n_in = 9000, 64
    W = workloads.gaussian(61, (n_out, n_in), 0.02)
    x = workloads.gaussian(62, (2, n_in))
    for fmt in ("q8_0", "affine4_g64"):
        raw = ORC.quantize(fmt, W)
        y = ORC.gemv(fmt, raw, n_out, n_in, x)
        deq = ORC.dequantize(fmt, raw, n_out, n_in)
        assert np.array_equal(y, np.stack([deq @ xt for xt in x.astype(np.float64)]))
        rows = np.array([0, 1, 4095, 4096, 8191, 8999])
        assert np.array_equal(ORC.gemv(fmt, raw, n_out, n_in, x, rows=rows), y[:, rows])
        assert np.allclose(ORC.gemv_abs(fmt, raw, n_out, n_in, x, rows=rows),
                           (np.abs(x.astype(np.float64)) @ np.abs(deq).T)[:, rows], rtol=1e-14)
