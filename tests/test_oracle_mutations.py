"""Plant mistakes in a copy of the oracle and show that its pins catch each one.

Every mutation edits the oracle's source text (one substring, which must occur
exactly once), loads the edited copy as a fresh module on the CPU, and runs all
the pin checks of ``test_oracle_pins.py`` against it: at least one must fail.
The real oracle is never modified.
"""
from __future__ import annotations

import importlib.util
import os
import types

import pytest

import test_oracle_pins as PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "qgemv_oracle.py")

MUTATIONS = {
    "q4_0 offset sign": ("return ((q - 8.0) * d[..., None])", "return ((q + 8.0) * d[..., None])"),
    "q4_0 nibble order": ("q = np.concatenate([lo, hi], axis=2)", "q = np.stack([lo, hi], axis=3).reshape(lo.shape[0], lo.shape[1], 32)"),
    "q4_0 packing order": ('out["qs"] = q[..., :16] | (q[..., 16:] << 4)', 'out["qs"] = q[..., 0::2] | (q[..., 1::2] << 4)'),
    "q4_0 unsigned max": ("m = np.take_along_axis(B, idx[..., None], axis=2)[..., 0]", "m = np.abs(np.take_along_axis(B, idx[..., None], axis=2)[..., 0])"),
    "affine dropped bias": ("return (q * s[..., None] + b[..., None]).reshape(n_out, n_in)", "return (q * s[..., None]).reshape(n_out, n_in)"),
    "affine bit order": ("q = np.stack([(words >> np.uint32(4 * k)) & np.uint32(0xF) for k in range(8)], axis=2)",
                         "q = np.stack([(words >> np.uint32(28 - 4 * k)) & np.uint32(0xF) for k in range(8)], axis=2)"),
    "affine bias from max": ("b16 = mn.astype(np.float16)", "b16 = mx.astype(np.float16)"),
    "q8_0 sign": ("return (q * d[..., None]).reshape(n_out, n_in)", "return (-q * d[..., None]).reshape(n_out, n_in)"),
    "q8_0 divisor": ("d32 = amax / np.float32(127)", "d32 = amax / np.float32(128)"),
    "q8_0 bytes without scale": ("return n // 32 * 34", "return n // 32 * 32"),
    "affine bytes without biases": ("return n // 2 + (n // 64) * 4", "return n // 2 + (n // 64) * 2"),
    "rounding half-even": ("return t + np.where(np.abs(frac) >= np.float32(0.5), np.sign(v), np.float32(0))",
                           "return np.round(v)"),
    "bf16 truncation": ("r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "r = u >> 16"),
    "gemv reversed x": ("y[t, r0:r1] = deq @ x64[t]", "y[t, r0:r1] = deq @ x64[t][::-1]"),
    "gemv wrong token": ("y[t, r0:r1] = deq @ x64[t]", "y[t, r0:r1] = deq @ x64[0]"),
    "argmax last index": ("return np.argmax(yy, axis=1).astype(np.int32)",
                          "return (yy.shape[1] - 1 - np.argmax(yy[:, ::-1], axis=1)).astype(np.int32)"),
    "draft argmax not mapped": ("return y, ids[j].astype(np.int32)", "return y, j.astype(np.int32)"),
    "experts wrong expert rows": ("sub = row_slice(f, packed, n_experts * n_out, n_in, e * n_out, (e + 1) * n_out)",
                                  "sub = row_slice(f, packed, n_experts * n_out, n_in, 0, n_out)"),
    "experts tokens reversed": ("y[g, :len(toks)] = gemv(f, sub, n_out, n_in, x[toks])",
                                "y[g, :len(toks)] = gemv(f, sub, n_out, n_in, x[toks[::-1]])"),
    "plan pairs by token not by expert": ("pairs = [i for i, v in enumerate(flat) if v == e]",
                                          "pairs = [i for i, v in enumerate(flat) if v == e][::-1]"),
    "plan groups of five": ("MAX_GROUP_SLOTS = 4     # tokens", "MAX_GROUP_SLOTS = 5     # tokens"),
    "plan slot_token off by one": ('"slot_token": np.array(slot_pair, dtype=np.int64) // topk,',
                                   '"slot_token": np.array(slot_pair, dtype=np.int64) // max(topk - 1, 1),'),
    "slots read token rows in down mode": ("rows = slots if x_by_slot else",
                                           "rows = slots if not x_by_slot else"),
    "swiglu gate and up swapped": ("return silu(y[..., 0::2]) * y[..., 1::2]", "return silu(y[..., 1::2]) * y[..., 0::2]"),
    "silu without the sigmoid": ("return v / (1.0 + np.exp(-v))", "return v / (1.0 + np.exp(v))"),
    "q5 offset 15": ("return ((q - 16.0) * d[..., None]).reshape(n_out, n_in)",
                     "return ((q - 15.0) * d[..., None]).reshape(n_out, n_in)"),
    "q5 high bit of the next element": ("hb = (blk[\"qh\"][..., None] >> np.arange(32, dtype=np.uint32)) & np.uint32(1)",
                                         "hb = (blk[\"qh\"][..., None] >> ((np.arange(32, dtype=np.uint32) + 1) % 32)) & np.uint32(1)"),
    "q5 divisor 15": ("d32 = m5 / np.float32(-16)", "d32 = m5 / np.float32(-15)"),
    "q5 unsigned max": ("m5 = np.take_along_axis(B, first[..., None], axis=2)[..., 0]",
                        "m5 = np.abs(np.take_along_axis(B, first[..., None], axis=2)[..., 0])"),
    "draft gather ignores affine scales": ("s = packed[nw * 4: nw * 4 + ng * 2].reshape(n_out, n_in // 32)[ids]",
                                           "s = packed[nw * 4: nw * 4 + ng * 2].reshape(n_out, n_in // 32)[:ids.size]"),
}


def _mutant(old: str, new: str) -> types.ModuleType:
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique / missing: {old!r}"
    spec = importlib.util.spec_from_loader("oracle_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    failed = []
    for check in PINS.ALL_CHECKS:
        try:
            check(mod)
        except Exception:          # an AssertionError, or the mutant crashing
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_unmutated_copy_passes_everything():
    mod = _mutant("GEMV_CHUNK = 1024", "GEMV_CHUNK = 1024")
    for check in PINS.ALL_CHECKS:
        check(mod)
