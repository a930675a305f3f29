"""The C ABI without a GPU: the library loads, exports every function that
include/qgemv.h declares, and rejects bad arguments before launching anything."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import block_quantized_token_format_gb300 as qg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b((?:qg|qgemv)\w*)\s*\(", text)))


def test_exports_every_declared_symbol():
    lib = ctypes.CDLL(qg._LIB_PATH)
    names = declared_functions()
    assert "qgemv" in names and "qgemv_argmax" in names and "qg_pack" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    assert qg.qg_abi_version() == 1
    for s in (0, -1, -2, -3, -4, -5):
        assert qg.qg_strerror(s) and qg.qg_strerror(s) != "unknown status"
    assert qg.qg_strerror(-99) == "unknown status"


A = 1 << 20          # a 16-byte-aligned fake device address (never dereferenced)


@pytest.mark.parametrize("args,code", [
    ((9, A, 8, 256, A, A, 1), -1),        # bad format
    ((0, A, 0, 256, A, A, 1), -1),        # n_out < 1
    ((0, A, 8, 48, A, A, 1), -1),         # n_in not a multiple of 32
    ((2, A, 8, 96, A, A, 1), -1),         # affine needs 64
    ((3, A, 8, 24, A, A, 1), -1),         # bf16 needs 16
    ((0, A, 8, 256, A, A, 0), -1),        # ntok 0
    ((0, A, 8, 256, A, A, 5), -1),        # ntok 5
    ((0, None, 8, 256, A, A, 1), -1),     # null W
    ((0, A, 8, 256, None, A, 1), -1),     # null x
    ((0, A, 8, 256, A, None, 1), -1),     # null y
    ((0, A + 8, 8, 256, A, A, 1), -2),    # W misaligned
    ((0, A, 8, 256, A + 4, A, 1), -2),    # x misaligned
    ((0, A, 8, 256, A, A + 2, 1), -2),    # y misaligned
])
def test_qgemv_rejects_before_launch(args, code):
    lib = qg.load_library()
    assert lib.qgemv(*args, None) == code


def test_argmax_rejects_before_launch():
    lib = qg.load_library()
    ws = qg.qgemv_argmax_workspace_bytes(100, 4)
    assert ws >= 16 + 4096 * 4 * 8
    assert qg.qgemv_argmax_workspace_bytes(100, 0) == 0
    assert lib.qgemv_argmax(0, A, 100, 256, A, A, A, 4, None, ws, None) == -4
    assert lib.qgemv_argmax(0, A, 100, 256, A, A, A, 4, A, ws - 1, None) == -4
    assert lib.qgemv_argmax(0, A, 100, 256, A, A, None, 4, A, ws, None) == -1
    assert lib.qgemv_argmax(0, A, 100, 256, A, A, A + 2, 4, A, ws, None) == -2
    assert lib.qgemv_argmax(0, A, 100, 256, A, A, A, 4, A + 8, ws, None) == -2


def test_draft_ids_calls_reject_before_launch():
    lib = qg.load_library()
    ws = qg.qgemv_argmax_workspace_bytes(100, 4)
    # qg_gather_rows(fmt, W, n_out, n_in, ids, n_ids, W_out, stream)
    assert lib.qg_gather_rows(9, A, 100, 256, A, 10, A, None) == -1          # bad format
    assert lib.qg_gather_rows(0, A, 100, 48, A, 10, A, None) == -1           # bad n_in
    assert lib.qg_gather_rows(0, None, 100, 256, A, 10, A, None) == -1       # null W
    assert lib.qg_gather_rows(0, A, 100, 256, None, 10, A, None) == -1       # null ids
    assert lib.qg_gather_rows(0, A, 100, 256, A, 10, None, None) == -1       # null out
    assert lib.qg_gather_rows(0, A, 100, 256, A, 0, A, None) == -1           # no ids
    assert lib.qg_gather_rows(0, A, 100, 256, A, 1 << 31, A, None) == -1     # too many ids
    assert lib.qg_gather_rows(0, A + 8, 100, 256, A, 10, A, None) == -2      # W misaligned
    assert lib.qg_gather_rows(0, A, 100, 256, A, 10, A + 8, None) == -2      # out misaligned
    assert lib.qg_gather_rows(0, A, 100, 256, A + 2, 10, A, None) == -2      # ids misaligned
    # qgemv_argmax_ids(fmt, W, n_sub, n_in, x, y, argmax, ntok, ids, ws, ws_bytes, stream)
    assert lib.qgemv_argmax_ids(0, A, 100, 256, A, A, A, 4, None, A, ws, None) == -1     # null ids
    assert lib.qgemv_argmax_ids(0, A, 100, 256, A, A, A, 4, A + 2, A, ws, None) == -2    # ids misaligned
    assert lib.qgemv_argmax_ids(0, A, 100, 256, A, A, A, 4, A, None, ws, None) == -4     # no workspace
    assert lib.qgemv_argmax_ids(0, A, 100, 256, A, A, A, 5, A, A, ws, None) == -1        # ntok 5


def test_expert_calls_reject_before_launch():
    lib = qg.load_library()
    assert qg.qg_expert_plan_ints(40) == 2 + 5 * 40
    assert qg.qg_expert_plan_ints(0) == 0 and qg.qg_expert_plan_ints(1025) == 0
    # qg_expert_plan(ids, ntok, topk, n_experts, plan, stream)
    assert lib.qg_expert_plan(None, 4, 10, 512, A, None) == -1
    assert lib.qg_expert_plan(A, 4, 10, 512, None, None) == -1
    assert lib.qg_expert_plan(A, 0, 10, 512, A, None) == -1
    assert lib.qg_expert_plan(A, 4, 0, 512, A, None) == -1
    assert lib.qg_expert_plan(A, 4, 10, 0, A, None) == -1
    assert lib.qg_expert_plan(A, 64, 17, 512, A, None) == -1          # 1088 pairs > 1024
    assert lib.qg_expert_plan(A + 2, 4, 10, 512, A, None) == -2
    assert lib.qg_expert_plan(A, 4, 10, 512, A + 2, None) == -2
    # qgemv_experts(fmt, W, n_experts, n_out, n_in, x, n_x, x_by_slot, plan, n_slots, y, stream)
    ok = (0, A, 8, 64, 256, A, 4, 0, A, 40, A, None, 0, 0)
    def call(**kw):
        names = ["fmt", "W", "ne", "no", "ni", "x", "nx", "bs", "plan", "ns", "y", "wn", "nno", "nni"]
        args = dict(zip(names, ok))
        args.update(kw)
        return lib.qgemv_experts(*[args[n] for n in names], None)
    assert call(fmt=9) == -1
    assert call(ne=0) == -1 and call(no=0) == -1
    assert call(ne=1 << 20, no=1 << 12) == -1                            # stack of 2^32 rows
    assert call(ni=48) == -1                                             # n_in not a multiple of 32
    assert call(ns=0) == -1 and call(ns=1025) == -1
    assert call(nx=0) == -1 and call(bs=8) == -1                        # unknown flag
    assert call(bs=4, no=63) == -1                                       # gate/up pairs need even n_out
    assert call(bs=1, nx=39) == -1                                      # one x row per slot needed
    assert call(W=None) == -1 and call(x=None) == -1 and call(plan=None) == -1 and call(y=None) == -1
    assert call(W=A + 8) == -2 and call(x=A + 4) == -2 and call(plan=A + 2) == -2 and call(y=A + 2) == -2
    assert call(wn=A, nno=0, nni=256) == -1 and call(wn=A, nno=64, nni=48) == -1     # bad next stack
    assert call(wn=A + 8, nno=64, nni=256) == -2


def test_expert_layer_rejects_before_launch():
    lib = qg.load_library()
    ws = qg.qgemv_expert_layer_workspace_bytes()
    assert ws >= 8
    # (fmt, Wgu, Wdn, n_experts, d_model, d_ff, x, ntok, ids, topk, plan, act, y, ws, ws_bytes, stream)
    ok = dict(fmt=0, wgu=A, wdn=A, ne=512, dm=2560, ff=640, x=A, ntok=4, ids=A, topk=10, plan=A, act=A, y=A,
              ws=A, wsb=ws)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.qgemv_expert_layer(*a.values(), None)
    assert call(fmt=9) == -1 and call(ne=0) == -1 and call(dm=48) == -1 and call(ff=0) == -1
    assert call(ne=1 << 20) == -1                                        # stacks of >= 2^31 rows
    assert call(ntok=0) == -1 and call(topk=0) == -1 and call(ntok=64, topk=17) == -1
    for k in ("wgu", "wdn", "x", "ids", "plan", "act", "y"):
        assert call(**{k: None}) == -1, k
    assert call(wgu=A + 8) == -2 and call(x=A + 4) == -2 and call(act=A + 4) == -2 and call(y=A + 2) == -2
    assert call(ids=A + 2) == -2 and call(plan=A + 2) == -2
    assert call(ws=None) == -4 and call(wsb=ws - 1) == -4 and call(ws=A + 8) == -2


def test_tile_override_grammar():
    lib = qg.load_library()
    for good in (b"rpw=4", b"depth=2,rpw=1", b"rpw=2,depth=4,warps=8,ctas=2", b"", None, b"rpw=1,", b"rpw=8", b"split=3,rpw=2", b"split=5", b"split=8", b"pre=1", b"pre=16,depth=16", b"rpw=3", b"rpw=5", b"rpw=6", b"gw=0", b"gw=4,rpw=2", b"gw=64"):
        assert lib.qg_set_tile_override(good) == 0, good
    for bad in (b"rpw=7", b"rpw=9", b"rpw=0", b"depth=1", b"depth=17", b"warps=0", b"warps=17", b"ctas=0", b"foo=1", b"rpw", b"rpw=x",
                b"rpw=-1", b"pf=2", b"split=0", b"split=9", b"pre=0", b"pre=17", b"gw=65", b"gw=-1"):
        assert lib.qg_set_tile_override(bad) == -1, bad
    assert lib.qg_set_tile_override(None) == 0


def test_phase_record_arguments():
    """The profiling hook validates on the host: a buffer needs at least one slot and 8-byte
    alignment; NULL turns it off.  (No launch here: the buffers are never dereferenced.)"""
    lib = qg.load_library()
    lib.qg_set_phase_record.argtypes = [ctypes.c_void_p, ctypes.c_int64]
    assert lib.qg_set_phase_record(None, 0) == 0
    assert lib.qg_set_phase_record(0x10000, 0) == -1
    assert lib.qg_set_phase_record(0x10004, 1) == -2
    assert lib.qg_set_phase_record(None, 5) == 0
    assert qg.QG_PHASE_WORDS == 16 and qg.QG_PHASE_SLOT_WORDS == 4096 * 16


def test_launch_options():
    lib = qg.load_library()
    assert lib.qg_set_launch_options(1) == 0
    assert lib.qg_set_launch_options(0) == 0
    assert lib.qg_set_launch_options(2) == -1
    assert lib.qg_set_launch_options(0xFFFF) == -1
