"""Python binding of the block-quantized weight mat-vec library (GB300, sm_103a).

A thin ctypes layer over ``_lib/libqgemv.so`` (C ABI in ``include/qgemv.h``):
the functions carry the C names and only marshal arguments.  Device buffers
are torch CUDA tensors (or raw device addresses); host buffers for the packer
are numpy arrays.  Every step of the mat-vec runs in the library's CUDA
kernels; if the library is missing, every call raises.

    y[t, o] = sum_i dequant(W)[o, i] * x[t, i],  ntok = 1..4
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "QG_Q8_0", "QG_Q4_0", "QG_AFFINE4_G64", "QG_BF16", "QG_Q5_0", "FORMATS", "QGError", "load_library",
    "qg_strerror", "qg_abi_version", "qg_canonical_bytes", "qg_packed_bytes", "qg_row_stride",
    "qg_quantize", "qg_to_device_layout", "qg_pack", "qgemv", "qgemv_argmax_workspace_bytes",
    "qgemv_argmax", "qg_set_tile_override", "qg_describe_tile", "weight_bytes", "qg_device_status",
    "qg_set_wait_limit", "QG_DEVICE_WAIT_TIMEOUT", "qgemv_argmax_noalloc", "qg_set_launch_options",
    "QG_LAUNCH_EARLY_START", "current_stream_handle", "qg_gather_rows", "qgemv_argmax_ids",
    "QG_DEVICE_BAD_ROW_ID", "qg_expert_plan_ints", "qg_expert_plan", "qgemv_experts", "qg_describe_expert_tile",
    "QG_DEVICE_BAD_PLAN", "QG_EXPERTS_X_BY_SLOT", "QG_EXPERTS_PLAN_READY",
    "QG_EXPERTS_SWIGLU", "qgemv_expert_layer", "qgemv_expert_layer_workspace_bytes",
    "qg_set_phase_record", "QG_PHASE_WORDS", "QG_PHASE_SLOT_WORDS",
]

QG_Q8_0, QG_Q4_0, QG_AFFINE4_G64, QG_BF16, QG_Q5_0 = 0, 1, 2, 3, 4
FORMATS = {"q8_0": QG_Q8_0, "q4_0": QG_Q4_0, "affine4_g64": QG_AFFINE4_G64, "bf16": QG_BF16, "q5_0": QG_Q5_0}

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libqgemv.so")
_lib = None


class QGError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {qg_strerror(status)} (status {status})")


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return FORMATS[fmt]
    return int(fmt)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library once (build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
    try:
        import torch  # noqa: F401  (load torch's CUDA runtime first so one copy is shared)
    except ImportError:
        pass
    lib = ctypes.CDLL(p)
    i64, vp, sz, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    sig = {
        "qg_strerror": (ctypes.c_char_p, [i32]),
        "qg_abi_version": (i32, []),
        "qg_canonical_bytes": (sz, [i32, i64, i64]),
        "qg_packed_bytes": (sz, [i32, i64, i64]),
        "qg_row_stride": (i64, [i32, i64]),
        "qg_quantize": (i32, [i32, vp, i64, i64, vp]),
        "qg_to_device_layout": (i32, [i32, vp, i64, i64, vp]),
        "qg_pack": (i32, [i32, vp, i64, i64, vp]),
        "qgemv": (i32, [i32, vp, i64, i64, vp, vp, i32, vp]),
        "qgemv_argmax_workspace_bytes": (sz, [i64, i32]),
        "qgemv_argmax": (i32, [i32, vp, i64, i64, vp, vp, vp, i32, vp, sz, vp]),
        "qg_set_tile_override": (i32, [ctypes.c_char_p]),
        "qg_describe_tile": (i32, [i32, i64, i64, i32, ctypes.c_char_p, sz]),
        "qg_device_status": (i32, [i32, ctypes.POINTER(ctypes.c_uint)]),
        "qg_set_wait_limit": (i32, [ctypes.c_uint, ctypes.c_uint]),
        "qgemv_argmax_noalloc": (i32, [i32, vp, i64, i64, vp, vp, vp, i32, vp]),
        "qg_set_launch_options": (i32, [ctypes.c_uint]),
        "qg_set_phase_record": (i32, [vp, i64]),
        "qg_gather_rows": (i32, [i32, vp, i64, i64, vp, i64, vp, vp]),
        "qgemv_argmax_ids": (i32, [i32, vp, i64, i64, vp, vp, vp, i32, vp, vp, sz, vp]),
        "qg_expert_plan_ints": (sz, [i64]),
        "qg_expert_plan": (i32, [vp, i32, i32, i32, vp, vp]),
        "qgemv_experts": (i32, [i32, vp, i64, i64, i64, vp, i64, ctypes.c_uint, vp, i64, vp, vp, i64, i64, vp]),
        "qg_describe_expert_tile": (i32, [i32, i64, i64, ctypes.c_char_p, sz]),
        "qgemv_expert_layer_workspace_bytes": (sz, []),
        "qgemv_expert_layer": (i32, [i32, vp, vp, i64, i64, i64, vp, i32, vp, i32, vp, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> int | None:
    """Device address of a torch tensor / raw int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    raise TypeError(f"expected a torch tensor or an address, got {type(t)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def current_stream_handle() -> int:
    """torch's current CUDA stream as a raw ``cudaStream_t`` (0 = the legacy default stream)."""
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


def _check(status: int, what: str) -> None:
    if status != 0:
        raise QGError(status, what)


# ----------------------------------------------------------------------------- sizes

def qg_strerror(status: int) -> str:
    return load_library().qg_strerror(int(status)).decode()


def qg_abi_version() -> int:
    return load_library().qg_abi_version()


def qg_canonical_bytes(fmt, n_out: int, n_in: int) -> int:
    return load_library().qg_canonical_bytes(_fmt(fmt), n_out, n_in)


weight_bytes = qg_canonical_bytes


def qg_packed_bytes(fmt, n_out: int, n_in: int) -> int:
    return load_library().qg_packed_bytes(_fmt(fmt), n_out, n_in)


def qg_row_stride(fmt, n_in: int) -> int:
    return load_library().qg_row_stride(_fmt(fmt), n_in)


# ----------------------------------------------------------------------------- host packer

def _f32_host(W) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.float32)
    if W.ndim != 2:
        raise ValueError("W must be [n_out, n_in]")
    return W


def qg_quantize(fmt, W) -> np.ndarray:
    """fp32 ``[n_out, n_in]`` -> canonical bytes (uint8)."""
    W = _f32_host(W)
    n_out, n_in = W.shape
    out = np.empty(max(1, qg_canonical_bytes(fmt, n_out, n_in)), dtype=np.uint8)
    _check(load_library().qg_quantize(_fmt(fmt), W.ctypes.data, n_out, n_in, out.ctypes.data), "qg_quantize")
    return out


def qg_to_device_layout(fmt, canonical, n_out: int, n_in: int) -> np.ndarray:
    src = np.ascontiguousarray(canonical, dtype=np.uint8)
    if src.size != qg_canonical_bytes(fmt, n_out, n_in):
        raise ValueError("canonical buffer has the wrong size")
    out = np.empty(max(1, qg_packed_bytes(fmt, n_out, n_in)), dtype=np.uint8)
    _check(load_library().qg_to_device_layout(_fmt(fmt), src.ctypes.data, n_out, n_in, out.ctypes.data),
           "qg_to_device_layout")
    return out


def qg_pack(fmt, W, out: np.ndarray | None = None) -> np.ndarray:
    """fp32 ``[n_out, n_in]`` -> device-layout bytes (uint8), optionally into ``out``."""
    W = _f32_host(W)
    n_out, n_in = W.shape
    n = qg_packed_bytes(fmt, n_out, n_in)
    if out is None:
        out = np.empty(max(1, n), dtype=np.uint8)
    if out.dtype != np.uint8 or not out.flags["C_CONTIGUOUS"] or out.size < n:
        raise ValueError("out must be a contiguous uint8 array of qg_packed_bytes bytes")
    _check(load_library().qg_pack(_fmt(fmt), W.ctypes.data, n_out, n_in, out.ctypes.data), "qg_pack")
    return out


# ----------------------------------------------------------------------------- the mat-vec

def qgemv(fmt, W, n_out: int, n_in: int, x, y, ntok: int | None = None, stream=None) -> None:
    """Enqueue ``y[t, o] = sum_i dequant(W)[o, i] * x[t, i]`` on ``stream`` (default: torch's
    current).  ``stream`` may be a torch stream or a raw ``cudaStream_t`` as an int; passing
    the int saves a torch lookup per call in launch-bound loops."""
    if ntok is None:
        ntok = x.shape[0] if getattr(x, "dim", lambda: 1)() == 2 else 1
    lib = _lib if _lib is not None else load_library()
    st = lib.qgemv(FORMATS[fmt] if isinstance(fmt, str) else int(fmt), _ptr(W), n_out, n_in, _ptr(x), _ptr(y),
                   int(ntok), stream if isinstance(stream, int) else _stream(stream))
    if st != 0:
        raise QGError(st, "qgemv")


def qgemv_argmax_workspace_bytes(n_out: int, ntok: int) -> int:
    return load_library().qgemv_argmax_workspace_bytes(n_out, ntok)


def qgemv_argmax(fmt, W, n_out: int, n_in: int, x, y, argmax, workspace, ntok: int | None = None,
                 workspace_bytes: int | None = None, stream=None) -> None:
    """Enqueue the mat-vec fused with the per-token first-index argmax (y may be None)."""
    if ntok is None:
        ntok = x.shape[0] if getattr(x, "dim", lambda: 1)() == 2 else 1
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    st = load_library().qgemv_argmax(_fmt(fmt), _ptr(W), n_out, n_in, _ptr(x), _ptr(y), _ptr(argmax),
                                     int(ntok), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "qgemv_argmax")


def qgemv_argmax_noalloc(fmt, W, n_out: int, n_in: int, x, y, argmax, ntok: int | None = None,
                         stream=None) -> None:
    """qgemv_argmax without a workspace, for callers that cannot allocate device memory:
    the scratch is a fixed array inside the library (calls that overlap on the GPU race)."""
    if ntok is None:
        ntok = x.shape[0] if getattr(x, "dim", lambda: 1)() == 2 else 1
    st = load_library().qgemv_argmax_noalloc(_fmt(fmt), _ptr(W), n_out, n_in, _ptr(x), _ptr(y), _ptr(argmax),
                                             int(ntok), _stream(stream))
    _check(st, "qgemv_argmax_noalloc")


def qg_gather_rows(fmt, W, n_out: int, n_in: int, ids, out, n_ids: int | None = None, stream=None) -> None:
    """Enqueue the copy of rows ``ids`` (device int32) of the packed matrix ``W`` into ``out``
    (a packed ``n_ids``-row matrix): the small head of a draft vocabulary."""
    if n_ids is None:
        n_ids = ids.numel()
    _check(load_library().qg_gather_rows(_fmt(fmt), _ptr(W), n_out, n_in, _ptr(ids), int(n_ids), _ptr(out),
                                         _stream(stream)), "qg_gather_rows")


def qgemv_argmax_ids(fmt, W_sub, n_sub: int, n_in: int, x, y, argmax, ids, workspace, ntok: int | None = None,
                     workspace_bytes: int | None = None, stream=None) -> None:
    """qgemv_argmax over a gathered head; argmax[t] is written as ids[winning row] (full-vocab id)."""
    if ntok is None:
        ntok = x.shape[0] if getattr(x, "dim", lambda: 1)() == 2 else 1
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    st = load_library().qgemv_argmax_ids(_fmt(fmt), _ptr(W_sub), n_sub, n_in, _ptr(x), _ptr(y), _ptr(argmax),
                                         int(ntok), _ptr(ids), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "qgemv_argmax_ids")


QG_DEVICE_BAD_ROW_ID = 2
QG_DEVICE_BAD_PLAN = 4
QG_EXPERTS_X_BY_SLOT = 1
QG_EXPERTS_PLAN_READY = 2
QG_EXPERTS_SWIGLU = 4


def qg_expert_plan_ints(n_pairs: int) -> int:
    """int32 entries of the plan of ``n_pairs`` routed (token, choice) pairs (0 if out of range)."""
    return int(load_library().qg_expert_plan_ints(int(n_pairs)))


def qg_expert_plan(ids, n_experts: int, plan, stream=None) -> None:
    """Enqueue the plan of the routing ``ids`` (device int32 ``[ntok, topk]``) into ``plan``
    (device int32, ``qg_expert_plan_ints(ntok * topk)`` entries)."""
    ntok, topk = int(ids.shape[0]), int(ids.shape[1])
    _check(load_library().qg_expert_plan(_ptr(ids), ntok, topk, int(n_experts), _ptr(plan), _stream(stream)),
           "qg_expert_plan")


def qgemv_experts(fmt, W, n_experts: int, n_out: int, n_in: int, x, plan, n_slots: int, y,
                  x_by_slot: bool = False, W_next=None, next_n_out: int = 0, next_n_in: int = 0,
                  plan_ready: bool = False, swiglu: bool = False, stream=None) -> None:
    """Enqueue the expert-grouped mat-vec: ``y[s] = W_e . x_row(s)`` for every slot s of the
    plan (``x_row(s) = x[slot_token[s]]``, or ``x[s]`` with ``x_by_slot``); optionally prefetch
    the active experts of the next projection's stack ``W_next`` into L2.  ``plan_ready``:
    the plan is complete when the launch begins (see QG_EXPERTS_PLAN_READY).  ``swiglu``: the
    rows pair up as (gate, up) and y receives silu(gate) * up, ``[n_slots, n_out / 2]``."""
    flags = ((QG_EXPERTS_X_BY_SLOT if x_by_slot else 0) | (QG_EXPERTS_PLAN_READY if plan_ready else 0)
             | (QG_EXPERTS_SWIGLU if swiglu else 0))
    _check(load_library().qgemv_experts(_fmt(fmt), _ptr(W), int(n_experts), int(n_out), int(n_in), _ptr(x),
                                        int(x.shape[0]), flags, _ptr(plan), int(n_slots), _ptr(y),
                                        _ptr(W_next), int(next_n_out), int(next_n_in), _stream(stream)),
           "qgemv_experts")


def qgemv_expert_layer_workspace_bytes() -> int:
    return int(load_library().qgemv_expert_layer_workspace_bytes())


def qgemv_expert_layer(fmt, W_gate_up, W_down, n_experts: int, d_model: int, d_ff: int, x, ids, plan, act, y,
                       workspace, stream=None) -> None:
    """Enqueue the whole routed-expert layer as one launch: plan (written to ``plan``),
    ``act = silu(gate) * up`` for every slot, then ``y = W_down . act``.  ``ids``: device
    int32 ``[ntok, topk]``; ``workspace``: zeroed once, ``qgemv_expert_layer_workspace_bytes()``."""
    ntok, topk = int(ids.shape[0]), int(ids.shape[1])
    _check(load_library().qgemv_expert_layer(_fmt(fmt), _ptr(W_gate_up), _ptr(W_down), int(n_experts), int(d_model),
                                             int(d_ff), _ptr(x), ntok, _ptr(ids), topk, _ptr(plan), _ptr(act), _ptr(y),
                                             _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                             _stream(stream)), "qgemv_expert_layer")


def qg_describe_expert_tile(fmt, n_out: int, n_in: int) -> str:
    buf = ctypes.create_string_buffer(128)
    _check(load_library().qg_describe_expert_tile(_fmt(fmt), n_out, n_in, buf, 128), "qg_describe_expert_tile")
    return buf.value.decode()


def qg_set_tile_override(spec: str | None) -> None:
    _check(load_library().qg_set_tile_override(spec.encode() if spec else None), "qg_set_tile_override")


def qg_device_status(clear: bool = True) -> int:
    """The current device's status word (QG_DEVICE_WAIT_TIMEOUT = 1 if a bounded wait gave up)."""
    v = ctypes.c_uint(0)
    _check(load_library().qg_device_status(1 if clear else 0, ctypes.byref(v)), "qg_device_status")
    return v.value


def qg_set_wait_limit(polls: int = 0, extra_tx_bytes: int = 0) -> None:
    """Test hook: mbarrier polls before a wait gives up (0 = default) and extra expected bytes."""
    _check(load_library().qg_set_wait_limit(int(polls), int(extra_tx_bytes)), "qg_set_wait_limit")


QG_DEVICE_WAIT_TIMEOUT = 1
QG_LAUNCH_EARLY_START = 1
QG_PHASE_WORDS = 16
QG_PHASE_SLOT_WORDS = 4096 * QG_PHASE_WORDS


def qg_set_phase_record(buf, slots: int = 0) -> None:
    """Profiling hook: per-CTA phase stamps of every later mat-vec launch into `buf`
    (a CUDA uint64/int64 tensor of slots * QG_PHASE_SLOT_WORDS words; None turns it off)."""
    if buf is None:
        _check(load_library().qg_set_phase_record(None, 0), "qg_set_phase_record")
        return
    if buf.numel() < slots * QG_PHASE_SLOT_WORDS or buf.element_size() != 8:
        raise ValueError("qg_set_phase_record: buffer smaller than slots * QG_PHASE_SLOT_WORDS 8-byte words")
    _check(load_library().qg_set_phase_record(_ptr(buf), int(slots)), "qg_set_phase_record")


def qg_set_launch_options(flags: int) -> None:
    """QG_LAUNCH_EARLY_START: overlap back-to-back calls (weights must not be written in flight)."""
    _check(load_library().qg_set_launch_options(int(flags)), "qg_set_launch_options")


def qg_describe_tile(fmt, n_out: int, n_in: int, ntok: int) -> str:
    buf = ctypes.create_string_buffer(160)
    _check(load_library().qg_describe_tile(_fmt(fmt), n_out, n_in, ntok, buf, len(buf)), "qg_describe_tile")
    return buf.value.decode()
