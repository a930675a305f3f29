"""CPU oracle for the block-quantized mat-vec: test infrastructure, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  See ``oracle/qgemv_oracle.py`` for what it computes and
which page passages each part follows.
"""
from .qgemv_oracle import *  # noqa: F401,F403
from .qgemv_oracle import (  # noqa: F401
    Q8_0, Q4_0, AFFINE4_G64, BF16, Q5_0, FMT_NAMES, BLOCK, fmt_id, weight_bytes, quantize, dequantize,
    gemv, gemv_abs, argmax_first, top2_gap, qgemv_argmax, round_half_away, row_slice,
    expert_plan, experts_gemv, experts_gemv_slots, MAX_GROUP_SLOTS, silu, swiglu_rows,
)
