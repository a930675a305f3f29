"""The no-allocation LM-head entry point, through the C ABI, against the
workspace entry point and the oracle.

qgemv_argmax_noalloc serves callers that cannot call cudaMalloc (a plugin whose
host framework owns all device memory, or a decode loop that must never touch
the allocator): its scratch is a fixed array inside the library.  It launches
the same kernel with the same geometry as qgemv_argmax, so on two calls in a
row its logits must be bitwise those of qgemv_argmax, its argmax identical, and
both must match the oracle (logits within the parity tolerance, argmax exact
wherever the oracle's top-2 gap is at least 1e-4).  This file is collected last
so that a stop at its first failure has run every other test.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle as ORC
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import block_quantized_token_format_gb300 as qg  # noqa: E402

TOL = 1e-3
GAP = 1e-4


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_tile_override(None)
    yield
    qg.qg_set_tile_override(None)


@pytest.mark.parametrize("fmt,n_out,n_in", [("q8_0", 30011, 2560), ("affine4_g64", 12345, 5120)])
def test_noalloc_matches_workspace_entry_point_twice(fmt, n_out, n_in):
    dev = torch.device("cuda:0")
    W = workloads.gaussian(7, (n_out, n_in), 0.02)
    x = workloads.activations(7, n_in, 4)
    canon = ORC.quantize(fmt, W)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n_out, n_in)).to(dev)
    xd = torch.from_numpy(x).to(dev)
    ref = ORC.gemv(fmt, canon, n_out, n_in, x)
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
    ref_am, gap = ORC.argmax_first(ref), ORC.top2_gap(ref)
    lib = qg.load_library()
    for ntok in (4, 1, 3):
        ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, ntok), dtype=torch.uint8, device=dev)
        y_ws = torch.empty((ntok, n_out), dtype=torch.float32, device=dev)
        am_ws = torch.empty(ntok, dtype=torch.int32, device=dev)
        qg.qgemv_argmax(fmt, packed, n_out, n_in, xd[:ntok], y_ws, am_ws, ws, ntok)
        torch.cuda.synchronize()
        y_ws, am_ws = y_ws.cpu().numpy(), am_ws.cpu().numpy()
        for call in range(2):
            y = torch.full((ntok, n_out), float("nan"), dtype=torch.float32, device=dev)
            am = torch.full((ntok,), -9, dtype=torch.int32, device=dev)
            st = lib.qgemv_argmax_noalloc(qg.FORMATS[fmt], packed.data_ptr(), n_out, n_in, xd.data_ptr(),
                                          y.data_ptr(), am.data_ptr(), ntok,
                                          torch.cuda.current_stream().cuda_stream)
            assert st == 0, qg.qg_strerror(st)
            torch.cuda.synchronize()
            y, am = y.cpu().numpy(), am.cpu().numpy()
            # the same kernel and geometry as the workspace call: the same bits
            assert np.array_equal(y.view(np.uint32), y_ws.view(np.uint32)), (fmt, ntok, call)
            assert np.array_equal(am, am_ws), (fmt, ntok, call)
            # and the oracle
            err = np.abs(y.astype(np.float64) - ref[:ntok]) / den[:ntok]
            assert err.max() <= TOL, (fmt, ntok, call, err.max())
            for t in range(ntok):
                if gap[t] >= GAP:
                    assert am[t] == ref_am[t], (fmt, ntok, call, t)
                else:
                    assert ref[t, am[t]] >= ref[t].max() - GAP, (fmt, ntok, call, t)


def test_noalloc_refuses_a_launch_larger_than_its_scratch():
    dev = torch.device("cuda:0")
    n_out, n_in = 200000, 256            # small rows: 8 one-warp CTAs fit on every SM
    packed = torch.zeros(qg.qg_packed_bytes("q8_0", n_out, n_in), dtype=torch.uint8, device=dev)
    xd = torch.zeros((4, n_in), dtype=torch.float32, device=dev)
    am = torch.zeros(4, dtype=torch.int32, device=dev)
    qg.qg_set_tile_override("warps=1,ctas=8,rpw=1,depth=2")      # 8 CTAs per SM
    grid = int(qg.qg_describe_tile("q8_0", n_out, n_in, 4).split("grid=")[1])
    if grid <= 1024:
        pytest.skip(f"this device runs that geometry on {grid} CTAs, within the scratch's 1024")
    with pytest.raises(qg.QGError) as e:
        qg.qgemv_argmax_noalloc("q8_0", packed, n_out, n_in, xd, None, am, 4)
    assert e.value.status == -4
