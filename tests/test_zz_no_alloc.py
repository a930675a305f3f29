"""The no-allocation LM-head entry point, through the C ABI, against the
workspace entry point.

qgemv_argmax_noalloc serves callers that cannot call cudaMalloc (a plugin whose
host framework owns all device memory, or a decode loop that must never touch
the allocator): its scratch is a fixed array inside the library.  Two calls in
a row must agree with qgemv_argmax (same kernel, caller-owned workspace) within
the parity tolerance, and the argmax must be identical.  This file is
collected last so that a stop at its first failure has run every other test.
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
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
    lib = qg.load_library()
    for ntok in (4, 1):
        ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, ntok), dtype=torch.uint8, device=dev)
        y_ref = torch.empty((ntok, n_out), dtype=torch.float32, device=dev)
        am_ref = torch.empty(ntok, dtype=torch.int32, device=dev)
        qg.qgemv_argmax(fmt, packed, n_out, n_in, xd, y_ref, am_ref, ws, ntok)
        torch.cuda.synchronize()
        for call in range(2):
            y = torch.full((ntok, n_out), float("nan"), dtype=torch.float32, device=dev)
            am = torch.full((ntok,), -9, dtype=torch.int32, device=dev)
            st = lib.qgemv_argmax_noalloc(qg.FORMATS[fmt], packed.data_ptr(), n_out, n_in, xd.data_ptr(),
                                          y.data_ptr(), am.data_ptr(), ntok,
                                          torch.cuda.current_stream().cuda_stream)
            assert st == 0, qg.qg_strerror(st)
            torch.cuda.synchronize()
            err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref.cpu().numpy()) / den[:ntok]
            assert err.max() <= TOL, (fmt, ntok, call, err.max())
            assert np.array_equal(am.cpu().numpy(), am_ref.cpu().numpy()), (fmt, ntok, call)


def test_noalloc_refuses_a_launch_larger_than_its_scratch():
    dev = torch.device("cuda:0")
    n_out, n_in = 200000, 256            # small rows: 8 one-warp CTAs fit on every SM
    packed = torch.zeros(qg.qg_packed_bytes("q8_0", n_out, n_in), dtype=torch.uint8, device=dev)
    xd = torch.zeros((4, n_in), dtype=torch.float32, device=dev)
    am = torch.zeros(4, dtype=torch.int32, device=dev)
    qg.qg_set_tile_override("warps=1,ctas=8,rpw=1,depth=2")      # 8 CTAs per SM: more than 1024 CTAs
    assert int(qg.qg_describe_tile("q8_0", n_out, n_in, 4).split("grid=")[1]) > 1024
    with pytest.raises(qg.QGError) as e:
        qg.qgemv_argmax_noalloc("q8_0", packed, n_out, n_in, xd, None, am, 4)
    assert e.value.status == -4
