"""Failure detection on the GPU without a GPU fault.

Every mbarrier wait in the kernels is bounded.  The test hook makes the first
wait of every warp impossible to satisfy (extra expected bytes that no copy
delivers) with a short poll limit: the kernel must give up, set the device
status word, drain its copies and exit normally; the host reads the status;
the context stays usable and the next call is correct again.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle as ORC
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import block_quantized_token_format_gb300 as qg  # noqa: E402


@pytest.fixture(autouse=True)
def _restore():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_wait_limit(0, 0)
    qg.qg_device_status(clear=True)
    yield
    qg.qg_set_wait_limit(0, 0)
    qg.qg_device_status(clear=True)


def test_bounded_wait_times_out_and_reports():
    n_out, n_in = 4000, 2560
    W = workloads.gaussian(1, (n_out, n_in), 0.02)
    x = workloads.activations(1, n_in, 2)
    canon = ORC.quantize("q8_0", W)
    dev = torch.device("cuda:0")
    packed = torch.from_numpy(qg.qg_to_device_layout("q8_0", canon, n_out, n_in)).to(dev)
    xd = torch.from_numpy(x).to(dev)
    y = torch.zeros((2, n_out), dtype=torch.float32, device=dev)
    assert qg.qg_device_status(clear=True) == 0

    qg.qg_set_wait_limit(2000, 16)
    qg.qgemv("q8_0", packed, n_out, n_in, xd, y, 2)
    torch.cuda.synchronize()                     # returns: the kernel exited on its own
    assert qg.qg_device_status(clear=True) & qg.QG_DEVICE_WAIT_TIMEOUT

    qg.qg_set_wait_limit(0, 0)
    qg.qgemv("q8_0", packed, n_out, n_in, xd, y, 2)
    torch.cuda.synchronize()
    assert qg.qg_device_status(clear=True) == 0
    ref = ORC.gemv("q8_0", canon, n_out, n_in, x)
    den = ORC.gemv_abs("q8_0", canon, n_out, n_in, x)
    assert np.max(np.abs(y.cpu().numpy() - ref) / den) <= 1e-3


def test_argmax_kernel_times_out_cleanly_and_workspace_survives():
    n_out, n_in = 3000, 2560
    W = workloads.gaussian(2, (n_out, n_in), 0.02)
    x = workloads.activations(2, n_in, 1)
    canon = ORC.quantize("q8_0", W)
    dev = torch.device("cuda:0")
    packed = torch.from_numpy(qg.qg_to_device_layout("q8_0", canon, n_out, n_in)).to(dev)
    xd = torch.from_numpy(x).to(dev)
    ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, 1), dtype=torch.uint8, device=dev)
    am = torch.zeros(1, dtype=torch.int32, device=dev)
    qg.qg_set_wait_limit(2000, 16)
    qg.qgemv_argmax("q8_0", packed, n_out, n_in, xd, None, am, ws, 1)
    torch.cuda.synchronize()
    assert qg.qg_device_status(clear=True) & qg.QG_DEVICE_WAIT_TIMEOUT
    assert ws[:4].view(torch.int32).cpu().item() == 0          # the ticket still resets
    qg.qg_set_wait_limit(0, 0)
    qg.qgemv_argmax("q8_0", packed, n_out, n_in, xd, None, am, ws, 1)
    torch.cuda.synchronize()
    ref = ORC.gemv("q8_0", canon, n_out, n_in, x)
    assert am.cpu().item() == ORC.argmax_first(ref)[0]
