"""Programmatic dependent launch (QG_LAUNCH_EARLY_START): a kernel may start its
weight copies before the previous kernel in the stream finishes, but must wait
for it before reading x or writing y / argmax / the workspace.

Checked with real dependencies: a chain of square mat-vecs where each call's
x is the previous call's y, and back-to-back fused-argmax calls sharing one
workspace; results must be bitwise those of ordinary launches.
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
def _reset():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_launch_options(0)
    yield
    qg.qg_set_launch_options(0)


def _chain(fmt, packed, n, x0, steps, ntok):
    dev = torch.device("cuda:0")
    bufs = [torch.from_numpy(np.ascontiguousarray(x0[:ntok])).to(dev)]
    for _ in range(steps):
        bufs.append(torch.empty((ntok, n), dtype=torch.float32, device=dev))
    for k in range(steps):
        qg.qgemv(fmt, packed, n, n, bufs[k], bufs[k + 1], ntok)
        # keep magnitudes bounded: scale in place on the same stream (a dependent kernel)
        bufs[k + 1].mul_(1.0 / float(np.sqrt(n) * 0.02))
    torch.cuda.synchronize()
    return [b.cpu().numpy() for b in bufs[1:]]


@pytest.mark.parametrize("fmt", ["q8_0", "affine4_g64"])
def test_dependent_chain_matches_plain_launches(fmt):
    n = 2560 if fmt == "q8_0" else 5120
    W = workloads.gaussian(3, (n, n), 0.02)
    canon = ORC.quantize(fmt, W)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n, n)).to(torch.device("cuda:0"))
    x0 = workloads.activations(3, n, 4)
    for ntok in (1, 4):
        qg.qg_set_launch_options(0)
        plain = _chain(fmt, packed, n, x0, 12, ntok)
        qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
        early = _chain(fmt, packed, n, x0, 12, ntok)
        for a, b in zip(plain, early):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        # and the first link against the oracle
        ref = ORC.gemv(fmt, canon, n, n, x0[:ntok]) / (np.sqrt(n) * 0.02)
        den = ORC.gemv_abs(fmt, canon, n, n, x0[:ntok]) / (np.sqrt(n) * 0.02)
        assert np.max(np.abs(early[0] - ref) / den) <= 1e-3


def test_back_to_back_argmax_on_one_workspace():
    dev = torch.device("cuda:0")
    n_out, n_in = 50000, 2560
    W = workloads.gaussian(4, (n_out, n_in), 0.02)
    canon = ORC.quantize("q8_0", W)
    packed = torch.from_numpy(qg.qg_to_device_layout("q8_0", canon, n_out, n_in)).to(dev)
    xs = [workloads.gaussian(100 + k, (4, n_in)) for k in range(6)]
    ref = [ORC.argmax_first(ORC.gemv("q8_0", canon, n_out, n_in, x)) for x in xs]
    ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, 4), dtype=torch.uint8, device=dev)
    qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
    xd = [torch.from_numpy(x).to(dev) for x in xs]
    outs = [torch.empty(4, dtype=torch.int32, device=dev) for _ in xs]
    for rep in range(3):
        for k in range(len(xs)):
            qg.qgemv_argmax("q8_0", packed, n_out, n_in, xd[k], None, outs[k], ws, 4)
        torch.cuda.synchronize()
        for k in range(len(xs)):
            assert np.array_equal(outs[k].cpu().numpy(), ref[k]), (rep, k)
    assert ws[:4].view(torch.int32).cpu().item() == 0
