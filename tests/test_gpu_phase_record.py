"""GPU: the profiling hook qg_set_phase_record.  With the hook on, a mat-vec call gives
bitwise the same outputs as with it off, and every CTA of the launch leaves ordered
stamps: global entry <= exit, an SM id below the SM count, and SM-clock phases in the
order the kernel passes them (copies issued, wait done, x staged, warp 0 done, CTA
done)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as ORC
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import block_quantized_token_format_gb300 as qg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_phase_record(None)
    qg.qg_set_tile_override(None)
    yield
    qg.qg_set_phase_record(None)


@pytest.mark.parametrize("fmt,n_out,n_in,argmax", [("q8_0", 3000, 2560, False), ("affine4_g64", 2000, 5120, True)])
def test_phase_stamps_ordered_and_results_unchanged(fmt, n_out, n_in, argmax):
    dev = torch.device("cuda:0")
    W = workloads.gaussian(91, (n_out, n_in), 0.02)
    x = torch.from_numpy(workloads.activations(92, n_in, 4)).to(dev)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, ORC.quantize(fmt, W), n_out, n_in)).to(dev)
    ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, 4), dtype=torch.uint8, device=dev)

    def run():
        y = torch.full((4, n_out), float("nan"), dtype=torch.float32, device=dev)
        am = torch.full((4,), -7, dtype=torch.int32, device=dev)
        if argmax:
            qg.qgemv_argmax(fmt, packed, n_out, n_in, x, y, am, ws, 4)
        else:
            qg.qgemv(fmt, packed, n_out, n_in, x, y, 4)
        torch.cuda.synchronize()
        return y.cpu().numpy(), am.cpu().numpy()

    y0, a0 = run()
    buf = torch.zeros(2 * qg.QG_PHASE_SLOT_WORDS, dtype=torch.int64, device=dev)
    qg.qg_set_phase_record(buf, 2)
    try:
        y1, a1 = run()
    finally:
        qg.qg_set_phase_record(None)
    y2, a2 = run()
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    assert np.array_equal(y0.view(np.uint32), y2.view(np.uint32))
    if argmax:
        assert np.array_equal(a0, a1) and np.array_equal(a0, a2)

    grid = int(qg.qg_describe_tile(fmt, n_out, n_in, 4).split("grid=")[1])
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rec = buf.view(2, -1)[0, :grid * qg.QG_PHASE_WORDS].reshape(grid, qg.QG_PHASE_WORDS).cpu().numpy()
    assert not np.any(buf.view(2, -1)[1].cpu().numpy()), "one launch fills one slot"
    t_in, t_out, smid = rec[:, 0], rec[:, 1], rec[:, 2]
    assert np.all(t_in > 0) and np.all(t_out >= t_in)
    assert np.all(smid < sms)
    clk = rec[:, 3:9].astype(np.int64)
    rel = (clk - clk[:, 3:4]) % (1 << 32)          # relative to the entry clock (word 6)
    order = rel[:, [0, 1, 2, 4, 5]]                 # issued, wait, x staged, warp 0 done, CTA done
    assert np.all(np.diff(order, axis=1) >= 0), order[:4]
    assert np.all(rel[:, 5] < (1 << 31))            # a CTA of this size ends within ~1 s of SM clock
