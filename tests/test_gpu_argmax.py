"""GPU parity of the fused LM-head argmax (qgemv_argmax) against the fp64 oracle.

The argmax must equal the oracle's first-index argmax bit for bit whenever the
oracle's top-2 gap is at least 1e-4 (absolute); below that, the GPU's id must
be one of the oracle's ids within 1e-4 of the maximum.  Independently of the
oracle, the GPU argmax must be the first-index argmax of the GPU's own logits,
and those logits must be bitwise the ones qgemv writes.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle as ORC
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import block_quantized_token_format_gb300 as qg  # noqa: E402

GAP = 1e-4
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_tile_override(None)


def dev():
    return torch.device("cuda:0")


def new_workspace(n_out, ntok=4):
    return torch.zeros(qg.qgemv_argmax_workspace_bytes(n_out, ntok), dtype=torch.uint8, device=dev())


def run_argmax(fmt, packed, n_out, n_in, x, ws, write_logits=True):
    ntok = x.shape[0]
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev())
    y = torch.full((ntok, n_out), float("nan"), dtype=torch.float32, device=dev()) if write_logits else None
    am = torch.full((ntok,), -7, dtype=torch.int32, device=dev())
    qg.qgemv_argmax(fmt, packed, n_out, n_in, xd, y, am, ws, ntok)
    torch.cuda.synchronize()
    return (y.cpu().numpy() if write_logits else None), am.cpu().numpy()


def run_qgemv(fmt, packed, n_out, n_in, x):
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev())
    y = torch.empty((x.shape[0], n_out), dtype=torch.float32, device=dev())
    qg.qgemv(fmt, packed, n_out, n_in, xd, y, x.shape[0])
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check_argmax(am, ref, what):
    ref_am = ORC.argmax_first(ref)
    gap = ORC.top2_gap(ref)
    for t in range(ref.shape[0]):
        if gap[t] >= GAP:
            assert am[t] == ref_am[t], f"{what} token {t}: {am[t]} != {ref_am[t]} (gap {gap[t]:.3g})"
        else:
            near = np.nonzero(ref[t] >= ref[t].max() - GAP)[0]
            assert am[t] in near, f"{what} token {t}: {am[t]} not within 1e-4 of the max"


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0", "affine4_g64", "bf16"])
@pytest.mark.parametrize("n_out", [1, 2, 33, 5000, 70001])
def test_argmax_small(fmt, n_out):
    n_in = 5120 if fmt == "affine4_g64" else 2560
    W = workloads.gaussian(n_out + 17, (n_out, n_in), 0.02)
    x = workloads.activations(n_out, n_in, 4)
    canon = ORC.quantize(fmt, W)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n_out, n_in)).to(dev())
    ref = ORC.gemv(fmt, canon, n_out, n_in, x)
    ws = new_workspace(n_out)
    for ntok in (1, 2, 3, 4):
        y, am = run_argmax(fmt, packed, n_out, n_in, x[:ntok], ws)
        assert np.array_equal(am, ORC.argmax_first(y)), "argmax of its own logits"
        assert np.array_equal(y.view(np.uint32), run_qgemv(fmt, packed, n_out, n_in, x[:ntok]).view(np.uint32))
        check_argmax(am, ref[:ntok], f"{fmt} n_out={n_out} ntok={ntok}")
        _, am2 = run_argmax(fmt, packed, n_out, n_in, x[:ntok], ws, write_logits=False)
        assert np.array_equal(am, am2)


def test_planted_max_and_ties():
    n_out, n_in = 40000, 2560
    x = workloads.activations(3, n_in, 4)
    W = workloads.gaussian(4, (n_out, n_in), 0.02)
    W[31337] = np.float32(0.06) * np.sign(x[0])           # unique max for token 0
    W[123] = np.float32(0.06) * np.sign(x[1])             # unique max for token 1
    W[39999] = np.float32(0.06) * np.sign(x[2])           # last row wins token 2
    W[7000] = W[21000] = W[35000] = np.float32(0.06) * np.sign(x[3])   # exact 3-way tie: lowest wins
    canon = ORC.quantize("q8_0", W)
    packed = torch.from_numpy(qg.qg_to_device_layout("q8_0", canon, n_out, n_in)).to(dev())
    ws = new_workspace(n_out)
    y, am = run_argmax("q8_0", packed, n_out, n_in, x, ws)
    assert list(am) == [31337, 123, 39999, 7000]
    assert y[3, 7000] == y[3, 21000] == y[3, 35000]


def test_workspace_reuse_across_calls_and_ntok():
    n_out, n_in = 9000, 2560
    W = workloads.gaussian(5, (n_out, n_in), 0.02)
    x = workloads.activations(5, n_in, 4)
    canon = ORC.quantize("q8_0", W)
    packed = torch.from_numpy(qg.qg_to_device_layout("q8_0", canon, n_out, n_in)).to(dev())
    ref = ORC.gemv("q8_0", canon, n_out, n_in, x)
    ws = new_workspace(n_out)
    for rep in range(3):
        for ntok in (4, 1, 3, 2):
            _, am = run_argmax("q8_0", packed, n_out, n_in, x[:ntok], ws, write_logits=(rep % 2 == 0))
            check_argmax(am, ref[:ntok], f"rep {rep} ntok {ntok}")
    ticket = ws[:4].view(torch.int32).cpu().item()
    assert ticket == 0


def _oracle_full(w, x, threads=16):
    """Oracle logits of a whole head, quantized chunk by chunk by the oracle itself, and the
    head's device bytes as the library's packer (qg_pack, the call the benchmark packs with)
    writes them.  Every chunk's packer bytes must equal the oracle's bytes carried into the
    device layout, so the bytes the kernel reads here are the tested bytes and the benched ones."""
    n_chunks = (w.n_out + workloads.ROW_CHUNK - 1) // workloads.ROW_CHUNK

    def one(c):
        Wc = workloads.weight_chunk(w.seed, w.n_out, w.n_in, c)
        canon = ORC.quantize(w.fmt, Wc)
        rows = Wc.shape[0]
        from_oracle = qg.qg_to_device_layout(w.fmt, canon, rows, w.n_in)
        packed = qg.qg_pack(w.fmt, Wc)
        same = np.array_equal(packed, from_oracle)
        return (c, same, packed, ORC.gemv(w.fmt, canon, rows, w.n_in, x), ORC.gemv_abs(w.fmt, canon, rows, w.n_in, x))

    ys, dens, packed = [None] * n_chunks, [None] * n_chunks, [None] * n_chunks
    with ThreadPoolExecutor(threads) as ex:
        for c, same, pk, y, den in ex.map(one, range(n_chunks)):
            assert same, f"{w.name}: qg_pack bytes differ from the oracle's in row chunk {c}"
            ys[c], dens[c], packed[c] = y, den, pk
    return np.concatenate(ys, axis=1), np.concatenate(dens, axis=1), np.concatenate(packed)


@pytest.mark.parametrize("name", ["q8_0_head_248320x2560", "affine4_head_248320x5120"])
def test_full_lm_head(name):
    w = workloads.WORKLOADS[name]
    x = workloads.activations(w.seed, w.n_in, 4)
    ref, den, packed_np = _oracle_full(w, x)
    packed = torch.from_numpy(packed_np).to(dev())
    ws = new_workspace(w.n_out)
    worst = 0.0
    for ntok in (1, 2, 3, 4):
        y, am = run_argmax(w.fmt, packed, w.n_out, w.n_in, x[:ntok], ws)
        rel = np.abs(y.astype(np.float64) - ref[:ntok]) / den[:ntok]
        worst = max(worst, float(rel.max()))
        assert rel.max() <= TOL, f"{name} ntok={ntok}: {rel.max():.3g}"
        assert np.array_equal(am, ORC.argmax_first(y))
        check_argmax(am, ref[:ntok], f"{name} ntok={ntok}")
    # the drafted vocabulary: the first 106299 rows of the same packed head
    if w.fmt == "q8_0":
        n_draft = workloads.WORKLOADS["q8_0_head_106299x2560"].n_out
        for ntok in (1, 4):
            y, am = run_argmax(w.fmt, packed, n_draft, w.n_in, x[:ntok], ws)
            check_argmax(am, ref[:ntok, :n_draft], f"draft ntok={ntok}")
    print(f"{name}: max normalised error {worst:.3g}, argmax {am}")


def _nan_scales(fmt, canon, n_out, n_in, rows):
    """Canonical bytes with every block scale of `rows` set to an fp16 NaN (0x7E00)."""
    c = canon.copy()
    if fmt == "q8_0":
        rb = n_in // 32 * 34
        for r in rows:
            for b in range(n_in // 32):
                c[r * rb + 34 * b:r * rb + 34 * b + 2] = (0x00, 0x7E)
    elif fmt == "affine4_g64":
        scales = c[n_out * n_in // 2:n_out * n_in // 2 + n_out * n_in // 32].view(np.uint16).reshape(n_out, -1)
        for r in rows:
            scales[r, :] = 0x7E00
    else:
        raise ValueError(fmt)
    return c


@pytest.mark.parametrize("fmt", ["q8_0", "affine4_g64"])
def test_nan_rows_never_win(fmt):
    """A row whose block scales are NaN has NaN logits and never wins the argmax, even when
    its finite counterpart would be the largest logit of every token."""
    n_out, n_in = 5003, 2560
    x = workloads.activations(21, n_in, 4)
    W = workloads.gaussian(21, (n_out, n_in), 0.02)
    W[1234] = 0.2 * np.sign(x[0])            # the winner of token 0 while its scales are finite
    W[77] = 0.2 * np.sign(x[3])              # the winner of token 3
    canon = ORC.quantize(fmt, W)
    nan_rows = [0, 1234, n_out - 1]
    bad = _nan_scales(fmt, canon, n_out, n_in, nan_rows)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, bad, n_out, n_in)).to(dev())
    ref = ORC.gemv(fmt, bad, n_out, n_in, x)
    den = ORC.gemv_abs(fmt, bad, n_out, n_in, x)
    assert np.isnan(ref[:, nan_rows]).all()
    ws = new_workspace(n_out)
    for ntok in (1, 4):
        y, am = run_argmax(fmt, packed, n_out, n_in, x[:ntok], ws)
        assert np.isnan(y[:, nan_rows]).all()
        fin = np.setdiff1d(np.arange(n_out), nan_rows)
        rel = np.abs(y[:, fin].astype(np.float64) - ref[:ntok, fin]) / den[:ntok, fin]
        assert rel.max() <= TOL
        assert not np.isin(am, nan_rows).any(), am
        assert np.array_equal(am, ORC.argmax_first(y))
        check_argmax(am, np.where(np.isnan(ref[:ntok]), -np.inf, ref[:ntok]), f"{fmt} NaN rows ntok={ntok}")
        if ntok == 4:
            assert am[3] == 77
        _, am2 = run_argmax(fmt, packed, n_out, n_in, x[:ntok], ws, write_logits=False)
        assert np.array_equal(am2, am)


@pytest.mark.parametrize("fmt", ["q8_0", "affine4_g64"])
def test_all_nan_logits_give_minus_one(fmt):
    n_out, n_in = 3001, 2560
    x = workloads.activations(22, n_in, 4)
    canon = ORC.quantize(fmt, workloads.gaussian(22, (n_out, n_in), 0.02))
    bad = _nan_scales(fmt, canon, n_out, n_in, range(n_out))
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, bad, n_out, n_in)).to(dev())
    ws = new_workspace(n_out)
    for ntok in (1, 3, 4):
        y, am = run_argmax(fmt, packed, n_out, n_in, x[:ntok], ws)
        assert np.isnan(y).all()
        assert (am == -1).all(), am
        _, am2 = run_argmax(fmt, packed, n_out, n_in, x[:ntok], ws, write_logits=False)
        assert (am2 == -1).all(), am2
