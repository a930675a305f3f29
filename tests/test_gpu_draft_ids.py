"""GPU parity of the id-list draft head: qg_gather_rows + qgemv_argmax_ids.

The drafter scores only a listed subset of the LM head's rows, copied once into a
small head ("Where the time goes on an M2 Max", MTP draft vocabulary subset), and
maps its argmax back to full-vocabulary ids (the drafter issue's Phase 2b d2t map).
Checked against the fp64 oracle: the gathered head's bytes are the listed rows of
the packed head; its logits match the oracle within 1e-3 of sum |w x|; the argmax
id equals ids[first-index argmax] of the oracle (bit for bit when the oracle's top-2
gap is >= 1e-4, else within the near-max set) and of the GPU's own logits.
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
FMTS = ["q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_tile_override(None)


def dev():
    return torch.device("cuda:0")


def n_in_for(fmt, base):
    m = {"q8_0": 32, "q4_0": 32, "affine4_g64": 64, "bf16": 16, "q5_0": 32}[fmt]
    return max(m, base // m * m)


def gather(fmt, packed, n_out, n_in, ids):
    idd = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev())
    out = torch.full((qg.qg_packed_bytes(fmt, len(ids), n_in),), 0xA5, dtype=torch.uint8, device=dev())
    qg.qg_gather_rows(fmt, packed, n_out, n_in, idd, out)
    torch.cuda.synchronize()
    return out, idd


def argmax_ids(fmt, small, n_sub, n_in, x, idd):
    ntok = x.shape[0]
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev())
    y = torch.full((ntok, n_sub), float("nan"), dtype=torch.float32, device=dev())
    am = torch.full((ntok,), -7, dtype=torch.int32, device=dev())
    ws = torch.zeros(qg.qgemv_argmax_workspace_bytes(n_sub, ntok), dtype=torch.uint8, device=dev())
    qg.qgemv_argmax_ids(fmt, small, n_sub, n_in, xd, y, am, idd, ws, ntok)
    torch.cuda.synchronize()
    return y.cpu().numpy(), am.cpu().numpy()


def check_ids_argmax(am, ref, ids, what):
    ref_j = ORC.argmax_first(ref)
    gap = ORC.top2_gap(ref)
    for t in range(ref.shape[0]):
        if gap[t] >= GAP:
            assert am[t] == ids[ref_j[t]], f"{what} token {t}: {am[t]} != {ids[ref_j[t]]} (gap {gap[t]:.3g})"
        else:
            near = set(int(v) for v in ids[np.nonzero(ref[t] >= ref[t].max() - GAP)[0]])
            assert int(am[t]) in near, f"{what} token {t}: {am[t]} not within 1e-4 of the max"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_out,n_in_base", [(97, 320), (3001, 2560), (1000, 6144)])
def test_gather_is_the_listed_rows(fmt, n_out, n_in_base):
    n_in = n_in_for(fmt, n_in_base)
    W = workloads.gaussian(n_out + 5 * n_in, (n_out, n_in), 0.02)
    packed_np = qg.qg_to_device_layout(fmt, ORC.quantize(fmt, W), n_out, n_in)
    packed = torch.from_numpy(packed_np).to(dev())
    g = np.random.default_rng(n_out)
    ids = np.concatenate([[n_out - 1, 0], g.integers(0, n_out, size=2 * n_out // 3), [n_out - 1]]).astype(np.int32)
    out, _ = gather(fmt, packed, n_out, n_in, ids)
    stride = qg.qg_row_stride(fmt, n_in)
    expect = packed_np.reshape(n_out, stride)[ids].reshape(-1)
    assert np.array_equal(out.cpu().numpy(), expect)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_argmax_ids_matches_oracle(fmt):
    n_out, n_in = 5000, (5120 if fmt == "affine4_g64" else 2560)
    W = workloads.gaussian(77, (n_out, n_in), 0.02)
    x = workloads.activations(77, n_in, 4)
    W[4321] = np.float32(0.06) * np.sign(x[2])          # token 2's maximum: in the list
    W[17] = np.float32(0.07) * np.sign(x[3])            # token 3's overall maximum: not listed
    canon = ORC.quantize(fmt, W)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n_out, n_in)).to(dev())
    ids = np.random.default_rng(9).permutation(n_out)[:1777].astype(np.int32)   # unsorted
    ids = ids[ids != 17]
    ids[5] = 4321
    small, idd = gather(fmt, packed, n_out, n_in, ids)
    ref, ref_am = ORC.qgemv_argmax_ids(fmt, canon, n_out, n_in, x, ids)
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x, rows=ids)
    for ntok in (1, 2, 3, 4):
        y, am = argmax_ids(fmt, small, ids.size, n_in, x[:ntok], idd)
        rel = np.abs(y.astype(np.float64) - ref[:ntok]) / den[:ntok]
        assert rel.max() <= TOL, f"{fmt} ntok={ntok}: {rel.max():.3g}"
        assert np.array_equal(am, ids[ORC.argmax_first(y)]), "ids of the argmax of its own logits"
        check_ids_argmax(am, ref[:ntok], ids, f"{fmt} ntok={ntok}")
        if ntok >= 3:
            assert am[2] == 4321 and am[2] == ref_am[2]
        if ntok == 4:
            assert am[3] != 17


def test_bad_id_gives_zero_row_and_status():
    fmt, n_out, n_in = "q8_0", 64, 256
    W = workloads.gaussian(3, (n_out, n_in), 0.02)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, ORC.quantize(fmt, W), n_out, n_in)).to(dev())
    qg.qg_device_status()                                   # start clean
    out, _ = gather(fmt, packed, n_out, n_in, np.array([5, n_out, -1, 7], dtype=np.int32))
    stride = qg.qg_row_stride(fmt, n_in)
    rows = out.cpu().numpy().reshape(4, stride)
    assert not rows[1].any() and not rows[2].any()
    assert rows[0].any() and rows[3].any()
    assert qg.qg_device_status() == qg.QG_DEVICE_BAD_ROW_ID
    assert qg.qg_device_status() == 0                       # cleared by the read


def _packed_head(w, threads=16):
    n_chunks = (w.n_out + workloads.ROW_CHUNK - 1) // workloads.ROW_CHUNK
    stride = qg.qg_row_stride(w.fmt, w.n_in)
    out = np.empty(w.n_out * stride, dtype=np.uint8)

    def one(c):
        Wc = workloads.weight_chunk(w.seed, w.n_out, w.n_in, c)
        r0 = c * workloads.ROW_CHUNK
        qg.qg_pack(w.fmt, Wc, out=out[r0 * stride:(r0 + Wc.shape[0]) * stride])

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(n_chunks)))
    return out


def test_full_head_with_the_draft_id_list():
    """248,320-row Q8_0 head, the seeded 106,299-id draft list: the oracle quantizes
    only the listed rows (quantization is row-local) and scores them."""
    name = "q8_0_head_248320x2560"
    w = workloads.WORKLOADS[name]
    k, seed = workloads.DRAFT_IDS[name]
    ids = workloads.draft_ids(seed, w.n_out, k)
    x = workloads.activations(w.seed, w.n_in, 4)
    packed = torch.from_numpy(_packed_head(w)).to(dev())
    small, idd = gather(w.fmt, packed, w.n_out, w.n_in, ids)
    canon_small = ORC.quantize(w.fmt, workloads.weight_rows(w.seed, w.n_out, w.n_in, ids))
    ref = ORC.gemv(w.fmt, canon_small, k, w.n_in, x)
    den = ORC.gemv_abs(w.fmt, canon_small, k, w.n_in, x)
    for ntok in (1, 4):
        y, am = argmax_ids(w.fmt, small, k, w.n_in, x[:ntok], idd)
        rel = np.abs(y.astype(np.float64) - ref[:ntok]) / den[:ntok]
        assert rel.max() <= TOL, f"ntok={ntok}: {rel.max():.3g}"
        check_ids_argmax(am, ref[:ntok], ids, f"draft ids ntok={ntok}")
    assert qg.qg_device_status() == 0
