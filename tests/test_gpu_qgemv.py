"""GPU parity: the CUDA mat-vec (through the C ABI) against the fp64 oracle.

Acceptance (per output): |y_gpu - y_ref| <= 1e-3 * sum_i |deq(W)[o,i] * x[t,i]|,
the denominator in fp64 from the oracle; all-zero rows give exactly 0.
fp32 accumulation over n_in <= 6144 terms stays well inside this bound.
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
FMTS = ["q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_tile_override(None)
    yield
    qg.qg_set_tile_override(None)


def dev():
    return torch.device("cuda:0")


def upload(fmt, canon, n_out, n_in):
    return torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n_out, n_in)).to(dev())


def gpu_qgemv(fmt, packed, n_out, n_in, x):
    ntok = x.shape[0]
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev())
    y = torch.full((ntok, n_out), float("nan"), dtype=torch.float32, device=dev())
    qg.qgemv(fmt, packed, n_out, n_in, xd, y, ntok)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check_close(y, ref, den, what=""):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), what
    zero = den == 0
    assert np.all(y[zero] == 0), what
    rel = np.abs(y[~zero] - ref[~zero]) / den[~zero]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= TOL, f"{what}: max normalised error {worst:.3g}"
    return worst


def n_in_for(fmt, base):
    m = {"q8_0": 32, "q4_0": 32, "affine4_g64": 64, "bf16": 16, "q5_0": 32}[fmt]
    return max(m, base // m * m)


# ----------------------------------------------------------------------------- small shapes, ragged tails

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_out,n_in_base", [(1, 64), (7, 128), (97, 320), (1000, 1088), (2561, 2560), (333, 6144)])
def test_small_shapes(fmt, n_out, n_in_base):
    n_in = n_in_for(fmt, n_in_base)
    W = workloads.gaussian(n_out * 7 + n_in, (n_out, n_in), 0.02)
    if n_out > 3:
        W[2] = 0.0
    x = workloads.gaussian(n_out + n_in, (4, n_in))
    canon = ORC.quantize(fmt, W)
    packed = upload(fmt, canon, n_out, n_in)
    ref = ORC.gemv(fmt, canon, n_out, n_in, x)
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
    for ntok in (1, 2, 3, 4):
        y = gpu_qgemv(fmt, packed, n_out, n_in, x[:ntok])
        check_close(y, ref[:ntok], den[:ntok], f"{fmt} {n_out}x{n_in} ntok={ntok}")


# ----------------------------------------------------------------------------- workload shapes, full oracle

SMALL_WORKLOADS = ["q8_0_2560x2560", "q8_0_6144x2560", "q8_0_10240x2560", "q8_0_12288x2560",
                   "q8_0_2560x6144", "q4_0_8192x2560", "bf16_8192x2560", "q5_0_8192x2560"]


@pytest.mark.parametrize("name", SMALL_WORKLOADS)
def test_workload_full(name):
    w = workloads.WORKLOADS[name]
    W = workloads.weights(w.seed, w.n_out, w.n_in)
    x = workloads.activations(w.seed, w.n_in, 4)
    canon = ORC.quantize(w.fmt, W)
    assert np.array_equal(qg.qg_quantize(w.fmt, W), canon)      # the packer's bytes are the oracle's
    packed = upload(w.fmt, canon, w.n_out, w.n_in)
    ref = ORC.gemv(w.fmt, canon, w.n_out, w.n_in, x)
    den = ORC.gemv_abs(w.fmt, canon, w.n_out, w.n_in, x)
    worst = 0.0
    for ntok in (1, 2, 3, 4):
        y = gpu_qgemv(w.fmt, packed, w.n_out, w.n_in, x[:ntok])
        worst = max(worst, check_close(y, ref[:ntok], den[:ntok], f"{name} ntok={ntok}"))
    print(f"{name}: max normalised error {worst:.3g}")


# ----------------------------------------------------------------------------- activations with outliers

IDP_FMTS = ["q8_0", "q4_0", "affine4_g64", "q5_0"]      # x staged as 16-bit integers per chunk


@pytest.mark.parametrize("fmt", FMTS)
def test_outlier_activations(fmt):
    """x shaped like a transformer hidden state: three massive channels (300..3000 against
    N(0,1)) and eight moderate ones (10..40), at 1e-3 like every other case."""
    n_out, n_in = 3000, n_in_for(fmt, 2560 if fmt != "affine4_g64" else 5120)
    W = workloads.gaussian(71, (n_out, n_in), 0.02)
    canon = ORC.quantize(fmt, W)
    packed = upload(fmt, canon, n_out, n_in)
    worst = 0.0
    for seed in (72, 73, 74):
        x = workloads.activations_with_outliers(seed, n_in, 4)
        ref = ORC.gemv(fmt, canon, n_out, n_in, x)
        den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
        for ntok in (1, 4):
            y = gpu_qgemv(fmt, packed, n_out, n_in, x[:ntok])
            worst = max(worst, check_close(y, ref[:ntok], den[:ntok], f"{fmt} outliers seed={seed} ntok={ntok}"))
    print(f"{fmt}: max normalised error with outlier channels {worst:.3g}")


def x_rounding_bound(fmt, canon, n_out, n_in, x):
    """The stated bound of the integer chunk dot's x rounding, per output: the sum over
    chunks c (32 columns, 16 for Q8_0) of 2^-14 * max_c |x| * sum_c |v|, where v is the
    weight (Q8_0, Q4_0, Q5_0) or, for the affine format w = s q + b, the code part s q
    (the bias multiplies the exact fp32 sum of x), bounded here by 15 |s|.  Affine
    canonical bytes: n_out * n_in / 8 uint32 code words, then the fp16 scales s, then
    the fp16 biases b, one per 64 weights."""
    if fmt == "affine4_g64":
        nw, ng = n_out * n_in // 8, n_out * n_in // 64
        sc = np.asarray(canon, dtype=np.uint8)[nw * 4: nw * 4 + ng * 2].view("<f2").astype(np.float64)
        w = np.repeat(15.0 * np.abs(sc).reshape(n_out, n_in // 64), 64, axis=1)
    else:
        w = np.abs(ORC.dequantize(fmt, canon, n_out, n_in))
    cw = 16 if fmt == "q8_0" else 32
    m = np.abs(x.astype(np.float64)).reshape(x.shape[0], -1, cw).max(axis=2)      # [ntok, chunks]
    sw = w.reshape(n_out, -1, cw).sum(axis=2)                                      # [n_out, chunks]
    return 2.0 ** -14 * (m @ sw.T)


@pytest.mark.parametrize("fmt", IDP_FMTS)
def test_x_rounding_error_within_stated_bound(fmt):
    """Where the weight mass sits far below a chunk's largest |x| (one entry 1e4, the rest
    about 1e-2, the weights of the large entries zero), the x rounding can exceed 1e-3 of
    sum|w x|.  The error must still respect the stated bound: the x-rounding term plus
    2e-4 of sum|w x| for fp32 rounding."""
    n_out, n_in = 500, n_in_for(fmt, 2560)
    cw = 16 if fmt == "q8_0" else 32
    W = workloads.gaussian(81, (n_out, n_in), 0.02)
    big = np.arange(0, n_in, cw) + 5                  # one large entry per chunk
    W[:, big] = 0.0
    x = workloads.gaussian(82, (4, n_in), 1e-2)
    x[:, big] = np.float32(1e4)
    x[1, big] = np.float32(-7.5e3)
    canon = ORC.quantize(fmt, W)
    packed = upload(fmt, canon, n_out, n_in)
    ref = ORC.gemv(fmt, canon, n_out, n_in, x)
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
    bound = x_rounding_bound(fmt, canon, n_out, n_in, x) + 2e-4 * den
    y = gpu_qgemv(fmt, packed, n_out, n_in, x).astype(np.float64)
    err = np.abs(y - ref)
    assert np.all(err <= bound), (fmt, float((err / bound).max()))
    print(f"{fmt}: adversarial x, max normalised error {float((err / np.maximum(den, 1e-300)).max()):.3g}, "
          f"max error / bound {float((err / bound).max()):.3g}")


# ----------------------------------------------------------------------------- invariances

@pytest.mark.parametrize("fmt", FMTS)
def test_token_count_invariance_bitwise(fmt):
    """Row t of an ntok=k call equals the ntok=1 call on x[t], bit for bit."""
    n_out, n_in = 3001, n_in_for(fmt, 2560 if fmt != "affine4_g64" else 5120)
    W = workloads.gaussian(5, (n_out, n_in), 0.02)
    x = workloads.activations(5, n_in, 4)
    packed = upload(fmt, ORC.quantize(fmt, W), n_out, n_in)
    singles = [gpu_qgemv(fmt, packed, n_out, n_in, x[t:t + 1])[0] for t in range(4)]
    for ntok in (2, 3, 4):
        y = gpu_qgemv(fmt, packed, n_out, n_in, x[:ntok])
        for t in range(ntok):
            assert np.array_equal(y[t].view(np.uint32), singles[t].view(np.uint32)), (fmt, ntok, t)
    same = gpu_qgemv(fmt, packed, n_out, n_in, np.repeat(x[:1], 4, axis=0))
    for t in range(4):
        assert np.array_equal(same[t].view(np.uint32), singles[0].view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
def test_tile_choice_does_not_change_bits(fmt):
    """The reduction order depends only on (fmt, n_in): every geometry gives the same bits."""
    n_out, n_in = 1537, n_in_for(fmt, 2560)
    W = workloads.gaussian(8, (n_out, n_in), 0.02)
    x = workloads.activations(8, n_in, 4)
    packed = upload(fmt, ORC.quantize(fmt, W), n_out, n_in)
    qg.qg_set_tile_override(None)
    base = {ntok: gpu_qgemv(fmt, packed, n_out, n_in, x[:ntok]) for ntok in (1, 3)}
    try:
        for spec in ["rpw=1,depth=2", "rpw=1,depth=4,warps=4", "rpw=2,depth=2,warps=2,ctas=1",
                     "rpw=2,depth=8", "rpw=4,depth=3,warps=8,ctas=2", "rpw=4,depth=16,warps=1",
                     "rpw=8,depth=2", "rpw=8,depth=5,warps=4,ctas=3"]:
            qg.qg_set_tile_override(spec)
            for ntok in ((1,) if "rpw=8" in spec else (1, 3)):   # 8 rows per warp: ntok <= 2
                y = gpu_qgemv(fmt, packed, n_out, n_in, x[:ntok])
                assert np.array_equal(y.view(np.uint32), base[ntok].view(np.uint32)), (fmt, spec, ntok)
    finally:
        qg.qg_set_tile_override(None)


# (rows per warp, ntok) pairs the library instantiates
RPW_NTOKS = ({(r, t) for r in (1, 2, 4) for t in (1, 2, 3, 4)} |
             {(8, 1), (8, 2), (8, 3), (6, 2), (6, 3), (6, 4), (5, 4), (3, 4)})


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_out,n_in_base", [(1, 64), (13, 320), (1537, 2560), (64, 12288)])
def test_multi_row_boxes_ragged(fmt, n_out, n_in_base):
    """rpw = 2, 4, 8: one tensor-copy box of rpw rows per step, partly past n_out
    (zero filled) and, for rows shorter than a step or a short last step, partly
    past the row's bytes; the rows must still land one full step apart."""
    n_in = n_in_for(fmt, n_in_base)
    W = workloads.gaussian(n_out * 11 + n_in, (n_out, n_in), 0.02)
    x = workloads.gaussian(n_out + 3 * n_in, (4, n_in))
    canon = ORC.quantize(fmt, W)
    packed = upload(fmt, canon, n_out, n_in)
    ref = ORC.gemv(fmt, canon, n_out, n_in, x)
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
    try:
        for spec in ("rpw=2,depth=3,warps=1", "rpw=4,depth=2,warps=3", "rpw=8,depth=2,warps=1",
                     "rpw=8,depth=4,warps=16,ctas=1", "rpw=3,depth=2,warps=5", "rpw=5,depth=3,warps=7",
                     "rpw=6,depth=2,warps=11,ctas=2", "rpw=6,depth=2,warps=16", "rpw=8,depth=3,warps=16",
                     "rpw=1,depth=2,warps=1,split=1",
                     "rpw=2,depth=3,warps=4,split=2", "rpw=4,depth=2,warps=9,split=3",
                     "rpw=1,depth=3,warps=16,ctas=2,split=4"):
            qg.qg_set_tile_override(spec)
            rpw = int(spec.split("rpw=")[1].split(",")[0])
            for ntok in (1, 2, 3, 4):
                if (rpw, ntok) not in RPW_NTOKS:
                    continue
                y = gpu_qgemv(fmt, packed, n_out, n_in, x[:ntok])
                check_close(y, ref[:ntok], den[:ntok], f"{fmt} {n_out}x{n_in} ntok={ntok} {spec}")
        qg.qg_set_tile_override("rpw=8")
        with pytest.raises(qg.QGError) as e:       # not instantiated: refused, nothing launched
            gpu_qgemv(fmt, packed, n_out, n_in, np.repeat(x[:1], 4, axis=0))
        assert e.value.status == -3
    finally:
        qg.qg_set_tile_override(None)


@pytest.mark.parametrize("fmt", FMTS)
def test_split_is_fixed_per_shape_and_token_invariant(fmt):
    """A row's steps may be split over a team of warps.  The split is chosen from
    (fmt, n_out, n_in) only, so every ntok gives the ntok=1 bits; a forced split
    changes the addition order (close to the oracle), never correctness."""
    n_out, n_in = 777, n_in_for(fmt, 6144)
    W = workloads.gaussian(31, (n_out, n_in), 0.02)
    x = workloads.activations(31, n_in, 4)
    canon = ORC.quantize(fmt, W)
    packed = upload(fmt, canon, n_out, n_in)
    ref = ORC.gemv(fmt, canon, n_out, n_in, x)
    den = ORC.gemv_abs(fmt, canon, n_out, n_in, x)
    assert ",split=" in qg.qg_describe_tile(fmt, n_out, n_in, 1)
    splits = {qg.qg_describe_tile(fmt, n_out, n_in, t).split("split=")[1].split(",")[0] for t in (1, 2, 3, 4)}
    assert len(splits) == 1, splits
    singles = [gpu_qgemv(fmt, packed, n_out, n_in, x[t:t + 1])[0] for t in range(4)]
    y4 = gpu_qgemv(fmt, packed, n_out, n_in, x)
    for t in range(4):
        assert np.array_equal(y4[t].view(np.uint32), singles[t].view(np.uint32)), (fmt, t)
    check_close(y4, ref, den, f"{fmt} default split")
    try:
        for p in (1, 2, 3, 4):
            qg.qg_set_tile_override(f"split={p}")
            y = gpu_qgemv(fmt, packed, n_out, n_in, x)
            check_close(y, ref, den, f"{fmt} split={p}")
            y1 = gpu_qgemv(fmt, packed, n_out, n_in, x[:1])
            assert np.array_equal(y1[0].view(np.uint32), y[0].view(np.uint32)), (fmt, p)
    finally:
        qg.qg_set_tile_override(None)


def test_plan_cache_follows_the_override():
    """Launch plans are cached per thread; every override change must reach the next
    call.  A forced split changes the addition order (and so, here, some bits);
    clearing the override restores the default bits exactly."""
    fmt, n_out, n_in = "q8_0", 777, 6144          # default split 3 (12 steps a row)
    W = workloads.gaussian(41, (n_out, n_in), 0.02)
    x = workloads.activations(41, n_in, 4)
    packed = upload(fmt, ORC.quantize(fmt, W), n_out, n_in)
    base = gpu_qgemv(fmt, packed, n_out, n_in, x)
    try:
        qg.qg_set_tile_override("split=1")
        forced = gpu_qgemv(fmt, packed, n_out, n_in, x)
        assert not np.array_equal(forced.view(np.uint32), base.view(np.uint32))
        qg.qg_set_tile_override("split=1,rpw=2")
        assert np.array_equal(gpu_qgemv(fmt, packed, n_out, n_in, x).view(np.uint32), forced.view(np.uint32))
    finally:
        qg.qg_set_tile_override(None)
    assert np.array_equal(gpu_qgemv(fmt, packed, n_out, n_in, x).view(np.uint32), base.view(np.uint32))


def test_deterministic_and_prefix_rows():
    n_out, n_in = 4099, 2560
    W = workloads.gaussian(9, (n_out, n_in), 0.02)
    x = workloads.activations(9, n_in, 4)
    packed = upload("q8_0", ORC.quantize("q8_0", W), n_out, n_in)
    a = gpu_qgemv("q8_0", packed, n_out, n_in, x)
    b = gpu_qgemv("q8_0", packed, n_out, n_in, x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # a row prefix of the packed matrix is the smaller matrix (drafted vocabulary)
    c = gpu_qgemv("q8_0", packed, 1234, n_in, x)
    assert np.array_equal(c.view(np.uint32), a[:, :1234].view(np.uint32))


def test_largest_n_in_and_unsupported():
    n_out = 64
    for fmt in FMTS:
        n_in = 12288
        W = workloads.gaussian(10, (n_out, n_in), 0.02)
        x = workloads.gaussian(11, (4, n_in))
        canon = ORC.quantize(fmt, W)
        y = gpu_qgemv(fmt, upload(fmt, canon, n_out, n_in), n_out, n_in, x)
        check_close(y, ORC.gemv(fmt, canon, n_out, n_in, x), ORC.gemv_abs(fmt, canon, n_out, n_in, x), fmt)
    # the integer chunk dot stages x as 16-bit integers: n_in 16384 fits at ntok 4 for
    # Q8_0, Q4_0 and the affine format
    for fmt in ("q8_0", "q4_0", "affine4_g64"):
        n_in = 16384
        W = workloads.gaussian(13, (n_out, n_in), 0.02)
        x = workloads.gaussian(14, (4, n_in))
        canon = ORC.quantize(fmt, W)
        y = gpu_qgemv(fmt, upload(fmt, canon, n_out, n_in), n_out, n_in, x)
        check_close(y, ORC.gemv(fmt, canon, n_out, n_in, x), ORC.gemv_abs(fmt, canon, n_out, n_in, x), fmt)
    # x for ntok=4 at n_in = 32768 does not fit in shared memory: refused, nothing launched
    big = torch.zeros(qg.qg_packed_bytes("q8_0", 4, 32768), dtype=torch.uint8, device=dev())
    xd = torch.zeros((4, 32768), dtype=torch.float32, device=dev())
    yd = torch.zeros((4, 4), dtype=torch.float32, device=dev())
    with pytest.raises(qg.QGError) as e:
        qg.qgemv("q8_0", big, 4, 32768, xd, yd, 4)
    assert e.value.status == -3


def test_stream_argument():
    n_out, n_in = 777, 2560
    W = workloads.gaussian(12, (n_out, n_in), 0.02)
    x = workloads.activations(12, n_in, 2)
    canon = ORC.quantize("q8_0", W)
    packed = upload("q8_0", canon, n_out, n_in)
    s = torch.cuda.Stream()
    xd = torch.from_numpy(x).to(dev())
    y = torch.empty((2, n_out), dtype=torch.float32, device=dev())
    torch.cuda.synchronize()
    qg.qgemv("q8_0", packed, n_out, n_in, xd, y, 2, stream=s)
    s.synchronize()
    check_close(y.cpu().numpy(), ORC.gemv("q8_0", canon, n_out, n_in, x), ORC.gemv_abs("q8_0", canon, n_out, n_in, x))
