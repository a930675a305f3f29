"""GPU parity of the routed-expert path: qg_expert_plan + qgemv_experts.

Track 2 Audit & Optimization Report (M5 Metal kernels), section 1 item 2: a plan
groups a step's (token, choice) pairs by expert and the gate/up and down
projections run each group with its own token count ne = 1..4.  Checked against
the fp64 oracle: the plan bit for bit; every slot's outputs within 1e-3 of
sum |w x|; outputs bitwise independent of ne, the group and the geometry, and equal
to the plain mat-vec's on the expert's rows; plan and kernel errors reported in
the device status word.
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

TOL = 1e-3
FMTS = ["q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"]


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qg.qg_set_tile_override(None)
    qg.qg_device_status(clear=True)
    yield
    qg.qg_set_tile_override(None)
    qg.qg_set_wait_limit(0, 0)
    qg.qg_device_status(clear=True)


def dev():
    return torch.device("cuda:0")


def n_in_for(fmt, base):
    m = {"q8_0": 32, "q4_0": 32, "affine4_g64": 64, "bf16": 16, "q5_0": 32}[fmt]
    return max(m, base // m * m)


def gpu_plan(ids, n_experts):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    idd = torch.from_numpy(ids).to(dev())
    n = ids.size
    plan = torch.full((qg.qg_expert_plan_ints(n),), -99, dtype=torch.int32, device=dev())
    qg.qg_expert_plan(idd, n_experts, plan)
    torch.cuda.synchronize()
    return plan


def oracle_plan_array(ids, n_experts):
    """The plan layout of the header, filled from the oracle's plan."""
    p = ORC.expert_plan(ids, n_experts)
    G = np.asarray(ids).size
    ng = len(p["group_expert"])
    a = np.full(2 + 5 * G, -99, dtype=np.int64)
    a[0] = ng
    a[1:2 + G] = G
    a[1:2 + ng] = p["group_start"]
    a[2 + G:2 + 2 * G] = -1
    a[2 + G:2 + G + ng] = p["group_expert"]
    a[2 + 2 * G:2 + 3 * G] = p["slot_pair"]
    a[2 + 3 * G:2 + 4 * G] = p["slot_token"]
    a[2 + 4 * G:2 + 5 * G] = p["pair_slot"]
    return a, p


def run_experts(fmt, packed, n_experts, n_out, n_in, x, plan, n_slots, by_slot=False, nxt=None):
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev())
    y = torch.full((n_slots, n_out), float("nan"), dtype=torch.float32, device=dev())
    W_next, nno, nni = nxt if nxt is not None else (None, 0, 0)
    qg.qgemv_experts(fmt, packed, n_experts, n_out, n_in, xd, plan, n_slots, y, x_by_slot=by_slot,
                     W_next=W_next, next_n_out=nno, next_n_in=nni)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def slot_reference(fmt, canon, n_experts, n_out, n_in, x, p, by_slot):
    """Oracle values and sum |w x| per slot."""
    ref = ORC.experts_gemv_slots(fmt, canon, n_experts, n_out, n_in, x, p, by_slot)
    G = int(p["group_start"][-1])
    den = np.empty((G, n_out))
    for g, e in enumerate(p["group_expert"]):
        sub = ORC.row_slice(fmt, canon, n_experts * n_out, n_in, int(e) * n_out, (int(e) + 1) * n_out)
        for s in range(int(p["group_start"][g]), int(p["group_start"][g + 1])):
            row = s if by_slot else int(p["slot_token"][s])
            den[s] = ORC.gemv_abs(fmt, sub, n_out, n_in, x[row:row + 1])[0]
    return ref, den


def check_close(y, ref, den, what):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), what
    zero = den == 0
    assert np.all(y[zero] == 0), what
    rel = np.abs(y[~zero] - ref[~zero]) / den[~zero]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= TOL, f"{what}: max normalised error {worst:.3g}"
    return worst


# ----------------------------------------------------------------------------- the plan

@pytest.mark.parametrize("ntok,topk,n_experts", [(1, 1, 1), (1, 10, 512), (3, 10, 512), (4, 10, 512),
                                                 (4, 8, 16), (2, 6, 3), (128, 8, 100), (1, 1024, 7)])
def test_plan_matches_oracle(ntok, topk, n_experts):
    rng = np.random.default_rng(ntok * 1000 + topk)
    for trial in range(3):
        if trial == 0 and topk <= n_experts and ntok <= 4:
            ids = workloads.routing(trial + 7, ntok, topk, n_experts, 0.65)
        else:                                   # any ids, repeats within a token included
            ids = rng.integers(0, n_experts, size=(ntok, topk)).astype(np.int32)
        got = gpu_plan(ids, n_experts).cpu().numpy()
        want, _ = oracle_plan_array(ids, n_experts)
        assert np.array_equal(got, want), (ntok, topk, n_experts, trial)
    assert qg.qg_device_status() == 0


def test_plan_rejects_an_expert_outside_the_stack():
    ids = np.array([[0, 3], [5, 1]], dtype=np.int32)
    got = gpu_plan(ids, 5).cpu().numpy()
    assert got[0] == 0
    assert qg.qg_device_status() == qg.QG_DEVICE_BAD_PLAN
    got = gpu_plan(np.array([[0, 3], [4, 1]], dtype=np.int32), 5).cpu().numpy()
    assert got[0] == 4 and qg.qg_device_status() == 0


# ----------------------------------------------------------------------------- the mat-vec, small ragged shapes

def _small_case(fmt, n_experts, n_out, n_in_base, seed):
    n_in = n_in_for(fmt, n_in_base)
    W = workloads.gaussian(seed, (n_experts * n_out, n_in), 0.02)
    W[3] = 0.0                                           # a zero row: exact zeros expected
    canon = ORC.quantize(fmt, W)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n_experts * n_out, n_in)).to(dev())
    return n_in, canon, packed


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_experts,n_out,n_in_base", [(6, 37, 640), (9, 64, 2560), (4, 5, 96)])
@pytest.mark.parametrize("by_slot", [False, True])
def test_experts_match_oracle(fmt, n_experts, n_out, n_in_base, by_slot):
    n_in, canon, packed = _small_case(fmt, n_experts, n_out, n_in_base, 300 + n_out)
    for ntok in (1, 2, 3, 4):
        topk = min(3, n_experts)
        ids = workloads.routing(ntok * 11 + n_out, ntok, topk, n_experts, 0.65)
        G = ntok * topk
        x = workloads.gaussian(ntok + n_in, (G if by_slot else ntok, n_in))
        plan_d = gpu_plan(ids, n_experts)
        _, p = oracle_plan_array(ids, n_experts)
        y = run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, G, by_slot)
        ref, den = slot_reference(fmt, canon, n_experts, n_out, n_in, x, p, by_slot)
        check_close(y, ref, den, f"{fmt} E={n_experts} {n_out}x{n_in} ntok={ntok} by_slot={by_slot}")
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_outputs_bitwise_independent_of_ne_group_and_tile(fmt):
    """Token t's outputs for expert 0 come out of a group of four tokens; the same token
    alone with expert 1 (same weights copied) must give the same bits, under every
    geometry, and the plain mat-vec on the expert's rows gives them too when it does not
    split."""
    n_out, n_in = 150, n_in_for(fmt, 2560)
    W0 = workloads.gaussian(41, (n_out, n_in), 0.02)
    W = np.concatenate([W0, W0, workloads.gaussian(42, (3 * n_out, n_in), 0.02)])
    n_experts = 5
    canon = ORC.quantize(fmt, W)
    packed = torch.from_numpy(qg.qg_to_device_layout(fmt, canon, n_experts * n_out, n_in)).to(dev())
    x = workloads.gaussian(43, (4, n_in))
    # expert 0: all four tokens; expert 1: token 2 only; experts 2-4 one token each
    ids = np.array([[0, 2], [0, 3], [0, 1], [0, 4]], dtype=np.int32)
    plan_d = gpu_plan(ids, n_experts)
    _, p = oracle_plan_array(ids, n_experts)
    slot = {int(i): int(s) for i, s in enumerate(p["pair_slot"])}
    results = []
    for spec in (None, "rpw=1", "rpw=2,depth=2,warps=4", "rpw=4,depth=3,warps=8", "rpw=4,warps=12,ctas=2",
                 "rpw=2,warps=1,depth=2", "gw=0", "gw=9"):
        qg.qg_set_tile_override(spec)
        results.append(run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, 8))
    qg.qg_set_tile_override(None)
    for r in results[1:]:
        assert np.array_equal(r.view(np.uint32), results[0].view(np.uint32))
    y = results[0]
    assert np.array_equal(y[slot[2 * 2 + 0]].view(np.uint32), y[slot[2 * 2 + 1]].view(np.uint32))
    tile = qg.qg_describe_tile(fmt, n_out, n_in, 1)
    if "split=1" in tile:
        xd = torch.from_numpy(x).to(dev())
        yd = torch.empty((4, n_out), dtype=torch.float32, device=dev())
        qg.qgemv(fmt, packed, n_out, n_in, xd, yd, 4)       # expert 0's rows are the stack's first
        torch.cuda.synchronize()
        yq = yd.cpu().numpy()
        for t in range(4):
            assert np.array_equal(y[slot[2 * t]].view(np.uint32), yq[t].view(np.uint32)), t


def check_swiglu(act, ref_y, den_y, what):
    """act = silu(gate) * up from the GPU against the oracle's gate / up rows (interleaved):
    the error allowed is the mat-vec tolerance carried through the activation,
    |d act| <= 1e-3 (|silu'(g) u| D_g + |silu(g)| D_u) + 1e-5 |act|."""
    g, u = ref_y[..., 0::2], ref_y[..., 1::2]
    Dg, Du = den_y[..., 0::2], den_y[..., 1::2]
    ref = ORC.swiglu_rows(ref_y)
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    bound = TOL * (np.abs(dsilu * u) * Dg + np.abs(ORC.silu(g)) * Du) + 1e-5 * np.abs(ref) + 1e-30
    act = act.astype(np.float64)
    assert np.all(np.isfinite(act)), what
    bad = np.abs(act - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs outside the bound"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_experts,d_ff,n_in_base", [(6, 37, 640), (5, 320, 2560)])
def test_swiglu_gate_up(fmt, n_experts, d_ff, n_in_base):
    """Gate / up rows interleaved per expert; y = silu(gate) * up."""
    n_out = 2 * d_ff
    n_in, canon, packed = _small_case(fmt, n_experts, n_out, n_in_base, 900 + d_ff)
    for ntok in (1, 2, 3, 4):
        ids = workloads.routing(ntok * 5 + d_ff, ntok, 3, n_experts, 0.65)
        G = ntok * 3
        x = workloads.gaussian(ntok + n_in + 1, (ntok, n_in), 2.0)      # gate values around +-1
        plan_d = gpu_plan(ids, n_experts)
        _, p = oracle_plan_array(ids, n_experts)
        xd = torch.from_numpy(x).to(dev())
        act = torch.full((G, d_ff), float("nan"), dtype=torch.float32, device=dev())
        qg.qgemv_experts(fmt, packed, n_experts, n_out, n_in, xd, plan_d, G, act, swiglu=True)
        torch.cuda.synchronize()
        ref, den = slot_reference(fmt, canon, n_experts, n_out, n_in, x, p, False)
        check_swiglu(act.cpu().numpy(), ref, den, f"{fmt} swiglu ntok={ntok}")
        # the same rows without the flag: the plain projection, whose pairs give the same act
        y = run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, G)
        check_close(y, ref, den, f"{fmt} gate/up ntok={ntok}")
    assert qg.qg_device_status() == 0


def test_more_groups_than_ctas():
    """About 300 one- and two-slot groups on a one-CTA-per-SM grid: CTAs take whole
    groups one after the other, restaging x between them."""
    fmt, n_experts, n_out = "q8_0", 400, 24
    n_in, canon, packed = _small_case(fmt, n_experts, n_out, 320, 77)
    rng = np.random.default_rng(8)
    ids = rng.integers(0, n_experts, size=(100, 3)).astype(np.int32)
    _, p = oracle_plan_array(ids, n_experts)
    assert len(p["group_expert"]) > 200
    plan_d = gpu_plan(ids, n_experts)
    qg.qg_set_tile_override("ctas=1")
    for by_slot in (False, True):
        x = workloads.gaussian(9, (300 if by_slot else 100, n_in))
        y = run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, 300, by_slot)
        ref, den = slot_reference(fmt, canon, n_experts, n_out, n_in, x, p, by_slot)
        check_close(y, ref, den, f"many groups by_slot={by_slot}")
    assert qg.qg_device_status() == 0


def test_bad_plan_entries_are_skipped_and_reported():
    fmt, n_experts, n_out = "q8_0", 4, 32
    n_in, canon, packed = _small_case(fmt, n_experts, n_out, 256, 91)
    ids = np.array([[0, 1], [2, 3]], dtype=np.int32)
    a, p = oracle_plan_array(ids, n_experts)
    x = workloads.gaussian(92, (2, n_in))
    ref, den = slot_reference(fmt, canon, n_experts, n_out, n_in, x, p, False)
    bad = a.copy()
    G = 4
    bad[2 + G + 1] = n_experts                 # group 1's expert outside the stack
    bad[2 + 3 * G + 2] = 9                     # slot 2 reads token row 9 of a 2-row x
    plan_d = torch.from_numpy(bad.astype(np.int32)).to(dev())
    y = run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, G)
    assert qg.qg_device_status() == qg.QG_DEVICE_BAD_PLAN
    assert np.all(np.isnan(y[1])) and np.all(np.isnan(y[2]))          # skipped groups write nothing
    check_close(y[[0, 3]], ref[[0, 3]], den[[0, 3]], "good groups of a bad plan")
    bad = a.copy()
    bad[0] = G + 1                             # more groups than slots
    y = run_experts(fmt, packed, n_experts, n_out, n_in, x, torch.from_numpy(bad.astype(np.int32)).to(dev()), G)
    assert qg.qg_device_status() == qg.QG_DEVICE_BAD_PLAN
    assert np.all(np.isnan(y))


def test_wait_timeout_reports_and_recovers():
    fmt, n_experts, n_out = "q8_0", 8, 256
    n_in, canon, packed = _small_case(fmt, n_experts, n_out, 2560, 93)
    ids = workloads.routing(3, 4, 4, n_experts, 0.65)
    plan_d = gpu_plan(ids, n_experts)
    x = workloads.gaussian(94, (4, n_in))
    qg.qg_set_wait_limit(2000, 16)
    run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, 16)
    assert qg.qg_device_status() & qg.QG_DEVICE_WAIT_TIMEOUT
    qg.qg_set_wait_limit(0, 0)
    y = run_experts(fmt, packed, n_experts, n_out, n_in, x, plan_d, 16)
    assert qg.qg_device_status() == 0
    _, p = oracle_plan_array(ids, n_experts)
    ref, den = slot_reference(fmt, canon, n_experts, n_out, n_in, x, p, False)
    check_close(y, ref, den, "after a timeout")


def test_plan_ready_chain_under_early_start():
    """plan -> gate/up -> down (QG_EXPERTS_PLAN_READY) for several routings back to back
    under early start, no host sync in between: every down output equals the one from
    the plain path (plan read after the wait), bit for bit."""
    fmt, n_experts, d_model, d_ff, topk = "q8_0", 16, 512, 128, 4
    _, canon_gu, gu = _small_case(fmt, n_experts, 2 * d_ff, d_model, 501)
    _, canon_dn, dn = _small_case(fmt, n_experts, d_model, d_ff, 502)
    runs = []
    for r in range(6):
        ntok = 1 + r % 4
        ids = workloads.routing(600 + r, ntok, topk, n_experts, 0.65)
        G = ntok * topk
        runs.append((torch.from_numpy(ids).to(dev()), G,
                     torch.from_numpy(workloads.gaussian(700 + r, (ntok, d_model))).to(dev()),
                     torch.from_numpy(workloads.gaussian(800 + r, (G, d_ff))).to(dev())))

    def chain(ready):
        outs = []
        for ids, G, x, h in runs:
            plan = torch.full((qg.qg_expert_plan_ints(G),), -5, dtype=torch.int32, device=dev())
            y_gu = torch.empty((G, 2 * d_ff), dtype=torch.float32, device=dev())
            y_dn = torch.empty((G, d_model), dtype=torch.float32, device=dev())
            qg.qg_expert_plan(ids, n_experts, plan)
            qg.qgemv_experts(fmt, gu, n_experts, 2 * d_ff, d_model, x, plan, G, y_gu, W_next=dn,
                             next_n_out=d_model, next_n_in=d_ff)
            qg.qgemv_experts(fmt, dn, n_experts, d_model, d_ff, h, plan, G, y_dn, x_by_slot=True, plan_ready=ready)
            outs.append((y_gu, y_dn, plan))      # every buffer stays alive until the sync
        torch.cuda.synchronize()
        return [(a.cpu().numpy(), b.cpu().numpy()) for a, b, _ in outs]

    qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
    try:
        plain = chain(False)
        for _ in range(3):
            ready = chain(True)
            for (a0, b0), (a1, b1) in zip(plain, ready):
                assert np.array_equal(a0.view(np.uint32), a1.view(np.uint32))
                assert np.array_equal(b0.view(np.uint32), b1.view(np.uint32))
    finally:
        qg.qg_set_launch_options(0)
    assert qg.qg_device_status() == 0
    # and the plain path against the oracle
    ids, G, x, h = runs[3]
    _, p = oracle_plan_array(ids.cpu().numpy(), n_experts)
    ref, den = slot_reference(fmt, canon_dn, n_experts, d_model, d_ff, h.cpu().numpy(), p, True)
    check_close(plain[3][1], ref, den, "plan-ready chain, down")


# ----------------------------------------------------------------------------- the full layer size, sampled

def _packed_stack(layer, n_out, n_in, seed, experts, threads=16):
    stride = qg.qg_row_stride(layer.fmt, n_in)
    out = np.empty(len(experts) * n_out * stride, dtype=np.uint8)

    def one(k):
        We = workloads.expert_matrix(seed, experts[k], n_out, n_in)
        qg.qg_pack(layer.fmt, We, out=out[k * n_out * stride:(k + 1) * n_out * stride])

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(len(experts))))
    return out


def test_full_size_layer_sampled():
    """The expert shapes of the routed-expert table (gate/up 2 x 640 x 2560, down
    2560 x 640, top-10 of 64 experts here, ntok 1..4, share 0.65): plan bit for bit,
    then for every group 8 sampled rows of each projection against the oracle."""
    layer = workloads.EXPERT_LAYERS["q8_0_experts_512x2560x640_top10"]
    n_experts = 64
    ff2, dm, ff = 2 * layer.d_ff, layer.d_model, layer.d_ff
    experts = list(range(n_experts))
    gu = torch.from_numpy(_packed_stack(layer, ff2, dm, layer.seed, experts)).to(dev())
    dn = torch.from_numpy(_packed_stack(layer, dm, ff, layer.seed + 1, experts)).to(dev())
    rng = np.random.default_rng(5)
    for ntok in (1, 2, 3, 4):
        ids = workloads.routing(layer.seed + ntok, ntok, layer.topk, n_experts, layer.share)
        G = ntok * layer.topk
        plan_d = gpu_plan(ids, n_experts)
        want, p = oracle_plan_array(ids, n_experts)
        assert np.array_equal(plan_d.cpu().numpy(), want)
        x = workloads.activations(layer.seed + ntok, dm, ntok)
        h = workloads.gaussian(layer.seed + 10 + ntok, (G, ff))
        y_gu = run_experts(layer.fmt, gu, n_experts, ff2, dm, x, plan_d, G)
        # with the down stack prefetched into L2: the same bits
        y_pf = run_experts(layer.fmt, gu, n_experts, ff2, dm, x, plan_d, G, nxt=(dn, dm, ff))
        assert np.array_equal(y_pf.view(np.uint32), y_gu.view(np.uint32))
        # the gated activation of the same launch (rows read as gate / up pairs)
        act_d = torch.empty((G, ff), dtype=torch.float32, device=dev())
        qg.qgemv_experts(layer.fmt, gu, n_experts, ff2, dm, torch.from_numpy(x).to(dev()), plan_d, G, act_d,
                         swiglu=True)
        torch.cuda.synchronize()
        act = act_d.cpu().numpy()
        y_dn = run_experts(layer.fmt, dn, n_experts, dm, ff, h, plan_d, G, by_slot=True)
        for g, e in enumerate(p["group_expert"]):
            e = int(e)
            for (yy, n_out, n_in, seed, xin, by_slot) in ((y_gu, ff2, dm, layer.seed, x, False),
                                                         (y_dn, dm, ff, layer.seed + 1, h, True)):
                pairs = np.sort(rng.choice(n_out // 2, size=4, replace=False))
                rows = np.stack([2 * pairs, 2 * pairs + 1], axis=1).reshape(-1)     # (gate, up) pairs
                canon = ORC.quantize(layer.fmt, workloads.expert_matrix(seed, e, n_out, n_in)[rows])
                for s in range(int(p["group_start"][g]), int(p["group_start"][g + 1])):
                    r = s if by_slot else int(p["slot_token"][s])
                    ref = ORC.gemv(layer.fmt, canon, len(rows), n_in, xin[r:r + 1])[0]
                    den = ORC.gemv_abs(layer.fmt, canon, len(rows), n_in, xin[r:r + 1])[0]
                    check_close(yy[s, rows][None], ref[None], den[None], f"ntok={ntok} group {g} slot {s}")
                    if not by_slot:
                        check_swiglu(act[s, pairs][None], ref[None], den[None], f"ntok={ntok} group {g} act")
    assert qg.qg_device_status() == 0


# ----------------------------------------------------------------------------- the layer in one launch

def _layer_case(fmt, n_experts, d_model, d_ff, seed):
    W_gu = workloads.gaussian(seed, (n_experts * 2 * d_ff, d_model), 0.02)
    W_dn = workloads.gaussian(seed + 1, (n_experts * d_model, d_ff), 0.05)
    c_gu, c_dn = ORC.quantize(fmt, W_gu), ORC.quantize(fmt, W_dn)
    gu = torch.from_numpy(qg.qg_to_device_layout(fmt, c_gu, n_experts * 2 * d_ff, d_model)).to(dev())
    dn = torch.from_numpy(qg.qg_to_device_layout(fmt, c_dn, n_experts * d_model, d_ff)).to(dev())
    return c_gu, c_dn, gu, dn


def _three_launches(fmt, gu, dn, n_experts, d_model, d_ff, xd, idd):
    G = idd.numel()
    plan = torch.full((qg.qg_expert_plan_ints(G),), -5, dtype=torch.int32, device=dev())
    act = torch.full((G, d_ff), float("nan"), dtype=torch.float32, device=dev())
    y = torch.full((G, d_model), float("nan"), dtype=torch.float32, device=dev())
    qg.qg_expert_plan(idd, n_experts, plan)
    qg.qgemv_experts(fmt, gu, n_experts, 2 * d_ff, d_model, xd, plan, G, act, swiglu=True)
    qg.qgemv_experts(fmt, dn, n_experts, d_model, d_ff, act, plan, G, y, x_by_slot=True)
    torch.cuda.synchronize()
    return plan.cpu().numpy(), act.cpu().numpy(), y.cpu().numpy()


def _one_launch(fmt, gu, dn, n_experts, d_model, d_ff, xd, idd, ws):
    G = idd.numel()
    plan = torch.full((qg.qg_expert_plan_ints(G),), -5, dtype=torch.int32, device=dev())
    act = torch.full((G, d_ff), float("nan"), dtype=torch.float32, device=dev())
    y = torch.full((G, d_model), float("nan"), dtype=torch.float32, device=dev())
    qg.qgemv_expert_layer(fmt, gu, dn, n_experts, d_model, d_ff, xd, idd, plan, act, y, ws)
    return plan, act, y


def check_layer_against_oracle(fmt, c_gu, c_dn, n_experts, d_model, d_ff, ids, x, act, y, what):
    """act against the oracle's silu(gate) * up; y against the oracle's down projection of
    the oracle's (fp64) activation, with the activation's tolerance carried through:
    |dy| <= 1e-3 sum |w act| + sum |w| |d act|."""
    _, p = oracle_plan_array(ids, n_experts)
    g_ref, g_den = slot_reference(fmt, c_gu, n_experts, 2 * d_ff, d_model, x, p, False)
    check_swiglu(act, g_ref, g_den, what + " act")
    gt, ut = g_ref[..., 0::2], g_ref[..., 1::2]
    sig = 1.0 / (1.0 + np.exp(-gt))
    act_ref = ORC.swiglu_rows(g_ref)
    act_tol = (TOL * (np.abs(sig * (1.0 + gt * (1.0 - sig)) * ut) * g_den[..., 0::2]
                      + np.abs(ORC.silu(gt)) * g_den[..., 1::2]) + 1e-5 * np.abs(act_ref))
    y_ref, y_den = slot_reference(fmt, c_dn, n_experts, d_model, d_ff, act_ref, p, True)
    _, y_carry = slot_reference(fmt, c_dn, n_experts, d_model, d_ff, act_tol, p, True)
    bound = TOL * y_den + y_carry + 1e-30
    assert np.all(np.isfinite(y)), what
    bad = np.abs(y.astype(np.float64) - y_ref) > bound
    assert not bad.any(), f"{what} y: {int(bad.sum())} outputs outside the bound"


@pytest.mark.parametrize("fmt", FMTS)
def test_layer_one_launch_equals_three_launches_and_oracle(fmt):
    n_experts, d_model, d_ff, topk = 16, 512, 128, 4
    c_gu, c_dn, gu, dn = _layer_case(fmt, n_experts, d_model, d_ff, 1100)
    ws = torch.zeros(qg.qgemv_expert_layer_workspace_bytes(), dtype=torch.uint8, device=dev())
    for ntok in (1, 2, 3, 4):
        ids = workloads.routing(1200 + ntok, ntok, topk, n_experts, 0.65)
        x = workloads.gaussian(1300 + ntok, (ntok, d_model), 2.0)
        xd, idd = torch.from_numpy(x).to(dev()), torch.from_numpy(ids).to(dev())
        plan3, act3, y3 = _three_launches(fmt, gu, dn, n_experts, d_model, d_ff, xd, idd)
        plan1, act1, y1 = _one_launch(fmt, gu, dn, n_experts, d_model, d_ff, xd, idd, ws)
        torch.cuda.synchronize()
        plan1, act1, y1 = plan1.cpu().numpy(), act1.cpu().numpy(), y1.cpu().numpy()
        want, _ = oracle_plan_array(ids, n_experts)
        assert np.array_equal(plan1, want) and np.array_equal(plan3, want)
        assert np.array_equal(act1.view(np.uint32), act3.view(np.uint32)), ntok
        assert np.array_equal(y1.view(np.uint32), y3.view(np.uint32)), ntok
        check_layer_against_oracle(fmt, c_gu, c_dn, n_experts, d_model, d_ff, ids, x, act1, y1, f"{fmt} ntok={ntok}")
    assert not ws.cpu().numpy().any()                     # the barrier words are zero again
    assert qg.qg_device_status() == 0


def test_layer_back_to_back_under_early_start():
    """Eight layer launches in a row on one workspace, early start on, no host sync:
    each equals the three-launch path bit for bit and the workspace ends zeroed."""
    fmt, n_experts, d_model, d_ff, topk = "q8_0", 24, 640, 192, 6
    _, _, gu, dn = _layer_case(fmt, n_experts, d_model, d_ff, 1400)
    ws = torch.zeros(qg.qgemv_expert_layer_workspace_bytes(), dtype=torch.uint8, device=dev())
    cases = []
    for r in range(8):
        ntok = 1 + r % 4
        ids = torch.from_numpy(workloads.routing(1500 + r, ntok, topk, n_experts, 0.3)).to(dev())
        x = torch.from_numpy(workloads.gaussian(1600 + r, (ntok, d_model))).to(dev())
        cases.append((ids, x))
    want = [_three_launches(fmt, gu, dn, n_experts, d_model, d_ff, x, ids) for ids, x in cases]
    qg.qg_set_launch_options(qg.QG_LAUNCH_EARLY_START)
    try:
        got = [_one_launch(fmt, gu, dn, n_experts, d_model, d_ff, x, ids, ws) for ids, x in cases]
        torch.cuda.synchronize()
    finally:
        qg.qg_set_launch_options(0)
    for (p3, a3, y3), (p1, a1, y1) in zip(want, got):
        assert np.array_equal(p1.cpu().numpy(), p3)
        assert np.array_equal(a1.cpu().numpy().view(np.uint32), a3.view(np.uint32))
        assert np.array_equal(y1.cpu().numpy().view(np.uint32), y3.view(np.uint32))
    assert not ws.cpu().numpy().any()
    assert qg.qg_device_status() == 0


def test_layer_full_size():
    """512 experts of the routed-expert table's size in one launch at ntok 4: equal to the
    three-launch path bit for bit (those are checked against the oracle above)."""
    layer = workloads.EXPERT_LAYERS["q8_0_experts_512x2560x640_top10"]
    n_experts, dm, ff = 64, layer.d_model, layer.d_ff
    experts = list(range(n_experts))
    gu = torch.from_numpy(_packed_stack(layer, 2 * ff, dm, layer.seed, experts)).to(dev())
    dn = torch.from_numpy(_packed_stack(layer, dm, ff, layer.seed + 1, experts)).to(dev())
    ws = torch.zeros(qg.qgemv_expert_layer_workspace_bytes(), dtype=torch.uint8, device=dev())
    for ntok in (1, 4):
        ids = workloads.routing(layer.seed + 40 + ntok, ntok, layer.topk, n_experts, layer.share)
        x = workloads.activations(layer.seed + ntok, dm, ntok)
        xd, idd = torch.from_numpy(x).to(dev()), torch.from_numpy(ids).to(dev())
        p3, a3, y3 = _three_launches(layer.fmt, gu, dn, n_experts, dm, ff, xd, idd)
        p1, a1, y1 = _one_launch(layer.fmt, gu, dn, n_experts, dm, ff, xd, idd, ws)
        torch.cuda.synchronize()
        assert np.array_equal(p1.cpu().numpy(), p3)
        assert np.array_equal(a1.cpu().numpy().view(np.uint32), a3.view(np.uint32))
        assert np.array_equal(y1.cpu().numpy().view(np.uint32), y3.view(np.uint32))
    assert qg.qg_device_status() == 0


def test_layer_bad_id_and_timeout_recover():
    fmt, n_experts, d_model, d_ff = "q8_0", 8, 256, 64
    _, _, gu, dn = _layer_case(fmt, n_experts, d_model, d_ff, 1700)
    ws = torch.zeros(qg.qgemv_expert_layer_workspace_bytes(), dtype=torch.uint8, device=dev())
    x = torch.from_numpy(workloads.gaussian(1701, (2, d_model))).to(dev())
    bad = torch.from_numpy(np.array([[0, 8], [3, 1]], dtype=np.int32)).to(dev())
    plan, act, y = _one_launch(fmt, gu, dn, n_experts, d_model, d_ff, x, bad, ws)
    torch.cuda.synchronize()
    assert plan.cpu().numpy()[0] == 0 and np.all(np.isnan(y.cpu().numpy()))
    assert qg.qg_device_status() == qg.QG_DEVICE_BAD_PLAN
    assert not ws.cpu().numpy().any()
    good = torch.from_numpy(np.array([[0, 7], [3, 1]], dtype=np.int32)).to(dev())
    qg.qg_set_wait_limit(2000, 16)
    _one_launch(fmt, gu, dn, n_experts, d_model, d_ff, x, good, ws)
    torch.cuda.synchronize()
    assert qg.qg_device_status() & qg.QG_DEVICE_WAIT_TIMEOUT
    qg.qg_set_wait_limit(0, 0)
    assert not ws.cpu().numpy().any()                     # every CTA still met and left the barrier
    p3, a3, y3 = _three_launches(fmt, gu, dn, n_experts, d_model, d_ff, x, good)
    p1, a1, y1 = _one_launch(fmt, gu, dn, n_experts, d_model, d_ff, x, good, ws)
    torch.cuda.synchronize()
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), y3.view(np.uint32))
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("fmt", ["q8_0", "affine4_g64"])
def test_one_x_row_and_repeated_experts(fmt):
    """A single x row (gate/up at ntok 1) gives bitwise the results of the same call with
    a second, unused row, also for a token that lists an expert more than once (one
    group of several slots, all reading the same row)."""
    n_experts, n_out, n_in = 12, 96, n_in_for(fmt, 2560)
    n_in, canon, packed = _small_case(fmt, n_experts, n_out, n_in, 1800)
    x1 = workloads.gaussian(1801, (1, n_in))
    x2 = np.concatenate([x1, workloads.gaussian(1802, (1, n_in))])    # a second, unused row
    for ids in (workloads.routing(1803, 1, 5, n_experts, 0.65), np.array([[3, 3, 5, 7, 3]], dtype=np.int32)):
        plan_d = gpu_plan(ids, n_experts)
        G = ids.size
        for swiglu in (False, True):
            outs = []
            for x in (x1, x2):
                xd = torch.from_numpy(x).to(dev())
                y = torch.full((G, n_out // 2 if swiglu else n_out), float("nan"), dtype=torch.float32, device=dev())
                qg.qgemv_experts(fmt, packed, n_experts, n_out, n_in, xd, plan_d, G, y, swiglu=swiglu)
                torch.cuda.synchronize()
                outs.append(y.cpu().numpy())
            assert np.all(np.isfinite(outs[0]))
            assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32)), (ids.tolist(), swiglu)
        _, p = oracle_plan_array(ids, n_experts)
        ref, den = slot_reference(fmt, canon, n_experts, n_out, n_in, x1, p, False)
        y = run_experts(fmt, packed, n_experts, n_out, n_in, x1, plan_d, G)
        check_close(y, ref, den, f"{fmt} one row {ids.tolist()}")
    assert qg.qg_device_status() == 0
