"""GPU parity of the owner-row backward (BD_BWD_OWNER_ROWS: every chunk's dK / dV
summed inside the kernel at the rows' owners, the reduce-scatter SUM / index_add
of the NeMo Automodel page "block-diagonal varlen CP for packed sequences",
Design overview, exchange.py) and of the forward that clears dQ on the side
(bd_attn_fwd_ex): against the oracle, per tensor and per document, and against
the window-partial path followed by bd_owner_sum."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("block_causal_varlen_gb300")
gu = pytest.importorskip("gpu_util")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    bd.load()


def owner_step(wl, q, k, v, do, zero_dq_in_fwd=True, accumulate=False, dk0=None, dv0=None):
    """Forward (clearing dQ on the side when asked) and owner-row backward of every
    chunk of every sequence. Returns out, lse (chunk views) and dq [B, S, H, d],
    dk, dv [B, S, Hkv, d] on the host."""
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=bd.BD_KV_WINDOW).upload("cuda")
    assert plan.owner_units() > 0
    qd = gu.as_chunks(q.cuda(), wl.cp)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    kd, vd, _ = gu.windows(plan, k.cuda(), v.cuda())
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((wl.B, wl.cp, wl.H, wl.L), float("nan"), dtype=torch.float32, device="cuda")
    dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
    if dk0 is None:
        dk = torch.full((wl.B, 1, wl.S, wl.Hkv, wl.d), float("nan"), dtype=torch.float32, device="cuda")
        dv = torch.full_like(dk, float("nan"))
    else:
        dk, dv = dk0.clone().cuda(), dv0.clone().cuda()
    flags = bd.BD_BWD_OWNER_ROWS
    if zero_dq_in_fwd:
        bd.bd_attn_fwd_ex(plan, qd, kd, vd, out, lse, dq_zero=dq)
        flags |= bd.BD_BWD_DQ_ZEROED
    else:
        bd.bd_attn_fwd(plan, qd, kd, vd, out, lse)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd_ex(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws, flags, accumulate_dkv=accumulate)
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    return (out.cpu(), lse.cpu(), dq.view(wl.B, wl.S, wl.H, wl.d).cpu(), dk.view(wl.B, wl.S, wl.Hkv, wl.d).cpu(),
            dv.view(wl.B, wl.S, wl.Hkv, wl.d).cpu())


def window_step(wl, q, k, v, do):
    """The reference path on the GPU: window partials, then bd_owner_sum_ex."""
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=bd.BD_KV_WINDOW).upload("cuda")
    qd = gu.as_chunks(q.cuda(), wl.cp)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    kd, vd, _ = gu.windows(plan, k.cuda(), v.cuda())
    out = torch.empty_like(qd)
    lse = torch.empty(wl.B, wl.cp, wl.H, wl.L, dtype=torch.float32, device="cuda")
    bd.bd_attn_fwd(plan, qd, kd, vd, out, lse)
    dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    dkw = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
    dvw = torch.zeros_like(dkw)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dkw, dvw, ws)
    dk = torch.empty(wl.B, 1, wl.S, wl.Hkv, wl.d, dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)
    bd.bd_owner_sum(plan, dkw, dvw, dk, dv, accumulate=False)
    torch.cuda.synchronize()
    return (out.cpu(), lse.cpu(), dq.view(wl.B, wl.S, wl.H, wl.d).cpu(), dk.view(wl.B, wl.S, wl.Hkv, wl.d).cpu(),
            dv.view(wl.B, wl.S, wl.Hkv, wl.d).cpu())


def _grad(got, want, cu, name):
    assert torch.isfinite(got).all(), f"{name}: non-finite values"
    rel = gu.max_rel(got, want)
    assert rel <= gu.GRAD_REL, f"{name}: max-rel {rel}"
    drel = gu.doc_rel(got, want, cu)
    assert drel <= gu.GRAD_REL, f"{name}: per-document max-rel {drel}"


@pytest.mark.parametrize("i", [1, 2])
def test_owner_rows_full_elementwise(i):
    """Every element of O, LSE, dQ, dK, dV against the oracle (per tensor and per
    document), with dQ cleared by the forward."""
    wl = workloads.config(i)
    q, k, v, do = workloads.tensors(wl)
    out, lse, dq, dk, dv = owner_step(wl, q, k, v, do)
    dt = torch.float64 if i == 1 else torch.float32
    for b in range(wl.B):
        o_ref, l_ref = oracle.attention_fwd(q[b], k[b], v[b], wl.cu[b], dtype=dt)
        o = out[b].reshape(wl.S, wl.H, wl.d)
        gu.o_check(o, o_ref)
        assert gu.doc_rel(o, o_ref, wl.cu[b]) <= gu.O_REL
        gu.lse_check(lse[b].permute(1, 0, 2).reshape(wl.H, wl.S), l_ref)
        gq, gk, gv, _, _ = oracle.attention_bwd(q[b], k[b], v[b], do[b], wl.cu[b], dtype=dt)
        _grad(dq[b], gq, wl.cu[b], "dQ")
        _grad(dk[b], gk, wl.cu[b], "dK")
        _grad(dv[b], gv, wl.cu[b], "dV")
        pad = wl.cu[b][-1]
        assert not dq[b, pad:].any() and not dk[b, pad:].any() and not dv[b, pad:].any()


EDGE = {   # (S, cp, cu): L a multiple of 128 so that the plan has an owner list
    "doc_over_every_chunk": (512, 4, [0, 512]),
    "tile_and_chunk_edges": (512, 2, [0, 128, 256, 384, 512]),
    "zero_and_one_token_docs": (768, 3, [0, 1, 1, 2, 200, 200, 640, 767]),
    "all_padding_chunk": (512, 2, [0, 40, 100]),
    "everything_padding": (256, 2, [0]),
}


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("name", sorted(EDGE))
def test_owner_rows_edge_layouts(name, d):
    S, cp, cu = EDGE[name]
    wl = dataclasses.replace(workloads.config(1), name=name, S=S, cp=cp, cu=[cu], H=4, Hkv=2, d=d)
    q, k, v, do = workloads.tensors(wl)
    out, lse, dq, dk, dv = owner_step(wl, q, k, v, do)
    gq, gk, gv, _, _ = oracle.attention_bwd(q[0], k[0], v[0], do[0], cu, dtype=torch.float64)
    if cu[-1] == 0:
        assert not dq.any() and not dk.any() and not dv.any()
        return
    _grad(dq[0], gq, cu, "dQ")
    _grad(dk[0], gk, cu, "dK")
    _grad(dv[0], gv, cu, "dV")
    pad = cu[-1]
    assert not dq[0, pad:].any() and not dk[0, pad:].any() and not dv[0, pad:].any()


@pytest.mark.parametrize("i", [2, 3, 5])
def test_owner_rows_equal_window_partials_summed(i):
    """The in-kernel owner sum equals the window-partial path plus bd_owner_sum up to
    fp32 rounding order (dK / dV of long documents sum hundreds of per-step partials
    with cancellation, so they are compared at 1e-3 of the tensor maximum, far below
    the size of any missing or doubled contribution); the forward that clears dQ
    leaves O and LSE bit-identical."""
    wl = workloads.config(i)
    q, k, v, do = workloads.tensors(wl)
    a = owner_step(wl, q, k, v, do)
    w = window_step(wl, q, k, v, do)
    assert torch.equal(a[0], w[0]) and torch.equal(a[1], w[1])
    for x, y, n in zip(a[2:], w[2:], ("dQ", "dK", "dV")):
        assert torch.isfinite(x).all(), n
        assert gu.max_rel(x, y) <= (1e-5 if n == "dQ" else 1e-3), n


def test_owner_rows_deterministic_and_dq_clearing_equivalent():
    """dK / dV of the owner path are bit-reproducible; dQ cleared by the forward
    equals dQ cleared by the statistics kernel (up to the reduce-add order)."""
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    a = owner_step(wl, q, k, v, do, zero_dq_in_fwd=True)
    b = owner_step(wl, q, k, v, do, zero_dq_in_fwd=False)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    assert gu.max_rel(a[2], b[2]) <= 1e-5


def test_owner_rows_accumulate():
    """accumulate_dkv = 1 adds the owner sums into what dk / dv held."""
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    base = owner_step(wl, q, k, v, do)
    g = torch.Generator().manual_seed(5)
    dk0 = torch.randn(wl.B, 1, wl.S, wl.Hkv, wl.d, generator=g)
    dv0 = torch.randn(wl.B, 1, wl.S, wl.Hkv, wl.d, generator=g)
    acc = owner_step(wl, q, k, v, do, accumulate=True, dk0=dk0, dv0=dv0)
    want_k = dk0.view_as(base[3]) + base[3]
    want_v = dv0.view_as(base[4]) + base[4]
    assert (acc[3] - want_k).abs().max().item() <= 1e-5 * want_k.abs().max().item()
    assert (acc[4] - want_v).abs().max().item() <= 1e-5 * want_v.abs().max().item()


@pytest.mark.parametrize("i", [3, 4])
def test_owner_rows_sampled_full_size(i):
    """Full-size workloads in the launch configuration the benchmark times: sampled
    dQ rows and dK / dV columns against the oracle (per tensor and per document),
    and dV summed over each document equal to dO summed over it."""
    wl = workloads.config(i)
    q, k, v, do = workloads.tensors(wl)
    _, _, dq, dk, dv = owner_step(wl, q, k, v, do)
    rng = np.random.default_rng(i)
    b = 0
    rows = gu.sample_rows(wl, b, n_rand=16 if i == 4 else 24)
    gq = oracle.attention_bwd_rows(q[b], k[b], v[b], do[b], wl.cu[b], rows)
    assert gu.max_rel(dq[b, rows], gq) <= gu.GRAD_REL
    cu = wl.cu[b]
    cols = set()
    for d in range(len(cu) - 1):
        a_, e_ = cu[d], cu[d + 1]
        if e_ > a_:
            cols.update(range(max(a_, e_ - 8), e_))
            cols.update(int(x) for x in rng.integers(max(a_, e_ - 384), e_, size=min(8, e_ - max(a_, e_ - 384))))
    cols = sorted(cols)
    gk, gv = oracle.attention_bwd_cols(q[b], k[b], v[b], do[b], cu, cols)
    assert gu.max_rel(dk[b, cols], gk) <= gu.GRAD_REL
    assert gu.max_rel(dv[b, cols], gv) <= gu.GRAD_REL
    G = wl.H // wl.Hkv
    for d in range(len(cu) - 1):
        a_, e_ = cu[d], cu[d + 1]
        if e_ <= a_:
            continue
        sv = dv[b, a_:e_].double().sum(0)
        so = do[b, a_:e_].double().view(e_ - a_, wl.Hkv, G, wl.d).sum((0, 2))
        assert (sv - so).abs().max().item() <= 2e-2 * max(1.0, so.abs().max().item())
    pad = cu[-1]
    assert not dq[b, pad:].any() and not dk[b, pad:].any() and not dv[b, pad:].any()


def test_fwd_ex_clears_dq_and_keeps_outputs():
    """bd_attn_fwd_ex zeroes every element of dq_zero (NaN before) and gives the
    same O and LSE, bit for bit, as bd_attn_fwd; at head dim 64, 128 and 256."""
    for d in (64, 128, 256):
        wl = dataclasses.replace(workloads.config(2), d=d)
        q, k, v, _ = workloads.tensors(wl)
        plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d).upload("cuda")
        qd = gu.as_chunks(q.cuda(), wl.cp)
        kd, vd = k.cuda().unsqueeze(1), v.cuda().unsqueeze(1)
        o1, o2 = torch.empty_like(qd), torch.empty_like(qd)
        l1 = torch.empty(wl.B, wl.cp, wl.H, wl.L, dtype=torch.float32, device="cuda")
        l2 = torch.empty_like(l1)
        dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
        bd.bd_attn_fwd(plan, qd, kd, vd, o1, l1)
        bd.bd_attn_fwd_ex(plan, qd, kd, vd, o2, l2, dq_zero=dq)
        torch.cuda.synchronize()
        bd.bd_check_status(plan)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        assert torch.count_nonzero(dq).item() == 0


def test_owner_flag_refused_without_owner_list():
    """An all-gathered plan has no owner list: BD_ERR_UNSUPPORTED before any launch
    (dq, filled with NaN, is untouched)."""
    wl = workloads.config(1)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_GATHER)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.zeros(wl.B, 1, wl.S, wl.Hkv, wl.d, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.BDError) as e:
        bd.bd_attn_bwd_ex(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws, bd.BD_BWD_OWNER_ROWS)
    assert e.value.status == -7
    torch.cuda.synchronize()
    assert torch.isnan(dq).all()
