"""GPU backward parity: dQ, dK, dV from the CUDA path (through the C ABI)
against the oracle on the same seeded bf16 inputs; the owner summation of
needed-only-window partials; gradient identities at full size."""
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


def run_bwd(wl, q, k, v, do, mode, accumulate=False):
    """Forward then backward of every chunk of every sequence in batched calls.
    Returns dq [B, S, H, d] and dk, dv as owner-row tensors [B, S, Hkv, d]
    (needed-only windows are summed at their owners by bd_owner_sum)."""
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, mode)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.full(kd.shape, float("nan"), dtype=torch.float32, device="cuda")
    dv = torch.full(vd.shape, float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws)
    if mode == bd.BD_KV_WINDOW:
        dk_full = torch.zeros(wl.B, 1, wl.S, wl.Hkv, wl.d, dtype=torch.float32, device="cuda")
        dv_full = torch.zeros_like(dk_full)
        # window rows past each chunk's window are not written: give them zeros
        for b in range(wl.B):
            for c in range(wl.cp):
                hdr, _ = plan.chunk(b * wl.cp + c)
                n = hdr["kv_end"] - hdr["kv_start"]
                dk[b, c, n:] = 0
                dv[b, c, n:] = 0
        bd.bd_owner_sum(plan, dk, dv, dk_full, dv_full)
        dk, dv = dk_full, dv_full
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    return (dq.view(wl.B, wl.S, wl.H, wl.d).cpu(), dk.view(wl.B, wl.S, wl.Hkv, wl.d).cpu(),
            dv.view(wl.B, wl.S, wl.Hkv, wl.d).cpu())


def grad_check(got, want, name):
    assert torch.isfinite(got).all(), f"{name}: non-finite values"
    rel = gu.max_rel(got, want)
    assert rel <= gu.GRAD_REL, f"{name}: max-rel {rel}"
    return rel


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("i", [1, 2])
def test_bwd_full_elementwise(i, mode):
    wl = workloads.config(i)
    q, k, v, do = workloads.tensors(wl)
    dq, dk, dv = run_bwd(wl, q, k, v, do, mode)
    for b in range(wl.B):
        gq, gk, gv, _, _ = oracle.attention_bwd(q[b], k[b], v[b], do[b], wl.cu[b],
                                                dtype=torch.float64 if i == 1 else torch.float32)
        grad_check(dq[b], gq, "dQ")
        grad_check(dk[b], gk, "dK")
        grad_check(dv[b], gv, "dV")
        # per document too: a wrong short document would hide under the tensor maximum
        for got, want, name in ((dq[b], gq, "dQ"), (dk[b], gk, "dK"), (dv[b], gv, "dV")):
            assert gu.doc_rel(got, want, wl.cu[b]) <= gu.GRAD_REL, f"{name}: per-document max-rel"
        pad = wl.cu[b][-1]
        assert not dq[b, pad:].any() and not dk[b, pad:].any() and not dv[b, pad:].any()


def test_bwd_chunk_partials_match_oracle_partials():
    """Per-chunk calls in window mode: each window buffer holds exactly that
    chunk's partial, which the oracle's chunk backward gives independently."""
    wl = workloads.config(1)
    q, k, v, do = workloads.tensors(wl)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=bd.BD_KV_WINDOW).upload("cuda")
    _, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_WINDOW)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(kd.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws)
    torch.cuda.synchronize()
    for c in range(wl.cp):
        hdr, _ = plan.chunk(c)
        a, e = hdr["kv_start"], hdr["kv_end"]
        rows = slice(c * wl.L, (c + 1) * wl.L)
        gq, gk, gv = oracle.chunk_bwd(q[0, rows], k[0, a:e], v[0, a:e], do[0, rows], wl.cu[0], wl.S, c * wl.L,
                                      kv_base=a)
        grad_check(dq[0, c].cpu(), gq, "dQ chunk")
        grad_check(dk[0, c, : e - a].cpu(), gk, "dK partial")
        grad_check(dv[0, c, : e - a].cpu(), gv, "dV partial")


def test_bwd_accumulate_single_chunk_calls():
    """Successive single-chunk calls with accumulate_dkv=1 sum the chunk partials
    into one all-gathered K/V gradient (the reduce-scatter SUM done in place)."""
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    full = run_bwd(wl, q, k, v, do, 0)
    qd, dod = gu.as_chunks(q.cuda(), wl.cp), gu.as_chunks(do.cuda(), wl.cp)
    kd, vd = k.cuda().unsqueeze(1), v.cuda().unsqueeze(1)
    dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    for r in range(wl.cp):
        plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, ranks=[r]).upload("cuda")
        out = torch.empty_like(qd[:, r:r + 1])
        lse = torch.empty(wl.B, 1, wl.H, wl.L, dtype=torch.float32, device="cuda")
        bd.bd_attn_fwd(plan, qd[:, r:r + 1], kd, vd, out, lse, row_offset=r * wl.L)
        ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
        bd.bd_attn_bwd(plan, qd[:, r:r + 1], kd, vd, out, dod[:, r:r + 1], lse, dq[:, r:r + 1], dk, dv, ws,
                       accumulate_dkv=True)
    torch.cuda.synchronize()
    grad_check(dk.view_as(full[1]).cpu(), full[1].double(), "dK accumulated")
    grad_check(dv.view_as(full[2]).cpu(), full[2].double(), "dV accumulated")
    grad_check(dq.view_as(full[0]).cpu(), full[0].double(), "dQ per chunk")


def _sample_cols(wl, b, rng, n_tail=12, n_rand=12):
    """Key columns whose attending rows are few: the last rows of each document."""
    cu = wl.cu[b]
    cols = set()
    for d in range(len(cu) - 1):
        a, e = cu[d], cu[d + 1]
        if e <= a:
            continue
        cols.update(range(max(a, e - n_tail), e))
        lo = max(a, e - 384)
        cols.update(int(x) for x in rng.integers(lo, e, size=min(n_rand, e - lo)))
    if cu[-1] < wl.S:
        cols.update({cu[-1], wl.S - 1})
    return sorted(cols)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("i", [3, 4, 5])
def test_bwd_sampled_full_size(i, mode):
    wl = workloads.config(i)
    q, k, v, do = workloads.tensors(wl)
    dq, dk, dv = run_bwd(wl, q, k, v, do, mode)
    rng = np.random.default_rng(i)
    for b in range(wl.B):
        if wl.cu[b][-1] == 0:
            assert not dq[b].any() and not dk[b].any() and not dv[b].any()
            continue
        rows = gu.sample_rows(wl, b, n_rand=16 if i == 4 else 24)
        grad_check(dq[b, rows], oracle.attention_bwd_rows(q[b], k[b], v[b], do[b], wl.cu[b], rows), "dQ rows")
        cols = _sample_cols(wl, b, rng, n_tail=8 if i == 5 else 12, n_rand=4 if i == 5 else 12)
        if i == 5:
            cols = cols[:: max(1, len(cols) // 96)]
        gk, gv = oracle.attention_bwd_cols(q[b], k[b], v[b], do[b], wl.cu[b], cols)
        grad_check(dk[b, cols], gk, "dK cols")
        grad_check(dv[b, cols], gv, "dV cols")
        # identities over every document at full size: sum_j dV_j = sum_i dO_i (per K/V
        # head, over its query heads), sum_j dK_j = 0
        G = wl.H // wl.Hkv
        cu = wl.cu[b]
        for d in range(len(cu) - 1):
            a, e = cu[d], cu[d + 1]
            if e <= a:
                continue
            sv = dv[b, a:e].double().sum(0)                                   # [Hkv, d]
            so = do[b, a:e].double().view(e - a, wl.Hkv, G, wl.d).sum((0, 2))
            assert (sv - so).abs().max().item() <= 2e-2 * max(1.0, so.abs().max().item())
            # sum_j dK_j = 0 is exact only before bf16 rounding of O (inside D) and of
            # dS; on documents of a few tokens that residual is comparable to the
            # few-term L1 norm, so the identity is checked where it has many terms
            if e - a >= 64:
                sk = dk[b, a:e].double().sum(0)
                l1 = dk[b, a:e].double().abs().sum(0)
                assert (sk.abs() <= 2e-2 * l1 + 1e-4).all()
        pad = wl.cu[b][-1]
        assert not dq[b, pad:].any() and not dk[b, pad:].any() and not dv[b, pad:].any()


def test_bwd_window_matches_gather():
    wl = workloads.config(3)
    q, k, v, do = workloads.tensors(wl)
    g = run_bwd(wl, q, k, v, do, 0)
    w = run_bwd(wl, q, k, v, do, 1)
    for x, y, n in zip(g, w, ("dQ", "dK", "dV")):
        assert gu.max_rel(y, x) <= 1e-2, n


def test_bwd_dkv_deterministic():
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    a = run_bwd(wl, q, k, v, do, 0)
    b = run_bwd(wl, q, k, v, do, 0)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert gu.max_rel(a[0], b[0]) <= 1e-5   # dQ sums in arrival order


def test_claim_counters_reset_between_launches():
    """The forward takes its work units from counter slots in the device plan (one
    slot per launch, in turn) and the backward main kernel from counters in its
    workspace; the last CTA of each launch returns them to zero, so the same
    uploaded plan and workspace serve launch after launch with identical results."""
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    mode = bd.BD_KV_WINDOW
    plan, out1, lse1, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, mode)
    slots = slice(38, 38 + 2 * 8)  # the forward's (claim, done) slots
    assert torch.count_nonzero(plan.dev[slots]).item() == 0
    out2 = torch.empty_like(out1)
    lse2 = torch.empty_like(lse1)
    for _ in range(9):   # every slot used at least once
        bd.bd_attn_fwd(plan, qd, kd, vd, out2, lse2)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    nws = bd.bd_attn_bwd_workspace(plan)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    grads = []
    for _ in range(2):
        dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
        dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")  # window rows past kv_end stay unwritten
        dv = torch.zeros_like(dk)
        bd.bd_attn_bwd(plan, qd, kd, vd, out1, dod, lse1, dq, dk, dv, ws)
        grads.append((dq, dk, dv))
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    assert torch.count_nonzero(plan.dev[slots]).item() == 0
    ctr = ws[nws - 256:nws - 248].view(torch.int32)   # the backward's (claim, done)
    assert torch.count_nonzero(ctr).item() == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    (dq1, dk1, dv1), (dq2, dk2, dv2) = grads
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)   # dK/dV accumulate in TMEM: deterministic
    assert gu.max_rel(dq2, dq1) < 1e-5                        # dQ adds in arrival order


def test_overlapping_launches_on_one_plan():
    """Forward launches that share one device plan and run at the same time on
    unordered streams each take a counter slot of their own and give the outputs
    of a lone launch; so do backward launches sharing the plan but with a
    workspace each."""
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    plan, out_ref, lse_ref, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_GATHER)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = [(torch.empty_like(out_ref), torch.empty_like(lse_ref)) for _ in streams]
    grads = [(torch.empty(qd.shape, dtype=torch.float32, device="cuda"),
              torch.empty(kd.shape, dtype=torch.float32, device="cuda"),
              torch.empty(kd.shape, dtype=torch.float32, device="cuda"),
              torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")) for _ in streams]
    torch.cuda.synchronize()
    for rep in range(3):
        for s, (o, l) in zip(streams, outs):
            bd.bd_attn_fwd(plan, qd, kd, vd, o, l, stream=s)
        torch.cuda.synchronize()
        for o, l in outs:
            assert torch.equal(o, out_ref) and torch.equal(l, lse_ref), f"forward, round {rep}"
        for s, (dq, dk, dv, ws) in zip(streams, grads):
            bd.bd_attn_bwd(plan, qd, kd, vd, out_ref, dod, lse_ref, dq, dk, dv, ws, stream=s)
        torch.cuda.synchronize()
        bd.bd_check_status(plan)
        for dq, dk, dv, _ in grads[1:]:
            assert torch.equal(dk, grads[0][1]) and torch.equal(dv, grads[0][2]), f"backward, round {rep}"
            assert gu.max_rel(dq, grads[0][0]) < 1e-5


def test_pre_without_clearing_after_caller_zeroes_dq():
    """bd_attn_bwd_pre_ex with clear_dq = 0 and a dq the caller zeroed on another
    stream gives the gradients of the clearing form."""
    wl = workloads.config(2)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_GATHER)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    res = []
    for clear in (True, False):
        dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
        if not clear:
            side = torch.cuda.Stream()
            with torch.cuda.stream(side):
                dq.zero_()
            torch.cuda.current_stream().wait_stream(side)
        dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
        dv = torch.zeros_like(dk)
        bd.bd_attn_bwd_pre(plan, out, dod, lse, dq, ws, clear_dq=clear)
        bd.bd_attn_bwd_main(plan, qd, kd, vd, dod, dq, dk, dv, ws)
        torch.cuda.synchronize()
        res.append((dq.cpu(), dk.cpu(), dv.cpu()))
    (dq1, dk1, dv1), (dq2, dk2, dv2) = res
    assert torch.isfinite(dq2).all() and gu.max_rel(dq2, dq1) < 1e-5
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


def test_owner_sum_store_writes_every_owner_row():
    """bd_owner_sum_ex with accumulate = 0 stores the window sums into owner
    buffers that start as NaN: every row is written (padding rows with zeros) and
    the result equals adding into zeroed buffers, bit for bit."""
    wl = workloads.config(3)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_WINDOW)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws)
    shape = (wl.B, 1, wl.S, wl.Hkv, wl.d)
    add_k = torch.zeros(shape, dtype=torch.float32, device="cuda")
    add_v = torch.zeros_like(add_k)
    bd.bd_owner_sum(plan, dk, dv, add_k, add_v)
    st_k = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    st_v = torch.full_like(st_k, float("nan"))
    bd.bd_owner_sum(plan, dk, dv, st_k, st_v, accumulate=False)
    torch.cuda.synchronize()
    assert torch.equal(st_k, add_k) and torch.equal(st_v, add_v)
    pad = wl.cu[0][-1]
    assert not st_k[0, 0, pad:].any() and not st_v[0, 0, pad:].any()
