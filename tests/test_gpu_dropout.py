"""GPU attention dropout: forward O / LSE and backward dQ, dK, dV through the
C ABI against the dropout oracle on the same seeded bf16 inputs, same keep mask
(Philox4x32-10, regenerated on both sides from the seed)."""
import dataclasses

import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("block_causal_varlen_gb300")
gu = pytest.importorskip("gpu_util")

SEED = 0x0123456789ABCDEF


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    bd.load()


def _odd_chunks():
    """A layout whose chunk length is odd (L = 201): query rows of chunk 1 start
    on an odd row, which takes the backward's unaligned keep-bit path."""
    wl = workloads.config(1)
    return dataclasses.replace(wl, name="odd_chunks_s402", S=402, cp=2, cu=[[0, 150, 300, 402]])


def _run(wl, mode, p, seed):
    q, k, v, do = workloads.tensors(wl)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode)
    plan.set_dropout(p, seed).upload("cuda")
    qd = gu.as_chunks(q.cuda(), wl.cp)
    if mode == bd.BD_KV_GATHER:
        kd, vd = k.cuda().unsqueeze(1), v.cuda().unsqueeze(1)
    else:
        kd, vd, _ = gu.windows(plan, k.cuda(), v.cuda())
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((wl.B, wl.cp, wl.H, wl.L), float("nan"), dtype=torch.float32, device="cuda")
    bd.bd_attn_fwd(plan, qd, kd, vd, out, lse)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws)
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    return plan, (q, k, v, do), out.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def _check(wl, mode, p, seed):
    plan, (q, k, v, do), out, lse, dq, dk, dv = _run(wl, mode, p, seed)
    for b in range(wl.B):
        for r in range(wl.cp):
            rows = slice(r * wl.L, (r + 1) * wl.L)
            hdr, _ = plan.chunk(b * wl.cp + r)
            a = 0 if mode == bd.BD_KV_GATHER else hdr["kv_start"]
            e = wl.S if mode == bd.BD_KV_GATHER else hdr["kv_end"]
            o_ref, l_ref = oracle.chunk_fwd_dropout(q[b, rows], k[b, a:e], v[b, a:e], wl.cu[b], wl.S, r * wl.L,
                                                    p, seed, b=b, kv_base=a)
            gu.o_check(out[b, r].float(), o_ref)
            gu.lse_check(lse[b, r], l_ref)
            dq_ref, dk_ref, dv_ref = oracle.chunk_bwd_dropout(q[b, rows], k[b, a:e], v[b, a:e], do[b, rows],
                                                              wl.cu[b], wl.S, r * wl.L, p, seed, b=b, kv_base=a)
            assert gu.max_rel(dq[b, r], dq_ref) <= gu.GRAD_REL
            if mode == bd.BD_KV_WINDOW:
                n = e - a
                assert gu.max_rel(dk[b, r, :n], dk_ref) <= gu.GRAD_REL
                assert gu.max_rel(dv[b, r, :n], dv_ref) <= gu.GRAD_REL
    if mode == bd.BD_KV_GATHER:
        for b in range(wl.B):
            _, dk_ref, dv_ref, _, _ = oracle.attention_bwd_dropout(q[b], k[b], v[b], do[b], wl.cu[b], p, seed, b=b)
            assert gu.max_rel(dk[b, 0], dk_ref) <= gu.GRAD_REL
            assert gu.max_rel(dv[b, 0], dv_ref) <= gu.GRAD_REL


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("p", [0.1, 0.4])
def test_dropout_tiny_layout(mode, p):
    _check(workloads.config(1), mode, p, SEED)


@pytest.mark.parametrize("mode", [0, 1])
def test_dropout_llama_shaped_layout(mode):
    _check(workloads.config(2), mode, 0.2, SEED + 1)


def test_dropout_odd_chunk_length():
    _check(_odd_chunks(), bd.BD_KV_WINDOW, 0.3, SEED + 2)


def test_zero_probability_equals_plain_kernels():
    wl = workloads.config(1)
    r0 = _run(wl, bd.BD_KV_WINDOW, 0.0, SEED)
    q, k, v, _ = workloads.tensors(wl)
    plan, out, lse, _ = gu.run_fwd(wl, q, k, v, bd.BD_KV_WINDOW)
    assert torch.equal(r0[2], out.cpu()) and torch.equal(r0[3], lse.cpu())


def test_same_seed_same_result_other_seed_differs():
    wl = workloads.config(1)
    a = _run(wl, bd.BD_KV_GATHER, 0.3, 7)
    b = _run(wl, bd.BD_KV_GATHER, 0.3, 7)
    c = _run(wl, bd.BD_KV_GATHER, 0.3, 8)
    assert torch.equal(a[2], b[2]) and torch.equal(a[5], b[5])
    assert not torch.equal(a[2], c[2])


def test_dropout_two_sequences():
    """Two sequences in one batched launch: the sequence index is a counter word,
    so each sequence gets its own mask."""
    wl = dataclasses.replace(workloads.config(1), name="two_seqs_s512", B=2, cu=[[0, 200, 350, 512], [0, 100, 300]])
    for mode in (bd.BD_KV_GATHER, bd.BD_KV_WINDOW):
        _check(wl, mode, 0.25, SEED + 3)


@pytest.mark.parametrize("i", [3, 4])
def test_dropout_full_size_sampled(i):
    """Full-size workloads in the launch configuration the benchmark times
    (needed-only windows, owner sums): O, LSE and dQ on sampled rows, dK / dV on
    sampled key columns, against the row / column dropout oracles."""
    import numpy as np
    wl = workloads.config(i)
    mode, p, seed = bd.BD_KV_WINDOW, 0.1, SEED + 9
    plan, (q, k, v, do), out, lse, dq, dkw, dvw = _run(wl, mode, p, seed)
    # owner rows from the window partials (what bd_owner_sum computes in the step)
    dk = torch.zeros(wl.B, 1, wl.S, wl.Hkv, wl.d, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    bd.bd_owner_sum(plan, dkw.cuda(), dvw.cuda(), dk, dv)
    torch.cuda.synchronize()
    dk, dv = dk.view(wl.B, wl.S, wl.Hkv, wl.d).cpu(), dv.view(wl.B, wl.S, wl.Hkv, wl.d).cpu()
    out = out.view(wl.B, wl.S, wl.H, wl.d)
    lse = lse.permute(0, 2, 1, 3).reshape(wl.B, wl.H, wl.S)
    dq = dq.view(wl.B, wl.S, wl.H, wl.d)
    rng = np.random.default_rng(i)
    b = 0
    cu = wl.cu[b]
    rows = gu.sample_rows(wl, b, n_rand=12 if i == 4 else 24)
    o_r, l_r, dq_r = oracle.attention_rows_dropout(q[b], k[b], v[b], do[b], cu, rows, p, seed, b=b)
    gu.o_check(out[b, rows].float(), o_r)
    gu.lse_check(lse[b][:, rows], l_r)
    assert gu.max_rel(dq[b, rows], dq_r) <= gu.GRAD_REL
    # key columns near document ends (few attending rows): the last rows of each document
    cols = sorted({e - 1 - t for e in cu[1:] for t in range(0, 6 if i == 4 else 3)} |
                  {int(x) for x in rng.integers(max(0, cu[-1] - 64), cu[-1], size=4)})
    dk_c, dv_c = oracle.attention_bwd_cols_dropout(q[b], k[b], v[b], do[b], cu, cols, p, seed, b=b)
    assert gu.max_rel(dk[b, cols], dk_c) <= gu.GRAD_REL
    assert gu.max_rel(dv[b, cols], dv_c) <= gu.GRAD_REL
