"""Head dim 256 through the C ABI, forward and backward, against the oracle on
the same seeded bf16 inputs. The backward at this head dim takes 64-row query
steps and two passes over column halves of dK / dV / dQ (dQ^T added with
red.global), so these cases cover ragged 64-row tails, GQA groups, both K/V
modes, accumulation and dropout."""
import dataclasses

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


def _wl(base, **kw):
    return dataclasses.replace(workloads.config(base), name=f"d256_{base}", d=256, **kw)


def _bwd(wl, mode, p=0.0, seed=0):
    q, k, v, do = workloads.tensors(wl)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode)
    if p > 0:
        plan.set_dropout(p, seed)
    plan.upload("cuda")
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


def _check(wl, mode, p=0.0, seed=0):
    plan, (q, k, v, do), out, lse, dq, dk, dv = _bwd(wl, mode, p, seed)
    for b in range(wl.B):
        for r in range(wl.cp):
            rows = slice(r * wl.L, (r + 1) * wl.L)
            hdr, _ = plan.chunk(b * wl.cp + r)
            a = 0 if mode == bd.BD_KV_GATHER else hdr["kv_start"]
            e = wl.S if mode == bd.BD_KV_GATHER else hdr["kv_end"]
            args = (q[b, rows], k[b, a:e], v[b, a:e])
            if p > 0:
                o_ref, l_ref = oracle.chunk_fwd_dropout(*args, wl.cu[b], wl.S, r * wl.L, p, seed, b=b, kv_base=a)
                gq, gk, gv = oracle.chunk_bwd_dropout(*args, do[b, rows], wl.cu[b], wl.S, r * wl.L, p, seed, b=b,
                                                      kv_base=a)
            else:
                o_ref, l_ref = oracle.chunk_fwd(*args, wl.cu[b], wl.S, r * wl.L, kv_base=a)
                gq, gk, gv = oracle.chunk_bwd(*args, do[b, rows], wl.cu[b], wl.S, r * wl.L, kv_base=a)
            gu.o_check(out[b, r].float(), o_ref)
            gu.lse_check(lse[b, r], l_ref)
            assert torch.isfinite(dq[b, r]).all()
            assert gu.max_rel(dq[b, r], gq) <= gu.GRAD_REL
            if mode == bd.BD_KV_WINDOW and e > a:
                assert gu.max_rel(dk[b, r, :e - a], gk) <= gu.GRAD_REL
                assert gu.max_rel(dv[b, r, :e - a], gv) <= gu.GRAD_REL
    if mode == bd.BD_KV_GATHER:
        for b in range(wl.B):
            fn = oracle.attention_bwd_dropout if p > 0 else oracle.attention_bwd
            extra = (p, seed) if p > 0 else ()
            kw = {"b": b} if p > 0 else {}
            _, gk, gv, _, _ = fn(q[b], k[b], v[b], do[b], wl.cu[b], *extra, **kw)
            assert gu.max_rel(dk[b, 0], gk) <= gu.GRAD_REL
            assert gu.max_rel(dv[b, 0], gv) <= gu.GRAD_REL
            pad = wl.cu[b][-1]
            assert not dk[b, 0, pad:].any() and not dv[b, 0, pad:].any()


@pytest.mark.parametrize("mode", [0, 1])
def test_d256_tiny_mha(mode):
    _check(_wl(1), mode)


@pytest.mark.parametrize("mode", [0, 1])
def test_d256_gqa_4k(mode):
    """The 4k uniform-document layout with 8 query heads over 2 K/V heads."""
    _check(_wl(2, H=8, Hkv=2), mode)


def test_d256_gqa_8_to_1():
    _check(_wl(2, H=8, Hkv=1), bd.BD_KV_WINDOW)


def test_d256_odd_chunk_rows():
    """L = 201: chunk 1 starts on an odd row and every chunk ends in a ragged
    64-row step whose rows past L must not be added to dQ."""
    wl = dataclasses.replace(_wl(1), S=402, cp=2, cu=[[0, 150, 300, 402]])
    for mode in (bd.BD_KV_GATHER, bd.BD_KV_WINDOW):
        _check(wl, mode)


def test_d256_two_sequences():
    wl = dataclasses.replace(_wl(1), B=2, cu=[[0, 200, 350, 512], [0, 100, 300]])
    _check(wl, bd.BD_KV_GATHER)


@pytest.mark.parametrize("mode", [0, 1])
def test_d256_dropout(mode):
    _check(_wl(1), mode, p=0.2, seed=0x5EED)


def test_d256_accumulate_into_shared_kv():
    """accumulate_dkv=1 adds both column halves onto what dK / dV held."""
    wl = _wl(1)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_GATHER)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    base = torch.randn(kd.shape, generator=torch.Generator().manual_seed(5)).cuda()
    dk, dv = base.clone(), 2 * base
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws, accumulate_dkv=True)
    torch.cuda.synchronize()
    _, gk, gv, _, _ = oracle.attention_bwd(q[0], k[0], v[0], do[0], wl.cu[0])
    assert gu.max_rel((dk - base)[0, 0].cpu(), gk) <= gu.GRAD_REL
    assert gu.max_rel((dv - 2 * base)[0, 0].cpu(), gv) <= gu.GRAD_REL


@pytest.mark.parametrize("i", [3, 4])
def test_d256_sampled_full_size(i):
    """The 16k lognormal and 49k single-document workloads at head dim 256, in the
    launch configuration the benchmark times with --head-dim 256 (needed-only
    windows for the 16k layout, owner sums): O, LSE and dQ on sampled rows, dK and
    dV on sampled key columns, against the row / column oracles."""
    import numpy as np
    from test_gpu_bwd import _sample_cols, run_bwd
    wl = dataclasses.replace(workloads.config(i), d=256)
    mode = bd.BD_KV_WINDOW if wl.kv_mode == "window" else bd.BD_KV_GATHER
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, _ = gu.run_fwd(wl, q, k, v, mode)
    out = out.cpu().view(wl.B, wl.S, wl.H, wl.d)
    lse = lse.cpu().permute(0, 2, 1, 3).reshape(wl.B, wl.H, wl.S)
    dq, dk, dv = run_bwd(wl, q, k, v, do, mode)
    b, cu = 0, wl.cu[0]
    rows = gu.sample_rows(wl, b, n_rand=8 if i == 4 else 16)
    o_r, l_r = oracle.attention_fwd(q[b], k[b], v[b], cu, rows=rows)
    gu.o_check(out[b, rows].float(), o_r)
    gu.lse_check(lse[b][:, rows], l_r)
    assert gu.max_rel(dq[b, rows], oracle.attention_bwd_rows(q[b], k[b], v[b], do[b], cu, rows)) <= gu.GRAD_REL
    cols = _sample_cols(wl, b, np.random.default_rng(i), n_tail=8, n_rand=8)
    gk, gv = oracle.attention_bwd_cols(q[b], k[b], v[b], do[b], cu, cols)
    assert gu.max_rel(dk[b, cols], gk) <= gu.GRAD_REL
    assert gu.max_rel(dv[b, cols], gv) <= gu.GRAD_REL
