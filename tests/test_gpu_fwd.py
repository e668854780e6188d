"""GPU forward parity: the CUDA path (through the C ABI) against the oracle on
the same seeded bf16 inputs, on the five workloads, in both K/V exchange modes."""
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("block_causal_varlen_gb300")
gu = pytest.importorskip("gpu_util")

MODES = [0, 1]  # BD_KV_GATHER, BD_KV_WINDOW


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    bd.load()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("i", [1, 2])
def test_fwd_full_elementwise(i, mode):
    """Small workloads: every output element, every chunk, against the oracle's
    per-chunk forward (which itself equals whole-sequence attention)."""
    wl = workloads.config(i)
    q, k, v, _ = workloads.tensors(wl)
    plan, out, lse, _ = gu.run_fwd(wl, q, k, v, mode)
    out, lse = out.cpu(), lse.cpu()
    for b in range(wl.B):
        for r in range(wl.cp):
            rows = slice(r * wl.L, (r + 1) * wl.L)
            o_ref, l_ref = oracle.chunk_fwd(q[b, rows], k[b], v[b], wl.cu[b], wl.S, r * wl.L)
            gu.o_check(out[b, r].float(), o_ref)
            gu.lse_check(lse[b, r], l_ref)
        # per document too, over the whole sequence (a wrong short document would hide
        # under the tensor maximum)
        o_full, _ = oracle.attention_fwd(q[b], k[b], v[b], wl.cu[b], dtype=torch.float32 if i > 1 else torch.float64)
        assert gu.doc_rel(out[b].reshape(wl.S, wl.H, wl.d).float(), o_full, wl.cu[b]) <= gu.O_REL


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("i", [3, 4, 5])
def test_fwd_sampled_rows_full_size(i, mode):
    """Full-size workloads in the batched launch: sampled rows, every head."""
    wl = workloads.config(i)
    q, k, v, _ = workloads.tensors(wl)
    plan, out, lse, _ = gu.run_fwd(wl, q, k, v, mode)
    out = out.view(wl.B, wl.S, wl.H, wl.d).cpu()
    lse = lse.permute(0, 2, 1, 3).reshape(wl.B, wl.H, wl.S).cpu()
    for b in range(wl.B):
        rows = gu.sample_rows(wl, b, n_rand=24 if i == 4 else 40)
        o_ref, l_ref = oracle.attention_fwd(q[b], k[b], v[b], wl.cu[b], rows=rows)
        gu.o_check(out[b, rows].float(), o_ref)
        gu.lse_check(lse[b][:, rows], l_ref)
        if wl.cu[b][-1] == 0:   # the all-padding sequence: every row zero / -inf
            assert not out[b].float().abs().sum().item()
            assert torch.isneginf(lse[b]).all()


def test_fwd_outputs_fully_written_and_guard_bands_intact():
    """NaN-poisoned outputs are fully overwritten; bytes around them are untouched."""
    wl = workloads.config(2)
    q, k, v, _ = workloads.tensors(wl)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d).upload("cuda")
    qd = gu.as_chunks(q.cuda(), wl.cp)
    pad = 4096
    obuf = torch.full((2 * pad + q.numel(),), float("nan"), dtype=torch.bfloat16, device="cuda")
    obuf[:pad] = 7.0
    obuf[-pad:] = 7.0
    out = obuf[pad:pad + q.numel()].view_as(qd)
    lbuf = torch.full((2 * pad + wl.B * wl.cp * wl.H * wl.L,), 5.0, dtype=torch.float32, device="cuda")
    lse = lbuf[pad:-pad].view(wl.B, wl.cp, wl.H, wl.L)
    lse.fill_(float("nan"))
    bd.bd_attn_fwd(plan, qd, k.cuda().unsqueeze(1), v.cuda().unsqueeze(1), out, lse)
    torch.cuda.synchronize()
    assert not torch.isnan(out.float()).any() and not torch.isnan(lse).any()
    assert (obuf[:pad] == 7.0).all() and (obuf[-pad:] == 7.0).all()
    assert (lbuf[:pad] == 5.0).all() and (lbuf[-pad:] == 5.0).all()


@pytest.mark.parametrize("i", [1, 3])
def test_fwd_is_deterministic(i):
    wl = workloads.config(i)
    q, k, v, _ = workloads.tensors(wl)
    _, o1, l1, _ = gu.run_fwd(wl, q, k, v, 0)
    _, o2, l2, _ = gu.run_fwd(wl, q, k, v, 0)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_window_equals_gather_bitwise():
    wl = workloads.config(3)
    q, k, v, _ = workloads.tensors(wl)
    _, og, lg, _ = gu.run_fwd(wl, q, k, v, 0)
    _, ow, lw, _ = gu.run_fwd(wl, q, k, v, 1)
    assert torch.equal(og.view(torch.int16), ow.view(torch.int16))
    assert torch.equal(lg, lw)


def test_single_chunk_calls_equal_batched():
    """Per-rank calls (one plan per chunk, row_offset checked) equal the batched grid."""
    wl = workloads.config(2)
    q, k, v, _ = workloads.tensors(wl)
    _, ob, lb, _ = gu.run_fwd(wl, q, k, v, 0)
    qd = gu.as_chunks(q.cuda(), wl.cp)
    for r in range(wl.cp):
        plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, ranks=[r]).upload("cuda")
        out = torch.empty_like(qd[:, r:r + 1])
        lse = torch.empty(wl.B, 1, wl.H, wl.L, dtype=torch.float32, device="cuda")
        bd.bd_attn_fwd(plan, qd[:, r:r + 1], k.cuda().unsqueeze(1), v.cuda().unsqueeze(1), out, lse,
                       row_offset=r * wl.L)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ob[:, r:r + 1].view(torch.int16))
        assert torch.equal(lse, lb[:, r:r + 1])
        with pytest.raises(bd.BDError):
            bd.bd_attn_fwd(plan, qd[:, r:r + 1], k.cuda().unsqueeze(1), v.cuda().unsqueeze(1), out, lse,
                           row_offset=r * wl.L + 1)


def test_fwd_rejects_bad_tensors_before_launch():
    wl = workloads.config(1)
    q, k, v, _ = workloads.tensors(wl)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d).upload("cuda")
    qd = gu.as_chunks(q.cuda(), wl.cp)
    kd, vd = k.cuda().unsqueeze(1), v.cuda().unsqueeze(1)
    out = torch.empty_like(qd)
    lse = torch.empty(wl.B, wl.cp, wl.H, wl.L, dtype=torch.float32, device="cuda")
    with pytest.raises(bd.BDError):   # K shorter than the valid rows
        bd.bd_attn_fwd(plan, qd, kd[:, :, :100], vd, out, lse)
    with pytest.raises(bd.BDError):   # misaligned base
        bad = torch.empty(qd.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + qd.numel()].view_as(qd)
        bd.bd_attn_fwd(plan, bad, kd, vd, out, lse)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("base,H,Hkv", [(1, 4, 4), (2, 8, 2)])
def test_fwd_head_dim_256(base, H, Hkv, mode):
    """Head dim 256 (one query head per CTA): every element against the oracle,
    on the tiny layout (MHA) and the 4k layout with GQA 4:1."""
    import dataclasses
    wl = dataclasses.replace(workloads.config(base), name=f"d256_{base}", H=H, Hkv=Hkv, d=256)
    q, k, v, _ = workloads.tensors(wl)
    plan, out, lse, _ = gu.run_fwd(wl, q, k, v, mode)
    out, lse = out.cpu(), lse.cpu()
    for b in range(wl.B):
        for r in range(wl.cp):
            rows = slice(r * wl.L, (r + 1) * wl.L)
            o_ref, l_ref = oracle.chunk_fwd(q[b, rows], k[b], v[b], wl.cu[b], wl.S, r * wl.L)
            gu.o_check(out[b, r].float(), o_ref)
            gu.lse_check(lse[b, r], l_ref)
