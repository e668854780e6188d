"""GQA 8:1 (32 query heads on 4 K/V heads) through the C ABI against the oracle:
forward O / LSE and backward dQ, dK, dV on the 4k Llama-shaped layout, both K/V
modes (the GPU varlen tests of the NeMo Automodel page cover GQA 8:1)."""
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


@pytest.mark.parametrize("mode", [0, 1])
def test_gqa_8_to_1(mode):
    wl = dataclasses.replace(workloads.config(2), name="llama8b_s4096_h32kv4_d128_cp2", Hkv=4)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, mode)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws)
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    out, lse, dq, dk, dv = (t.cpu() for t in (out, lse, dq, dk, dv))
    b = 0
    for r in range(wl.cp):
        rows = slice(r * wl.L, (r + 1) * wl.L)
        hdr, _ = plan.chunk(r)
        a = 0 if mode == bd.BD_KV_GATHER else hdr["kv_start"]
        e = wl.S if mode == bd.BD_KV_GATHER else hdr["kv_end"]
        o_ref, l_ref = oracle.chunk_fwd(q[b, rows], k[b, a:e], v[b, a:e], wl.cu[b], wl.S, r * wl.L, kv_base=a)
        gu.o_check(out[b, r].float(), o_ref)
        gu.lse_check(lse[b, r], l_ref)
        dq_ref, dkw, dvw = oracle.chunk_bwd(q[b, rows], k[b, a:e], v[b, a:e], do[b, rows], wl.cu[b], wl.S,
                                            r * wl.L, kv_base=a)
        assert gu.max_rel(dq[b, r], dq_ref) <= gu.GRAD_REL
        if mode == bd.BD_KV_WINDOW:
            assert gu.max_rel(dk[b, r, :e - a], dkw) <= gu.GRAD_REL
            assert gu.max_rel(dv[b, r, :e - a], dvw) <= gu.GRAD_REL
    if mode == bd.BD_KV_GATHER:
        _, dk_ref, dv_ref, _, _ = oracle.attention_bwd(q[b], k[b], v[b], do[b], wl.cu[b])
        assert gu.max_rel(dk[b, 0], dk_ref) <= gu.GRAD_REL
        assert gu.max_rel(dv[b, 0], dv_ref) <= gu.GRAD_REL
