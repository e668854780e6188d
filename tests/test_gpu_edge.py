"""GPU edge layouts through the C ABI, forward and backward, every element against
the oracle: zero-length and length-1 documents, documents ending exactly on a
tile or chunk edge, chunk lengths that are not multiples of the 128-row tile
(including odd ones), an all-padding chunk, one and four chunks."""
import dataclasses

import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("block_causal_varlen_gb300")
gu = pytest.importorskip("gpu_util")

LAYOUTS = {
    "zero_length_docs": (512, 2, [0, 50, 50, 200, 200, 512]),
    "length_one_docs": (512, 2, [0, 1, 2, 3, 4, 130, 131, 512]),
    "tile_and_chunk_edges": (512, 2, [0, 128, 256, 384, 512]),
    "odd_chunk_rows": (402, 2, [0, 150, 300, 402]),
    "ragged_tile_tail": (390, 3, [0, 77, 260, 389]),
    "all_padding_chunk": (512, 2, [0, 40, 100]),
    "one_chunk": (320, 1, [0, 100, 320]),
    "four_chunks_one_doc": (512, 4, [0, 512]),
}


def _wl(name, d):
    S, cp, cu = LAYOUTS[name]
    return dataclasses.replace(workloads.config(1), name=name, S=S, cp=cp, cu=[cu], H=4, Hkv=2, d=d)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    bd.load()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_edge_layout_fwd_bwd(name, mode, d):
    wl = _wl(name, d)
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
    cu = wl.cu[0]
    for r in range(wl.cp):
        rows = slice(r * wl.L, (r + 1) * wl.L)
        hdr, _ = plan.chunk(r)
        a = 0 if mode == bd.BD_KV_GATHER else hdr["kv_start"]
        e = wl.S if mode == bd.BD_KV_GATHER else hdr["kv_end"]
        o_ref, l_ref = oracle.chunk_fwd(q[0, rows], k[0, a:e], v[0, a:e], cu, wl.S, r * wl.L, kv_base=a)
        gu.o_check(out[0, r].float(), o_ref)
        gu.lse_check(lse[0, r], l_ref)
        dq_ref, dkw, dvw = oracle.chunk_bwd(q[0, rows], k[0, a:e], v[0, a:e], do[0, rows], cu, wl.S, r * wl.L,
                                            kv_base=a)
        assert torch.isfinite(dq[0, r]).all()
        assert gu.max_rel(dq[0, r], dq_ref) <= gu.GRAD_REL
        if mode == bd.BD_KV_WINDOW and e > a:
            assert gu.max_rel(dk[0, r, :e - a], dkw) <= gu.GRAD_REL
            assert gu.max_rel(dv[0, r, :e - a], dvw) <= gu.GRAD_REL
    if mode == bd.BD_KV_GATHER:
        dq_ref, dk_ref, dv_ref, o_ref, _ = oracle.attention_bwd(q[0], k[0], v[0], do[0], cu)
        assert gu.max_rel(dk[0, 0], dk_ref) <= gu.GRAD_REL
        assert gu.max_rel(dv[0, 0], dv_ref) <= gu.GRAD_REL
        # per document too: a wrong short document would hide under the tensor maximum
        assert gu.doc_rel(dq.view(wl.S, wl.H, wl.d), dq_ref, cu) <= gu.GRAD_REL
        assert gu.doc_rel(dk[0, 0], dk_ref, cu) <= gu.GRAD_REL
        assert gu.doc_rel(dv[0, 0], dv_ref, cu) <= gu.GRAD_REL
        assert gu.doc_rel(out[0].reshape(wl.S, wl.H, wl.d).float(), o_ref, cu) <= gu.O_REL
        # padding rows and columns: exact zeros
        sv = cu[-1]
        assert not dq.view(wl.S, wl.H, wl.d)[sv:].abs().sum().item()
        assert not dk[0, 0, sv:].abs().sum().item() and not dv[0, 0, sv:].abs().sum().item()


# Head counts that do not fill the statistics kernel's head blocks (at most
# 4096 / d heads of whole rows per 8 KB box: 40 heads at d 128 and 24 at d 256 leave
# the second block partly past H), odd small counts (3 heads at d 64: 16-row boxes
# of 384 pieces), on chunks of 201 rows (a box straddles L) whose last 22 rows are
# padding.
HEAD_SHAPES = [(40, 8, 128), (3, 1, 64), (24, 8, 256), (6, 2, 128)]


@pytest.mark.parametrize("H,Hkv,d", HEAD_SHAPES)
def test_head_counts_fwd_bwd(H, Hkv, d):
    cu = [0, 37, 150, 380]
    wl = dataclasses.replace(workloads.config(1), name=f"heads_{H}_{Hkv}_{d}", S=402, cp=2, cu=[cu], H=H, Hkv=Hkv,
                             d=d)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, bd.BD_KV_GATHER)
    dod = gu.as_chunks(do.cuda(), wl.cp)
    dq = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.zeros(kd.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, dq, dk, dv, ws)
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    out, lse, dq, dk, dv = (t.cpu() for t in (out, lse, dq, dk, dv))
    dq_ref, dk_ref, dv_ref, o_ref, l_ref = oracle.attention_bwd(q[0], k[0], v[0], do[0], cu)
    for r in range(wl.cp):
        rows = slice(r * wl.L, (r + 1) * wl.L)
        gu.o_check(out[0, r].float(), o_ref[rows])
        gu.lse_check(lse[0, r], l_ref[:, rows])
    assert torch.isfinite(dq).all()
    assert gu.max_rel(dq.reshape(wl.S, H, d), dq_ref) <= gu.GRAD_REL
    assert gu.max_rel(dk[0, 0], dk_ref) <= gu.GRAD_REL
    assert gu.max_rel(dv[0, 0], dv_ref) <= gu.GRAD_REL
    assert gu.doc_rel(dq.reshape(wl.S, H, d), dq_ref, cu) <= gu.GRAD_REL
    assert gu.doc_rel(dk[0, 0], dk_ref, cu) <= gu.GRAD_REL
    # padding rows: no gradient
    assert torch.count_nonzero(dq.reshape(wl.S, H, d)[cu[-1]:]) == 0
