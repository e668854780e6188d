"""bd_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (no allocator is available to them, or a memory cap forbids one more
allocation). It takes its workspace from a fixed device array inside the
library instead of a caller buffer.

Called through the C ABI (ctypes), it must give the same gradients as
bd_attn_bwd with a caller workspace, on two calls in a row (the shared array
keeps the previous call's contents): dK / dV bit for bit (they accumulate in
a fixed order), dQ up to the order of its fp32 reduce-adds, also when adding
into existing dK / dV and at head dim 256 (its own kernel); and it must refuse
plans whose workspace does not fit the array before launching anything. This
file is collected last; it passes alone in a fresh process and after the other
tests."""
import ctypes as C
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


def _call_noalloc(lib, plan, qd, kd, vd, out, dod, lse, dq, dk, dv, accumulate=0):
    ts = [bd._tensor(x, n) for x, n in ((qd, "q"), (kd, "k"), (vd, "v"), (out, "out"), (dod, "dout"))]
    tl = bd._rowstat(lse, "lse")
    tq, tk, tv = bd._tensor(dq, "dq"), bd._tensor(dk, "dk"), bd._tensor(dv, "dv")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.bd_attn_bwd_noalloc(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts], C.byref(tl),
                                   C.byref(tq), C.byref(tk), C.byref(tv), accumulate, stream)


@pytest.mark.parametrize("i,mode,d,acc", [(2, bd.BD_KV_GATHER, 128, 0), (3, bd.BD_KV_WINDOW, 128, 0),
                                          (1, bd.BD_KV_GATHER, 256, 1), (2, bd.BD_KV_WINDOW, 256, 1)])
def test_noalloc_matches_workspace_backward_twice(i, mode, d, acc):
    lib = bd.load()
    wl = dataclasses.replace(workloads.config(i), d=d)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, mode)
    assert bd.bd_attn_bwd_workspace(plan) <= lib.bd_attn_bwd_noalloc_capacity()
    dod = gu.as_chunks(do.cuda(), wl.cp)
    g = torch.Generator().manual_seed(11)
    # dK / dV start from random values when adding into them, from zeros otherwise
    # (window rows past each chunk's window are not written)
    dk0 = torch.randn(kd.shape, generator=g).cuda() if acc else torch.zeros(kd.shape, device="cuda")
    dv0 = torch.randn(vd.shape, generator=g).cuda() if acc else torch.zeros(vd.shape, device="cuda")
    ref = [torch.empty(qd.shape, dtype=torch.float32, device="cuda"), dk0.clone(), dv0.clone()]
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, *ref, ws, accumulate_dkv=bool(acc))
    torch.cuda.synchronize()
    for call in range(2):
        got = [torch.full_like(ref[0], float("nan")), dk0.clone(), dv0.clone()]
        st = _call_noalloc(lib, plan, qd, kd, vd, out, dod, lse, *got, accumulate=acc)
        assert st == 0, lib.bd_last_error().decode()
        torch.cuda.synchronize()
        bd.bd_check_status(plan)
        assert torch.isfinite(got[0]).all(), f"call {call}: dQ not fully written"
        assert gu.max_rel(got[0].cpu(), ref[0].cpu()) <= 1e-5, f"call {call}: dQ"
        assert torch.equal(got[1], ref[1]), f"call {call}: dK differs from the workspace form"
        assert torch.equal(got[2], ref[2]), f"call {call}: dV differs from the workspace form"
    if i == 1:   # and against the oracle, sequence 0, all-gathered K/V
        gq, gk, gv, _, _ = oracle.attention_bwd(q[0], k[0], v[0], do[0], wl.cu[0])
        dq_, dk_, dv_ = (t.view(wl.S, -1, wl.d).cpu() for t in got)
        base_k = dk0.view(wl.S, -1, wl.d).cpu() if acc else 0
        base_v = dv0.view(wl.S, -1, wl.d).cpu() if acc else 0
        assert gu.max_rel(dq_, gq) <= gu.GRAD_REL
        assert gu.max_rel(dk_ - base_k, gk) <= gu.GRAD_REL
        assert gu.max_rel(dv_ - base_v, gv) <= gu.GRAD_REL


def test_noalloc_rejects_plans_beyond_its_capacity():
    lib = bd.load()
    # 64 heads x 65536 rows: the workspace is far above the fixed scratch
    plan = bd.Plan([[0, 65536]], 65536, 1, 64, 8, 128).upload("cuda")
    assert bd.bd_attn_bwd_workspace(plan) > lib.bd_attn_bwd_noalloc_capacity()
    qd = torch.empty(1, 1, 65536, 64, 128, dtype=torch.bfloat16, device="cuda")
    kd = torch.empty(1, 1, 65536, 8, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, 64, 65536, dtype=torch.float32, device="cuda")
    dq = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(kd.shape, dtype=torch.float32, device="cuda")
    st = _call_noalloc(lib, plan, qd, kd, kd, qd, qd, lse, dq, dk, dk)
    assert st == bd._abi.BD_ERR_CAPACITY
    assert b"scratch" in lib.bd_last_error()
