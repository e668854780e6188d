"""bd_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (no allocator is available to them, or a memory cap forbids one more
allocation). It takes its workspace from a fixed device array inside the
library instead of a caller buffer.

Called through the C ABI (ctypes), it must give the same gradients as
bd_attn_bwd with a caller workspace, on two calls in a row (the shared array
keeps the previous call's contents), and must refuse plans whose workspace
does not fit the array before launching anything. This file is collected
last; it passes alone in a fresh process and after the other tests."""
import ctypes as C

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("block_causal_varlen_gb300")
gu = pytest.importorskip("gpu_util")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    bd.load()


def _call_noalloc(lib, plan, qd, kd, vd, out, dod, lse, dq, dk, dv):
    ts = [bd._tensor(x, n) for x, n in ((qd, "q"), (kd, "k"), (vd, "v"), (out, "out"), (dod, "dout"))]
    tl = bd._rowstat(lse, "lse")
    tq, tk, tv = bd._tensor(dq, "dq"), bd._tensor(dk, "dk"), bd._tensor(dv, "dv")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.bd_attn_bwd_noalloc(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts], C.byref(tl),
                                   C.byref(tq), C.byref(tk), C.byref(tv), 0, stream)


@pytest.mark.parametrize("i,mode", [(2, bd.BD_KV_GATHER), (3, bd.BD_KV_WINDOW)])
def test_noalloc_matches_workspace_backward_twice(i, mode):
    lib = bd.load()
    wl = workloads.config(i)
    q, k, v, do = workloads.tensors(wl)
    plan, out, lse, (qd, kd, vd) = gu.run_fwd(wl, q, k, v, mode)
    assert bd.bd_attn_bwd_workspace(plan) <= lib.bd_attn_bwd_noalloc_capacity()
    dod = gu.as_chunks(do.cuda(), wl.cp)
    ref = [torch.empty(qd.shape, dtype=torch.float32, device="cuda"),
           torch.empty(kd.shape, dtype=torch.float32, device="cuda"),
           torch.empty(vd.shape, dtype=torch.float32, device="cuda")]
    ws = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device="cuda")
    bd.bd_attn_bwd(plan, qd, kd, vd, out, dod, lse, *ref, ws)
    torch.cuda.synchronize()
    for call in range(2):
        got = [torch.full_like(t, float("nan")) for t in ref]
        st = _call_noalloc(lib, plan, qd, kd, vd, out, dod, lse, *got)
        assert st == 0, lib.bd_last_error().decode()
        torch.cuda.synchronize()
        bd.bd_check_status(plan)
        for g, r, name in zip(got, ref, ("dQ", "dK", "dV")):
            if mode == bd.BD_KV_WINDOW and name != "dQ":
                # rows past each chunk's window are not part of the result
                for c in range(wl.cp):
                    hdr, _ = plan.chunk(c)
                    n = hdr["kv_end"] - hdr["kv_start"]
                    g[:, c, n:] = 0
                    r[:, c, n:] = 0
            assert torch.isfinite(g).all(), f"call {call}: {name} not fully written"
            assert gu.max_rel(g.cpu(), r.cpu()) <= gu.GRAD_REL, f"call {call}: {name}"


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
