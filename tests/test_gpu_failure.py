"""Failure detection without a GPU fault: a kernel's bounded wait on an mbarrier
that nothing arrives at gives up after a short limit, records the failure in the
plan's status word, and the host reads it as BD_ERR_DEVICE_TIMEOUT; the context
stays usable. Host-side validation rejects bad inputs before any launch."""
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


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = bd.load()
    wl = workloads.config(1)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d).upload("cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.bd_selftest_bounded_wait(plan.dev_ptr, 5000, stream) == 0
    st = lib.bd_check_status(plan.dev_ptr, 1, stream)
    assert st == bd._abi.BD_ERR_DEVICE_TIMEOUT, st
    assert b"timed out" in lib.bd_last_error()
    assert lib.bd_check_status(plan.dev_ptr, 0, stream) == 0   # reset above
    # the context still runs real work correctly
    q, k, v, _ = workloads.tensors(wl)
    _, out, lse, _ = gu.run_fwd(wl, q, k, v, 0)
    assert torch.isfinite(out.float()).all()


def test_selftest_rejects_bad_arguments():
    lib = bd.load()
    wl = workloads.config(1)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d).upload("cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.bd_selftest_bounded_wait(plan.dev_ptr, 0, stream) == bd._abi.BD_ERR_ARG
    assert lib.bd_selftest_bounded_wait(None, 10, stream) == bd._abi.BD_ERR_ARG
