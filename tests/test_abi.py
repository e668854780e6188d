"""The C ABI library loads and exports every function include/bd_attn.h declares
(no compute call: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^BD_API\s+[\w\s\*]+?\b(bd_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ("bd_segment", "bd_attn_fwd", "bd_attn_bwd", "bd_plan_build", "bd_owner_sum"):
        assert want in names


def test_library_exports_every_declared_symbol():
    from block_causal_varlen_gb300 import _abi
    lib = _abi.load()
    raw = ctypes.CDLL(_abi.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name
        assert name in _abi.EXPORTS, f"binding lacks {name}"
    assert lib.bd_version() >= 100


def test_library_does_not_need_a_driver_to_load():
    # libcuda is resolved lazily through the runtime's entry-point query
    from block_causal_varlen_gb300 import _abi
    deps = os.popen(f"ldd {_abi.LIB_PATH}").read()
    assert "libcuda.so" not in deps


def test_python_binding_fails_loudly_without_the_library(tmp_path):
    from block_causal_varlen_gb300 import _abi
    saved = _abi._lib
    try:
        _abi._lib = None
        with pytest.raises(RuntimeError):
            _abi.load(str(tmp_path / "missing.so"))
    finally:
        _abi._lib = saved


def test_padded_len():
    from block_causal_varlen_gb300 import _abi
    lib = _abi.load()
    assert lib.bd_padded_len(16381, 4) == 16384
    assert lib.bd_padded_len(16384, 4) == 16384
    assert lib.bd_padded_len(0, 3) == 0


def test_binding_checks_dtypes_and_devices_before_the_library():
    """The C ABI carries no dtypes, so the binding rejects a wrong dtype (which would
    make a kernel read or write past a buffer) or a host tensor before any call."""
    import torch
    bd = pytest.importorskip("block_causal_varlen_gb300")
    plan = bd.Plan([[0, 200, 350, 512]], 512, 2, 4, 4, 64)
    bf = torch.zeros(1, 2, 256, 4, 64, dtype=torch.bfloat16)
    f32 = torch.zeros(1, 2, 256, 4, 64, dtype=torch.float32)
    kv = torch.zeros(1, 1, 512, 4, 64, dtype=torch.bfloat16)
    dkv = torch.zeros(1, 1, 512, 4, 64, dtype=torch.float32)
    lse = torch.zeros(1, 2, 4, 256, dtype=torch.float32)
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(TypeError, match="dq: dtype"):   # bf16 dq: fp32 reduce-adds would overrun it
        bd.bd_attn_bwd_main(plan, bf, kv, kv, bf, bf, kv, dkv, ws)
    with pytest.raises(TypeError, match="dout: dtype"):
        bd.bd_attn_bwd_pre(plan, bf, f32, lse, f32, ws)
    with pytest.raises(TypeError, match="dk_win: dtype"):
        bd.bd_owner_sum(plan, kv, dkv, dkv, dkv)
    with pytest.raises(TypeError, match="must be a CUDA tensor"):   # right dtypes, host memory
        bd.bd_attn_bwd(plan, bf, kv, kv, bf, bf, lse, f32, dkv, dkv, ws)
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        bd.bd_attn_fwd(plan, bf, kv, kv, bf, lse)


# declared entry points the binding serves through the Plan class rather than a
# module-level function of the same name, and the fault-path self-test
_VIA_PLAN = {"bd_plan_bytes": "Plan", "bd_plan_build": "Plan", "bd_plan_chunk": "Plan.chunk",
             "bd_plan_useful_pairs": "Plan.useful_pairs", "bd_plan_set_dropout": "Plan.set_dropout",
             "bd_selftest_bounded_wait": "tests only"}


def test_binding_has_a_function_for_every_declared_entry_point():
    bd = pytest.importorskip("block_causal_varlen_gb300")
    for name in _declared():
        if name in _VIA_PLAN:
            continue
        assert callable(getattr(bd, name, None)), f"binding lacks {name}"


def test_small_wrappers():
    import torch
    bd = pytest.importorskip("block_causal_varlen_gb300")
    assert bd.bd_padded_len(16381, 4) == 16384 and bd.bd_padded_len(0, 3) == 0
    with pytest.raises(bd.BDError):
        bd.bd_padded_len(5, 0)
    assert "cp" in bd.bd_last_error()
    assert bd.bd_version() >= 100 and bd.bd_attn_bwd_noalloc_capacity() >= 1 << 20
    plan = bd.Plan([[0, 200, 350, 512]], 512, 2, 4, 4, 64)
    bf = torch.zeros(1, 2, 256, 4, 64, dtype=torch.bfloat16)
    kv = torch.zeros(1, 1, 512, 4, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 4, 256, dtype=torch.float32)
    with pytest.raises(TypeError, match="dq: dtype"):
        bd.bd_attn_bwd_noalloc(plan, bf, kv, kv, bf, bf, lse, bf, kv, kv)
