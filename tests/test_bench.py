"""Host logic of bench.py on the CPU: workload selection, tile statistics, the
source digest that keeps recorded DRAM counters honest, the peaks file, the
reference arm's JSON line and the GPU arm's refusal to run without a GPU."""
import argparse
import importlib.util
import json
import math
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_head_dim_override_renames_the_workload():
    b = _bench()
    wl = b.bench_workload(argparse.Namespace(workload=3, head_dim=256))
    assert wl.d == 256 and wl.name == "lognormal_s16384_h32kv8_d256_cp4_window"
    wl = b.bench_workload(argparse.Namespace(workload=4, head_dim=0))
    assert wl.d == 128 and wl.name == "single_doc_s49152_h32kv8_d128_cp8"


def test_tile_stats_single_document_is_dense_causal():
    """One document over the whole sequence: nothing can be skipped, and the
    dense causal count per head is the closed form sum over chunks and query
    tiles of the key tiles up to the diagonal."""
    lib = pytest.importorskip("block_causal_varlen_gb300")
    b = _bench()
    import workloads
    wl = workloads.config(4)
    plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d)
    st = b.tile_stats(plan, wl)
    n = wl.S // 128
    assert st["dense_causal_per_head"] == n * (n + 1) // 2
    assert st["visited_per_head"] == st["dense_causal_per_head"] and st["skipped_fraction"] == 0.0


def test_tile_stats_lognormal_layout():
    lib = pytest.importorskip("block_causal_varlen_gb300")
    b = _bench()
    import workloads
    wl = workloads.config(3)
    plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=lib.BD_KV_WINDOW)
    st = b.tile_stats(plan, wl)
    n = wl.S // 128
    assert st["dense_causal_per_head"] == n * (n + 1) // 2
    assert 0 < st["visited_per_head"] < st["dense_causal_per_head"]
    assert math.isclose(st["skipped_fraction"], 1 - st["visited_per_head"] / st["dense_causal_per_head"])


def _copy_sources(tmp_path):
    dst = tmp_path / "block_causal_varlen_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "block_causal_varlen_gb300", "csrc"), dst)
    return dst


def test_source_digest_ignores_comments_but_not_code(tmp_path):
    b = _bench()
    src = _copy_sources(tmp_path)
    b.ROOT = str(tmp_path)
    base = {k: b.kernel_source_digest(k) for k in b.KERNEL_SOURCES}
    f = src / "attn_fwd.cu"
    text = f.read_text()
    f.write_text("// a new comment line\n\n" + text.replace("#include", "/* block\ncomment */\n#include", 1))
    assert b.kernel_source_digest("bd_fwd_kernel") == base["bd_fwd_kernel"]
    f.write_text(text + "\nstatic int bd_unused_marker = 1;\n")
    assert b.kernel_source_digest("bd_fwd_kernel") != base["bd_fwd_kernel"]
    assert b.kernel_source_digest("bd_bwd_kernel") == base["bd_bwd_kernel"]   # another kernel's sources


def test_recorded_traffic_is_dropped_once_sources_change(tmp_path):
    b = _bench()
    src = _copy_sources(tmp_path)
    (tmp_path / "profiles").mkdir()
    b.ROOT = str(tmp_path)
    rec = {"bd_bwd_kernel:wl": {"bytes": 123, "source_sha256": b.kernel_source_digest("bd_bwd_kernel")}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert b.kernel_traffic("bd_bwd_kernel", "wl") == 123
    assert b.kernel_traffic("bd_bwd_kernel", "other_workload") is None
    (src / "attn_bwd.cu").write_text((src / "attn_bwd.cu").read_text() + "\nstatic int bd_unused_marker = 2;\n")
    assert b.kernel_traffic("bd_bwd_kernel", "wl") is None


def test_peaks_file_and_fallback(tmp_path):
    b = _bench()
    b.ROOT = str(tmp_path)
    pk, src = b.peaks()
    assert src == "fallback" and pk == b.FALLBACK
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6748.0, "bf16_tflops": {"value": 1910.4}, "bf16_tflops_sustained": 1713.8}))
    pk, src = b.peaks()
    assert src == "measured" and pk == {"hbm_gbs": 6748.0, "bf16_tflops": 1910.4, "bf16_tflops_sustained": 1713.8}


def _run(args, timeout=600):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, cwd=ROOT, env=env)


def test_reference_arm_prints_one_json_line():
    r = _run(["--impl", "reference", "--workload", "1", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["value"] > 0 and j["steps"] == 2 and j["warmup"] == 1
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["cpu_model"] and j["cpu_baseline"]["blas"] and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["value"] == j["value"]
    assert j["config"]["workload"] == "tiny_s512_3docs_h4_d64_cp2" and j["config"]["d"] == 64


def test_our_arm_refuses_to_run_without_a_gpu():
    r = _run(["--workload", "1", "--steps", "1", "--warmup", "3", "--no-cpu", "--no-e2e"], timeout=300)
    assert r.returncode != 0 and "needs a CUDA GPU" in (r.stderr + r.stdout)


def test_plan_timing_reports_build_and_size_on_the_host():
    lib = pytest.importorskip("block_causal_varlen_gb300")
    b = _bench()
    import workloads
    wl = workloads.config(3)
    plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=lib.BD_KV_WINDOW)
    out = b.plan_timing(lib, plan, wl, lib.BD_KV_WINDOW, "cpu", reps=2)
    assert out["bytes"] == plan.host.nbytes > 0 and out["build_ms"] > 0 and "error" not in out


def test_reference_arm_under_torchrun_prints_once():
    """Launched like the multi-GPU runs (torchrun, two ranks on 127.0.0.1): rank 0
    alone prints the JSON line, every rank exits 0."""
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--workload", "1", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
