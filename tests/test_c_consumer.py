"""include/bd_attn.h from C: a C99 program (tests/c/consumer.c) compiled with
-std=c99 -pedantic -Werror against the header, linked to libbd.so, calls the host
entry points. Its segmentation equals the hand-derived fixture bit for bit, and
the ABI structs have the sizes the Python binding assumes. No GPU is used."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "segment_tiny_3docs.txt")


@pytest.fixture(scope="module")
def consumer_output(tmp_path_factory):
    from block_causal_varlen_gb300 import _abi
    _abi.load()   # the library must have been built
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("c") / "consumer")
    libdir = os.path.dirname(_abi.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "consumer.c"), "-o", exe, "-L", libdir, "-lbd",
                    f"-Wl,-rpath,{libdir}"], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout.splitlines()


def test_c_segmentation_matches_the_fixture(consumer_output):
    want = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    got = [ln.split() for ln in consumer_output]
    assert got[0] == want[0]                                  # layout line
    chunks_w = [w for w in want if w[0] in ("chunk", "seg")]
    chunks_g = [g for g in got if g[0] in ("chunk", "seg")]
    assert len(chunks_w) == len(chunks_g)
    for w, g in zip(chunks_w, chunks_g):
        if w[0] == "chunk":   # the fixture adds the useful-pair count at the end
            assert g == w[:8]
        else:
            assert g == w
    # the plan built through bd_plan_desc gives the same chunk headers
    plan_chunks = [g[1:] for g in got if g[0] == "plan_chunk"]
    assert plan_chunks == [w[1:8] for w in want if w[0] == "chunk"]
    useful = sum(int(w[8]) for w in want if w[0] == "chunk")
    assert [g for g in got if g[0] == "useful"] == [["useful", str(useful)]]


def test_c_rejections_and_doc_ids(consumer_output):
    line = {ln.split()[0]: ln.split()[1:] for ln in consumer_output}
    assert line["doc_ids_to_cu"] == ["2", "0", "2", "5"]
    assert line["reject"] == ["-2", "-3", "-4"]   # BD_ERR_CU_SEQLENS, NOT_DIVISIBLE, RANK


def test_c_struct_sizes_match_the_binding(consumer_output):
    from block_causal_varlen_gb300 import _abi
    line = {ln.split()[0]: ln.split()[1:] for ln in consumer_output}
    want = [ctypes.sizeof(t) for t in (_abi.bd_segment_t, _abi.bd_chunk_hdr, _abi.bd_plan_desc, _abi.bd_tensor,
                                       _abi.bd_rowstat, _abi.bd_xfer_t)]
    assert [int(x) for x in line["sizeof"]] == want
    assert int(line["version"][0]) >= 100
