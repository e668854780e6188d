"""Multi-rank semantics on CPU with real gloo collectives (world size 2 and 4).

Each rank owns one contiguous query chunk (NeMo Automodel page
"block-diagonal varlen CP for packed sequences", Design overview, batch.py),
computes its chunk with the oracle over its needed-only K/V window, and:
  * the all-gathered chunk outputs equal full-sequence attention
    (Key correctness property 1);
  * reduce-scatter SUM of the per-chunk dK/dV partials over the whole
    sequence gives each rank its owned rows of the full gradient (the
    backward of the fused K/V all-gather, Design overview, exchange.py);
  * an all-padding rank takes part in every collective and contributes zeros.
This pins what a sharded run of the path must compute; the GPU path runs the
same chunks as one batched launch on one device.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cu, S, H, Hkv, d, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = torch.Generator().manual_seed(123)
        q = torch.randn(S, H, d, generator=g, dtype=torch.float64)
        k = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
        v = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
        do = torch.randn(S, H, d, generator=g, dtype=torch.float64)
        L = S // world
        seg = oracle.segment_chunk(cu, S, world, rank)["hdr"]
        a, e = seg["kv_start"], seg["kv_end"]
        rows = slice(rank * L, (rank + 1) * L)
        o, lse = oracle.chunk_fwd(q[rows], k[a:e], v[a:e], cu, S, rank * L, kv_base=a)
        dq, dkw, dvw = oracle.chunk_bwd(q[rows], k[a:e], v[a:e], do[rows], cu, S, rank * L, kv_base=a)
        # all-gather outputs
        o_all = [torch.empty_like(o) for _ in range(world)]
        dist.all_gather(o_all, o)
        dq_all = [torch.empty_like(dq) for _ in range(world)]
        dist.all_gather(dq_all, dq)
        # window partial -> full-length partial, then reduce-scatter SUM to owners
        dk_part = torch.zeros(S, Hkv, d, dtype=torch.float64)
        dv_part = torch.zeros(S, Hkv, d, dtype=torch.float64)
        dk_part[a:e] = dkw
        dv_part[a:e] = dvw
        dk_own = torch.empty(L, Hkv, d, dtype=torch.float64)
        dv_own = torch.empty(L, Hkv, d, dtype=torch.float64)
        dist.reduce_scatter(dk_own, list(dk_part.split(L)), op=dist.ReduceOp.SUM)
        dist.reduce_scatter(dv_own, list(dv_part.split(L)), op=dist.ReduceOp.SUM)
        # the full answer, for comparison
        gq, gk, gv, go, _ = oracle.attention_bwd(q, k, v, do, cu)
        res = {
            "o": (torch.cat(o_all) - go).abs().max().item(),
            "dq": (torch.cat(dq_all) - gq).abs().max().item(),
            "dk": (dk_own - gk[rows]).abs().max().item(),
            "dv": (dv_own - gv[rows]).abs().max().item(),
            "window": (a, e),
        }
        out_q.put((rank, res))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,cu,S", [
    (2, [0, 10, 24, 30], 32),          # a document straddles the rank boundary
    (4, [0, 3, 29], 32),               # one document spans three ranks
    (2, [0, 9, 14], 32),               # rank 1 is all padding
])
def test_chunks_over_gloo_ranks_equal_full_attention(world, cu, S):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cu, S, 4, 2, 8, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        r, res = q.get(timeout=120)
        results[r] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, res in results.items():
        for key in ("o", "dq", "dk", "dv"):
            assert res[key] < 1e-12, (r, key, res[key])
