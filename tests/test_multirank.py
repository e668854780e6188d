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


def _xchg_worker(rank, world, port, cu, S, H, Hkv, d, out_q):
    """Needed-only exchange driven by the library's transfer plans."""
    import block_causal_varlen_gb300 as bd
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = torch.Generator().manual_seed(321)
        q = torch.randn(S, H, d, generator=g, dtype=torch.float64)
        k = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
        v = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
        do = torch.randn(S, H, d, generator=g, dtype=torch.float64)
        L = S // world
        own = slice(rank * L, (rank + 1) * L)
        kv_own = torch.stack([k[own], v[own]])                 # this rank's rows only
        plans = [bd.bd_exchange_plan(cu, S, world, r)[1] for r in range(world)]
        # forward: every rank sends the rows each receiver's plan asks of it
        send = [torch.cat([kv_own[:, x[1] - rank * L: x[1] - rank * L + x[2]] for x in plans[t] if x[0] == rank],
                          dim=1) if any(x[0] == rank for x in plans[t]) else torch.zeros(2, 0, Hkv, d, dtype=torch.float64)
                for t in range(world)]
        recv_sizes = [sum(x[2] for x in plans[rank] if x[0] == src) for src in range(world)]
        recv = [torch.empty(2, n, Hkv, d, dtype=torch.float64) for n in recv_sizes]
        reqs = []
        for t in range(world):
            if t != rank and send[t].shape[1]:   # receivers post a recv exactly for non-empty slices
                reqs.append(dist.isend(send[t].contiguous(), t))
        for src in range(world):
            if src == rank:
                recv[src] = send[rank]
            elif recv_sizes[src]:
                dist.recv(recv[src], src)
        for rq in reqs:
            rq.wait()
        W = sum(x[2] for x in plans[rank])
        win = torch.zeros(2, W, Hkv, d, dtype=torch.float64)
        off = {src: 0 for src in range(world)}
        for src, row, n, dst in plans[rank]:
            win[:, dst:dst + n] = recv[src][:, off[src]:off[src] + n]
            off[src] += n
        seg = oracle.segment_chunk(cu, S, world, rank)["hdr"]
        a = seg["kv_start"]
        err_win = (win - torch.stack([k[a:a + W], v[a:a + W]])).abs().max().item() if W else 0.0
        o, _ = oracle.chunk_fwd(q[own], win[0], win[1], cu, S, rank * L, kv_base=a)
        _, dkw, dvw = oracle.chunk_bwd(q[own], win[0], win[1], do[own], cu, S, rank * L, kv_base=a)
        # backward: window partials go back to their owners (index_add there)
        part = torch.stack([dkw, dvw])
        back = [torch.cat([part[:, x[3]:x[3] + x[2]] for x in plans[rank] if x[0] == t], dim=1)
                if any(x[0] == t for x in plans[rank]) else torch.zeros(2, 0, Hkv, d, dtype=torch.float64)
                for t in range(world)]
        acc = torch.zeros(2, L, Hkv, d, dtype=torch.float64)
        reqs = [dist.isend(back[t].contiguous(), t) for t in range(world) if t != rank and back[t].shape[1]]
        for src in range(world):
            rows = [x for x in plans[src] if x[0] == rank]
            if not rows:
                continue
            n = sum(x[2] for x in rows)
            buf = back[rank] if src == rank else torch.empty(2, n, Hkv, d, dtype=torch.float64)
            if src != rank:
                dist.recv(buf, src)
            o2 = 0
            for _, row, cnt, _ in rows:
                acc[:, row - rank * L: row - rank * L + cnt] += buf[:, o2:o2 + cnt]
                o2 += cnt
        for rq in reqs:
            rq.wait()
        _, gk, gv, go, _ = oracle.attention_bwd(q, k, v, do, cu)
        out_q.put((rank, {"win": err_win, "o": (o - go[own]).abs().max().item(),
                          "dk": (acc[0] - gk[own]).abs().max().item(),
                          "dv": (acc[1] - gv[own]).abs().max().item()}))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,cu,S", [
    (2, [0, 10, 24, 30], 32),          # halo from the left neighbour
    (4, [0, 3, 29], 32),               # all-to-all-v: a document spans four ranks
    (4, [0, 5, 9, 20, 32], 32),        # mixed
])
def test_needed_only_exchange_over_gloo(world, cu, S):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_xchg_worker, args=(r, world, port, cu, S, 4, 2, 8, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, res in results.items():
        for key, val in res.items():
            assert val < 1e-12, (r, key, val)
