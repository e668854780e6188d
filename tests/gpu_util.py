"""Helpers shared by the GPU parity tests: device tensors in the library's
layouts, needed-only K/V windows, tolerances and comparisons."""
from __future__ import annotations

import math

import numpy as np
import torch

import block_causal_varlen_gb300 as bd

# Tolerances (bf16 inputs, fp32 accumulation): O max-abs 2e-2 and max-rel 1e-2,
# LSE abs 1e-3 on valid rows (padding exactly -inf), gradients max-rel 5e-2,
# where max-rel = max|x - ref| / max|ref| over the compared tensor.
O_ABS, O_REL, LSE_ABS, GRAD_REL = 2e-2, 1e-2, 1e-3, 5e-2


def max_rel(x, ref):
    x = x.double()
    ref = ref.double()
    den = ref.abs().max().item()
    return (x - ref).abs().max().item() / (den if den > 0 else 1.0)


def as_chunks(t, cp):
    """[B, S, heads, d] -> view [B, cp, L, heads, d]."""
    B, S, Hh, d = t.shape
    return t.view(B, cp, S // cp, Hh, d)


def windows(plan, k, v):
    """Needed-only K/V windows [B, C, W, Hkv, d] gathered from full K/V [B, S, Hkv, d]."""
    B = k.shape[0]
    W = max(1, plan.kv_rows())
    kw = torch.zeros(B, plan.nchunks, W, k.shape[2], k.shape[3], dtype=k.dtype, device=k.device)
    vw = torch.zeros_like(kw)
    starts = []
    for b in range(B):
        row = []
        for c in range(plan.nchunks):
            hdr, _ = plan.chunk(b * plan.nchunks + c)
            a, e = hdr["kv_start"], hdr["kv_end"]
            kw[b, c, : e - a] = k[b, a:e]
            vw[b, c, : e - a] = v[b, a:e]
            row.append((a, e))
        starts.append(row)
    return kw, vw, starts


def run_fwd(wl, q, k, v, mode, device="cuda", poison=True):
    """Forward of every chunk of every sequence in one batched call."""
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode).upload(device)
    qd = as_chunks(q.to(device), wl.cp)
    if mode == bd.BD_KV_GATHER:
        kd = k.to(device).unsqueeze(1)
        vd = v.to(device).unsqueeze(1)
    else:
        kd, vd, _ = windows(plan, k.to(device), v.to(device))
    out = torch.empty_like(qd)
    lse = torch.empty(wl.B, wl.cp, wl.H, wl.L, dtype=torch.float32, device=device)
    if poison:
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
    bd.bd_attn_fwd(plan, qd, kd, vd, out, lse)
    torch.cuda.synchronize()
    bd.bd_check_status(plan)
    return plan, out, lse, (qd, kd, vd)


def sample_rows(wl, b, n_rand=48, seed=0):
    """Rows that exercise tile edges, chunk edges, document edges, padding and random rows."""
    rng = np.random.default_rng(seed + b)
    S, L = wl.S, wl.L
    cu = wl.cu[b]
    rows = {0, S - 1, L - 1, min(L, S - 1), 127, 128, 129}
    for x in cu:
        for dx in (-1, 0, 1):
            if 0 <= x + dx < S:
                rows.add(x + dx)
    for r in range(wl.cp):
        rows.update({r * L, r * L + 1, min(S - 1, r * L + L - 1)})
    rows.update(int(x) for x in rng.integers(0, S, size=n_rand))
    return sorted(rows)


def lse_check(got, want):
    """got/want fp32/fp64 [..]: -inf exactly where want is -inf, else |diff| <= LSE_ABS."""
    pad = torch.isneginf(want)
    assert torch.equal(torch.isneginf(got), pad), "padding rows must have LSE = -inf exactly"
    if (~pad).any():
        err = (got[~pad].double() - want[~pad].double()).abs().max().item()
        assert err <= LSE_ABS, f"LSE err {err}"
        return err
    return 0.0


def o_check(got, want):
    err_abs = (got.double() - want.double()).abs().max().item()
    err_rel = max_rel(got, want)
    assert math.isfinite(err_abs) and err_abs <= O_ABS and err_rel <= O_REL, (err_abs, err_rel)
    return err_abs, err_rel


def doc_rel(x, ref, cu, floor=1e-2):
    """Largest per-document max-rel over the documents of one sequence: rows
    [cu[k], cu[k+1]) of x / ref (dim 0 = row), each normalised by that document's
    own max|ref|, floored at `floor` x the whole tensor's max|ref| (a document whose
    exact values are ~0, e.g. dK of a one-token document, is judged against that
    floor instead of its own rounding noise)."""
    x = x.double()
    ref = ref.double()
    top = ref.abs().max().item()
    worst = 0.0
    for a, e in zip(cu[:-1], cu[1:]):
        if e <= a:
            continue
        den = max(ref[a:e].abs().max().item(), floor * top)
        if den > 0:
            worst = max(worst, (x[a:e] - ref[a:e]).abs().max().item() / den)
    return worst
