"""Oracle for attention dropout: counter-based keep mask, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The NeMo Automodel page "block-diagonal varlen CP for packed sequences" lists
native Flash attention dropout among the paths it forwards and tests (Proof,
GPU varlen tests) but gives no formulas. The plain reading used here is
standard attention dropout on the normalised probabilities, with the keep mask
drawn from a counter-based generator so that the backward regenerates exactly
the mask the forward used:

    keep_ij = u_ij >= t,          t = floor(p * 2**32 + 1/2), at most 2**32 - 1 (p in [0, 1))
    P'_ij   = P_ij * keep_ij / (1 - p),   O_i = sum_j P'_ij v_j,   LSE unchanged
    D_i     = <dO_i, O_i>,        dP_ij = <dO_i, v_j>
    dS_ij   = P_ij * (keep_ij * dP_ij / (1 - p) - D_i)
    dV_j    = sum_i P'_ij dO_i,   dQ, dK from dS as without dropout.

(D_i = sum_k P'_ik dP_ik = <dO_i, O_i> because O is the dropped output.)

u_ij is word 2 (i mod 2) + (j mod 2) of Philox4x32-10 at counter
(j // 2, i // 2, h, b) under the key (seed mod 2**32, seed // 2**32), with i the
query row and j the key row of sequence b in global (sequence) rows and h the
query head: one call covers a 2 x 2 block of (query, key) pairs, so a thread
that walks keys of one row and a thread that walks queries of one key both use
two of each call's four words. Philox4x32-10 is
written from its published definition (Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011): ten rounds of

    (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key advanced by the Weyl increments
(0x9E3779B9, 0xBB67AE85) after each round.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .attention import _chunk_geometry, _heads, _softmax_block, block_causal_mask

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counters, key):
    """Philox4x32-10 of each row of ``counters`` (uint32 [N, 4]) under ``key`` (k0, k1).

    Returns uint32 [N, 4]."""
    c = np.asarray(counters, dtype=np.uint64).reshape(-1, 4).copy()
    k0, k1 = np.uint64(int(key[0]) & 0xFFFFFFFF), np.uint64(int(key[1]) & 0xFFFFFFFF)
    for _ in range(10):
        p0 = np.uint64(M0) * c[:, 0]
        p1 = np.uint64(M1) * c[:, 2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = np.stack([hi1 ^ c[:, 1] ^ k0, lo1, hi0 ^ c[:, 3] ^ k1, lo0], axis=1)
        k0 = (k0 + np.uint64(W0)) & MASK32
        k1 = (k1 + np.uint64(W1)) & MASK32
    return c.astype(np.uint32)


def keep_threshold(p: float) -> int:
    """The 32-bit threshold t of keep = (u >= t) for dropout probability p in [0, 1)."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(int(math.floor(p * 2.0 ** 32 + 0.5)), 2 ** 32 - 1)


def keep_mask(b: int, h: int, rows, cols, seed: int, p: float) -> torch.Tensor:
    """keep[i, j] for global query rows ``rows`` and key rows ``cols`` (bool [R, C])."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    t = keep_threshold(p)
    if t == 0:
        return torch.ones(len(rows), len(cols), dtype=torch.bool)
    rb, cb = np.unique(rows // 2), np.unique(cols // 2)
    cnt = np.zeros((len(rb), len(cb), 4), dtype=np.uint64)
    cnt[:, :, 0] = cb[None, :]
    cnt[:, :, 1] = rb[:, None]
    cnt[:, :, 2] = h
    cnt[:, :, 3] = b
    words = philox4x32_10(cnt.reshape(-1, 4), (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    words = words.reshape(len(rb), len(cb), 4)
    ri = np.searchsorted(rb, rows // 2)[:, None]
    ci = np.searchsorted(cb, cols // 2)[None, :]
    u = words[ri, ci, 2 * (rows % 2)[:, None] + (cols % 2)[None, :]]      # [R, C]
    return torch.from_numpy(u >= np.uint32(t))


def _dropout_block(b, h, rows, cols, p, seed, dtype):
    """keep / (1 - p) as a [R, C] tensor of ``dtype``."""
    return keep_mask(b, h, rows, cols, seed, p).to(dtype) / (1.0 - p)


def attention_fwd_dropout(q, k, v, cu, p: float, seed: int, b: int = 0, scale=None, dtype=torch.float64):
    """Full block-causal attention of sequence ``b`` with dropout. Returns O [S, H, d], LSE [H, S]."""
    S, H, d = q.shape
    G = _heads(H, k.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = block_causal_mask(cu, S)
    q, k, v = (t.to(dtype) for t in (q, k, v))
    ar = np.arange(S)
    o = torch.zeros(S, H, d, dtype=dtype)
    lse = torch.empty(H, S, dtype=dtype)
    for h in range(H):
        g = h // G
        lse[h], pr = _softmax_block(q[:, h], k[:, g], mask, scale)
        o[:, h] = (pr * _dropout_block(b, h, ar, ar, p, seed, dtype)) @ v[:, g]
    return o, lse


def attention_bwd_dropout(q, k, v, do, cu, p: float, seed: int, b: int = 0, scale=None, dtype=torch.float64):
    """Analytic gradients of sum(O * dO) with dropout for one whole sequence.

    Returns dQ, dK, dV, O, LSE."""
    S, H, d = q.shape
    Hkv = k.shape[1]
    G = _heads(H, Hkv)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = block_causal_mask(cu, S)
    q, k, v, do = (t.to(dtype) for t in (q, k, v, do))
    ar = np.arange(S)
    dq = torch.zeros(S, H, d, dtype=dtype)
    dk = torch.zeros(S, Hkv, d, dtype=dtype)
    dv = torch.zeros(S, Hkv, d, dtype=dtype)
    o = torch.zeros(S, H, d, dtype=dtype)
    lse = torch.empty(H, S, dtype=dtype)
    for h in range(H):
        g = h // G
        lse[h], pr = _softmax_block(q[:, h], k[:, g], mask, scale)
        z = _dropout_block(b, h, ar, ar, p, seed, dtype)
        pd = pr * z
        o[:, h] = pd @ v[:, g]
        dD = (do[:, h] * o[:, h]).sum(-1)
        dp = do[:, h] @ v[:, g].T
        ds = pr * (z * dp - dD[:, None])
        dv[:, g] += pd.T @ do[:, h]
        dq[:, h] = scale * (ds @ k[:, g])
        dk[:, g] += scale * (ds.T @ q[:, h])
    return dq, dk, dv, o, lse


def chunk_fwd_dropout(q_chunk, k_buf, v_buf, cu, S, row_offset, p: float, seed: int, b: int = 0, kv_base=0,
                      scale=None, dtype=torch.float64):
    """One query chunk with dropout (global row indices select the mask). Returns O [L, H, d], LSE [H, L]."""
    L, H, d = q_chunk.shape
    R = k_buf.shape[0]
    G = _heads(H, k_buf.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = _chunk_geometry(cu, S, row_offset, L, kv_base, R)
    q, k, v = (t.to(dtype) for t in (q_chunk, k_buf, v_buf))
    rows, cols = np.arange(row_offset, row_offset + L), np.arange(kv_base, kv_base + R)
    o = torch.zeros(L, H, d, dtype=dtype)
    lse = torch.empty(H, L, dtype=dtype)
    for h in range(H):
        g = h // G
        lse[h], pr = _softmax_block(q[:, h], k[:, g], mask, scale)
        o[:, h] = (pr * _dropout_block(b, h, rows, cols, p, seed, dtype)) @ v[:, g]
    return o, lse


def chunk_bwd_dropout(q_chunk, k_buf, v_buf, do_chunk, cu, S, row_offset, p: float, seed: int, b: int = 0,
                      kv_base=0, scale=None, dtype=torch.float64):
    """Backward of one query chunk with dropout: dQ [L, H, d] and the chunk's dK/dV partials [R, Hkv, d]."""
    L, H, d = q_chunk.shape
    R, Hkv, _ = k_buf.shape
    G = _heads(H, Hkv)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = _chunk_geometry(cu, S, row_offset, L, kv_base, R)
    q, k, v, do = (t.to(dtype) for t in (q_chunk, k_buf, v_buf, do_chunk))
    rows, cols = np.arange(row_offset, row_offset + L), np.arange(kv_base, kv_base + R)
    dq = torch.zeros(L, H, d, dtype=dtype)
    dk = torch.zeros(R, Hkv, d, dtype=dtype)
    dv = torch.zeros(R, Hkv, d, dtype=dtype)
    for h in range(H):
        g = h // G
        _, pr = _softmax_block(q[:, h], k[:, g], mask, scale)
        z = _dropout_block(b, h, rows, cols, p, seed, dtype)
        pd = pr * z
        o = pd @ v[:, g]
        dD = (do[:, h] * o).sum(-1)
        ds = pr * (z * (do[:, h] @ v[:, g].T) - dD[:, None])
        dv[:, g] += pd.T @ do[:, h]
        dq[:, h] = scale * (ds @ k[:, g])
        dk[:, g] += scale * (ds.T @ q[:, h])
    return dq, dk, dv


def _doc_extents(cu):
    return [(int(cu[d]), int(cu[d + 1])) for d in range(len(cu) - 1) if cu[d + 1] > cu[d]]


def attention_rows_dropout(q, k, v, do, cu, rows, p: float, seed: int, b: int = 0, scale=None,
                           dtype=torch.float64):
    """O [R, H, d], LSE [H, R] and dQ [R, H, d] with dropout for selected query
    rows of a whole sequence. Each row needs only its own document's keys up to
    itself, so rows are evaluated document by document."""
    S, H, d = q.shape
    G = _heads(H, k.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    rows = np.asarray(rows, dtype=np.int64)
    o = torch.zeros(len(rows), H, d, dtype=dtype)
    lse = torch.full((H, len(rows)), float("-inf"), dtype=dtype)
    dq = torch.zeros(len(rows), H, d, dtype=dtype)
    for a, e in _doc_extents(cu):
        sel = np.flatnonzero((rows >= a) & (rows < e))
        if len(sel) == 0:
            continue
        rr = rows[sel]
        keys = np.arange(a, int(rr.max()) + 1)
        mask = torch.from_numpy(keys[None, :] <= rr[:, None])
        tr, tk = torch.from_numpy(rr), torch.from_numpy(keys)
        qr, dor = q[tr].to(dtype), do[tr].to(dtype)           # only the slices used
        kk, vk = k[tk].to(dtype), v[tk].to(dtype)
        for h in range(H):
            g = h // G
            l_h, pr = _softmax_block(qr[:, h], kk[:, g], mask, scale)
            z = _dropout_block(b, h, rr, keys, p, seed, dtype)
            oh = (pr * z) @ vk[:, g]
            dD = (dor[:, h] * oh).sum(-1)
            ds = pr * (z * (dor[:, h] @ vk[:, g].T) - dD[:, None])
            o[sel, h] = oh
            lse[h, sel] = l_h
            dq[sel, h] = scale * (ds @ kk[:, g])
    return o, lse, dq


def attention_bwd_cols_dropout(q, k, v, do, cu, cols, p: float, seed: int, b: int = 0, scale=None,
                               dtype=torch.float64):
    """dK, dV [len(cols), Hkv, d] with dropout for selected key columns of a whole
    sequence, document by document: only the query rows of a column's document at
    or after the document's earliest selected column are evaluated."""
    S, H, d = q.shape
    Hkv = k.shape[1]
    G = _heads(H, Hkv)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    cols = np.asarray(cols, dtype=np.int64)
    dk = torch.zeros(len(cols), Hkv, d, dtype=dtype)
    dv = torch.zeros(len(cols), Hkv, d, dtype=dtype)
    for a, e in _doc_extents(cu):
        sel = np.flatnonzero((cols >= a) & (cols < e))
        if len(sel) == 0:
            continue
        rr = np.arange(int(cols[sel].min()), e)
        keys = np.arange(a, e)
        mask = torch.from_numpy(keys[None, :] <= rr[:, None])
        tr, tk = torch.from_numpy(rr), torch.from_numpy(keys)
        cidx = torch.from_numpy(cols[sel] - a)
        qr, dor = q[tr].to(dtype), do[tr].to(dtype)           # only the slices used
        kk, vk = k[tk].to(dtype), v[tk].to(dtype)
        for h in range(H):
            g = h // G
            _, pr = _softmax_block(qr[:, h], kk[:, g], mask, scale)
            z = _dropout_block(b, h, rr, keys, p, seed, dtype)
            oh = (pr * z) @ vk[:, g]
            dD = (dor[:, h] * oh).sum(-1)
            pc, zc = pr[:, cidx], z[:, cidx]
            ds = pc * (zc * (dor[:, h] @ vk[cidx, g].T) - dD[:, None])
            dv[sel, g] += (pc * zc).T @ dor[:, h]
            dk[sel, g] += scale * (ds.T @ qr[:, h])
    return dk, dv
