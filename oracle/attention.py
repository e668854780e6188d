"""Oracle dense masked attention: forward (O, LSE) and analytic backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the NeMo Automodel page "block-diagonal varlen CP for packed
sequences": the dense masked attention that the page calls numerically
identical to its varlen kernel (Summary; Design overview, kernels.py "dense
[B,1,L,S] mask builder"), over the per-document block-causal mask (Key
correctness property 1), evaluated one contiguous query chunk at a time with
K/V taken either from the whole sequence (fused all-gather) or from the
needed-only window that starts at the first document the chunk overlaps
(Summary; Design overview, exchange.py). The backward's dK/dV partials of a
chunk add up over chunks at the owning rows, which is what the reduce-scatter
SUM does (Design overview, exchange.py).

The page gives no formulas; the plain reading used here is standard softmax
attention with scale 1/sqrt(d):

    s_ij  = scale * <q_i, k_j>                     (unmasked pairs only)
    LSE_i = ln sum_j exp(s_ij)                      (natural log, scale inside)
    P_ij  = exp(s_ij - LSE_i),   O_i = sum_j P_ij v_j
    D_i   = <dO_i, O_i>,         dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - D_i)
    dV_j  = sum_i P_ij dO_i,     dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i

GQA: query head h reads key/value head h // (H // Hkv); dK/dV sum over the
query heads of a group. Padding rows: O = 0, LSE = -inf, zero gradients.

Tensors are per sequence: q, dO [S, H, d]; k, v [S, Hkv, d]. Everything is
computed in ``dtype`` (float64 by default) from the given values.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .segment import doc_ids

NEG_INF = float("-inf")


def block_causal_mask(cu, S: int, rows=None, cols=None) -> torch.Tensor:
    """Dense boolean mask M[i, j] = i valid and doc(i) == doc(j) and j <= i.

    ``rows`` / ``cols`` select global row / column indices (default: all).
    """
    ids = torch.from_numpy(doc_ids(cu, S))
    r = torch.arange(S) if rows is None else torch.as_tensor(rows, dtype=torch.long)
    c = torch.arange(S) if cols is None else torch.as_tensor(cols, dtype=torch.long)
    di = ids[r][:, None]
    dj = ids[c][None, :]
    return (di >= 0) & (di == dj) & (c[None, :] <= r[:, None])


def _heads(H, Hkv):
    if H % Hkv != 0:
        raise ValueError("H must be a multiple of Hkv")
    return H // Hkv


def _softmax_block(q, k, mask, scale):
    """Scores, LSE and probabilities for one head: q [R, d], k [C, d], mask [R, C]."""
    s = (q @ k.T) * scale
    s = s.masked_fill(~mask, NEG_INF)
    lse = torch.logsumexp(s, dim=-1)                       # -inf on rows with no key
    p = torch.where(mask, torch.exp(s - lse[:, None]), torch.zeros((), dtype=s.dtype))
    return lse, p


def attention_fwd(q, k, v, cu, scale=None, rows=None, dtype=torch.float64):
    """Full block-causal attention for one sequence (optionally only ``rows``).

    Returns O [R, H, d] and LSE [H, R] in ``dtype``.
    """
    S, H, d = q.shape
    G = _heads(H, k.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    r = torch.arange(S) if rows is None else torch.as_tensor(rows, dtype=torch.long)
    mask = block_causal_mask(cu, S, rows=r)
    q = q.to(dtype)[r]
    k = k.to(dtype)
    v = v.to(dtype)
    o = torch.zeros(len(r), H, d, dtype=dtype)
    lse = torch.empty(H, len(r), dtype=dtype)
    for h in range(H):
        g = h // G
        lse[h], p = _softmax_block(q[:, h], k[:, g], mask, scale)
        o[:, h] = p @ v[:, g]
    return o, lse


def attention_bwd(q, k, v, do, cu, scale=None, dtype=torch.float64):
    """Analytic gradients of sum(O * dO) for one whole sequence.

    Returns dQ [S, H, d], dK [S, Hkv, d], dV [S, Hkv, d], O, LSE.
    """
    S, H, d = q.shape
    Hkv = k.shape[1]
    G = _heads(H, Hkv)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = block_causal_mask(cu, S)
    q, k, v, do = (t.to(dtype) for t in (q, k, v, do))
    dq = torch.zeros(S, H, d, dtype=dtype)
    dk = torch.zeros(S, Hkv, d, dtype=dtype)
    dv = torch.zeros(S, Hkv, d, dtype=dtype)
    o = torch.zeros(S, H, d, dtype=dtype)
    lse = torch.empty(H, S, dtype=dtype)
    for h in range(H):
        g = h // G
        lse[h], p = _softmax_block(q[:, h], k[:, g], mask, scale)
        o[:, h] = p @ v[:, g]
        dD = (do[:, h] * o[:, h]).sum(-1)
        dp = do[:, h] @ v[:, g].T
        ds = p * (dp - dD[:, None])
        dv[:, g] += p.T @ do[:, h]
        dq[:, h] = scale * (ds @ k[:, g])
        dk[:, g] += scale * (ds.T @ q[:, h])
    return dq, dk, dv, o, lse


def _chunk_geometry(cu, S, row_offset, L, kv_base, R):
    rows = torch.arange(row_offset, row_offset + L)
    cols = torch.arange(kv_base, kv_base + R)
    mask = block_causal_mask(cu, S, rows=rows, cols=cols.clamp(max=S - 1))
    mask &= (cols < S)[None, :]
    return mask


def chunk_fwd(q_chunk, k_buf, v_buf, cu, S, row_offset, kv_base=0, scale=None,
              dtype=torch.float64):
    """One query chunk: rows [row_offset, row_offset + L) of the sequence.

    ``k_buf``/``v_buf`` [R, Hkv, d] hold global rows [kv_base, kv_base + R):
    the whole sequence (all-gather, kv_base = 0) or the needed-only window.
    Returns O [L, H, d], LSE [H, L].
    """
    L, H, d = q_chunk.shape
    G = _heads(H, k_buf.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = _chunk_geometry(cu, S, row_offset, L, kv_base, k_buf.shape[0])
    q, k, v = (t.to(dtype) for t in (q_chunk, k_buf, v_buf))
    o = torch.zeros(L, H, d, dtype=dtype)
    lse = torch.empty(H, L, dtype=dtype)
    for h in range(H):
        g = h // G
        lse[h], p = _softmax_block(q[:, h], k[:, g], mask, scale)
        o[:, h] = p @ v[:, g]
    return o, lse


def chunk_bwd(q_chunk, k_buf, v_buf, do_chunk, cu, S, row_offset, kv_base=0, scale=None,
              dtype=torch.float64):
    """Backward of one query chunk.

    Returns dQ [L, H, d] for the chunk's rows and the chunk's dK/dV partials
    [R, Hkv, d] over the K/V buffer rows: the contributions of this chunk's
    query rows only. Summed over all chunks at the owning rows they give the
    full dK/dV.
    """
    L, H, d = q_chunk.shape
    R, Hkv, _ = k_buf.shape
    G = _heads(H, Hkv)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask = _chunk_geometry(cu, S, row_offset, L, kv_base, R)
    q, k, v, do = (t.to(dtype) for t in (q_chunk, k_buf, v_buf, do_chunk))
    dq = torch.zeros(L, H, d, dtype=dtype)
    dk = torch.zeros(R, Hkv, d, dtype=dtype)
    dv = torch.zeros(R, Hkv, d, dtype=dtype)
    for h in range(H):
        g = h // G
        _, p = _softmax_block(q[:, h], k[:, g], mask, scale)
        o = p @ v[:, g]
        dD = (do[:, h] * o).sum(-1)
        ds = p * (do[:, h] @ v[:, g].T - dD[:, None])
        dv[:, g] += p.T @ do[:, h]
        dq[:, h] = scale * (ds @ k[:, g])
        dk[:, g] += scale * (ds.T @ q[:, h])
    return dq, dk, dv


def attention_bwd_rows(q, k, v, do, cu, rows, scale=None, dtype=torch.float64):
    """dQ [len(rows), H, d] for selected query rows of a whole sequence.

    Each row needs only its own scores, so any row is cheap at any length.
    """
    S, H, d = q.shape
    G = _heads(H, k.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    rows = torch.as_tensor(rows, dtype=torch.long)
    mask = block_causal_mask(cu, S, rows=rows)
    q, k, v, do = (t.to(dtype) for t in (q, k, v, do))
    dq = torch.zeros(len(rows), H, d, dtype=dtype)
    for h in range(H):
        g = h // G
        _, p = _softmax_block(q[rows, h], k[:, g], mask, scale)
        o = p @ v[:, g]
        dD = (do[rows, h] * o).sum(-1)
        ds = p * (do[rows, h] @ v[:, g].T - dD[:, None])
        dq[:, h] = scale * (ds @ k[:, g])
    return dq


def attention_bwd_cols(q, k, v, do, cu, cols, scale=None, dtype=torch.float64):
    """dK, dV [len(cols), Hkv, d] for selected key columns of a whole sequence.

    Only the query rows that attend to some selected column are evaluated, so
    columns near the end of their documents are cheap at any sequence length.
    """
    S, H, d = q.shape
    Hkv = k.shape[1]
    G = _heads(H, Hkv)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    cols = torch.as_tensor(cols, dtype=torch.long)
    ids = doc_ids(cu, S)
    need = np.zeros(S, dtype=bool)
    for j in cols.tolist():
        if ids[j] >= 0:
            need |= (ids == ids[j]) & (np.arange(S) >= j)
    rows = torch.from_numpy(np.flatnonzero(need))
    dk = torch.zeros(len(cols), Hkv, d, dtype=dtype)
    dv = torch.zeros(len(cols), Hkv, d, dtype=dtype)
    if len(rows) == 0:
        return dk, dv
    mask_full = block_causal_mask(cu, S, rows=rows)            # [R, S]
    q, k, v, do = (t.to(dtype) for t in (q, k, v, do))
    for h in range(H):
        g = h // G
        _, p = _softmax_block(q[rows, h], k[:, g], mask_full, scale)
        o = p @ v[:, g]
        dD = (do[rows, h] * o).sum(-1)
        pc = p[:, cols]
        ds = pc * (do[rows, h] @ v[cols, g].T - dD[:, None])
        dv[:, g] += pc.T @ do[rows, h]
        dk[:, g] += scale * (ds.T @ q[rows, h])
    return dk, dv
