"""Pins for the oracle: it is checked against things other than itself.

* brute force: per-pair Python loops over document ids (fp64, tiny sizes);
* a library special case: per document, torch's causal
  scaled_dot_product_attention (and its autograd) on that document's slice;
* central finite differences of sum(O * dO);
* invariants: chunks concatenated equal the whole sequence, chunk dK/dV
  partials sum to the full dK/dV, needed-only window equals full K/V,
  padding rows give zeros, a single document is plain causal attention;
* planted mistakes: each plausible slip in the oracle fails one of the pins.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attention as oatt
from oracle import segment as oseg

torch.set_default_dtype(torch.float32)

LAYOUTS = [
    # (cu_seqlens, S, cp) -- hand-built 2- and 3-document layouts, length-1
    # documents, a boundary on a chunk edge, a document spanning every chunk,
    # an all-padding chunk, zero-length documents.
    ([0, 10, 24], 24, 2),
    ([0, 5, 9, 20], 24, 3),
    ([0, 1, 2, 16], 16, 4),
    ([0, 8, 16], 16, 2),          # boundary exactly on the chunk edge
    ([0, 30], 32, 4),             # one document over every chunk + padding tail
    ([0, 7, 12], 32, 2),          # chunk 1 is all padding
    ([0, 0, 6, 6, 14], 16, 2),    # zero-length documents
    ([0], 8, 2),                  # no documents at all
]


def _rand(S, H, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(S, H, d, generator=g, dtype=torch.float64)
    k = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(S, H, d, generator=g, dtype=torch.float64)
    return q, k, v, do


def _brute(q, k, v, cu, S):
    """Per-pair loops straight from the definition (fp64, math module)."""
    _, H, d = q.shape
    G = H // k.shape[1]
    ids = [-1] * S
    for doc in range(len(cu) - 1):
        for t in range(cu[doc], cu[doc + 1]):
            ids[t] = doc
    scale = 1.0 / math.sqrt(d)
    o = [[[0.0] * d for _ in range(H)] for _ in range(S)]
    lse = [[-math.inf] * S for _ in range(H)]
    for h in range(H):
        g = h // G
        for i in range(S):
            keys = [j for j in range(S) if ids[i] >= 0 and ids[j] == ids[i] and j <= i]
            if not keys:
                continue
            s = [scale * sum(float(q[i, h, c]) * float(k[j, g, c]) for c in range(d)) for j in keys]
            m = max(s)
            z = sum(math.exp(x - m) for x in s)
            lse[h][i] = m + math.log(z)
            for jj, j in enumerate(keys):
                p = math.exp(s[jj] - lse[h][i])
                for c in range(d):
                    o[i][h][c] += p * float(v[j, g, c])
    return torch.tensor(o, dtype=torch.float64), torch.tensor(lse, dtype=torch.float64)


def _sdpa_per_doc(q, k, v, cu, S, requires_grad=False):
    """Whole-sequence attention built from torch's causal SDPA, one document at a time."""
    _, H, d = q.shape
    G = H // k.shape[1]
    outs = []
    for doc in range(len(cu) - 1):
        a, b = cu[doc], cu[doc + 1]
        if b == a:
            continue
        qd = q[a:b].transpose(0, 1)                                   # [H, l, d]
        kd = k[a:b].repeat_interleave(G, dim=1).transpose(0, 1)
        vd = v[a:b].repeat_interleave(G, dim=1).transpose(0, 1)
        outs.append(F.scaled_dot_product_attention(qd, kd, vd, is_causal=True).transpose(0, 1))
    pad = S - cu[-1]
    if pad:
        outs.append(torch.zeros(pad, H, d, dtype=q.dtype))
    return torch.cat(outs, 0)


def _lse_per_doc(q, k, cu, S):
    _, H, d = q.shape
    G = H // k.shape[1]
    lse = torch.full((H, S), -math.inf, dtype=torch.float64)
    for doc in range(len(cu) - 1):
        a, b = cu[doc], cu[doc + 1]
        if b == a:
            continue
        for h in range(H):
            s = (q[a:b, h] @ k[a:b, h // G].T) / math.sqrt(d)
            s = s.masked_fill(~torch.ones(b - a, b - a, dtype=torch.bool).tril(), -math.inf)
            lse[h, a:b] = torch.logsumexp(s, -1)
    return lse


@pytest.mark.parametrize("cu,S,cp", LAYOUTS)
def test_fwd_matches_brute_force(cu, S, cp):
    q, k, v, _ = _rand(S, 2, 1, 4, seed=S + len(cu))
    o, lse = oracle.attention_fwd(q, k, v, cu)
    ob, lb = _brute(q, k, v, cu, S)
    assert torch.allclose(o, ob, atol=1e-12, rtol=0)
    assert torch.equal(torch.isinf(lse), torch.isinf(lb))
    fin = torch.isfinite(lb)
    assert torch.allclose(lse[fin], lb[fin], atol=1e-12, rtol=0)


@pytest.mark.parametrize("cu,S,cp", LAYOUTS)
@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 1)])
def test_fwd_matches_sdpa_per_document(cu, S, cp, H, Hkv):
    q, k, v, _ = _rand(S, H, Hkv, 8, seed=7 * S + H)
    o, lse = oracle.attention_fwd(q, k, v, cu)
    assert torch.allclose(o, _sdpa_per_doc(q, k, v, cu, S), atol=1e-12, rtol=0)
    ref = _lse_per_doc(q, k, cu, S)
    assert torch.equal(torch.isinf(lse), torch.isinf(ref))
    fin = torch.isfinite(ref)
    assert torch.allclose(lse[fin], ref[fin], atol=1e-12, rtol=0)


@pytest.mark.parametrize("cu,S,cp", LAYOUTS)
def test_bwd_matches_autograd_through_sdpa(cu, S, cp):
    q, k, v, do = _rand(S, 4, 2, 8, seed=11 * S)
    dq, dk, dv, o, _ = oracle.attention_bwd(q, k, v, do, cu)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    oa = _sdpa_per_doc(qa, ka, va, cu, S)
    loss = (oa * do).sum() + 0.0 * (qa.sum() + ka.sum() + va.sum())   # all-padding layout has no graph
    loss.backward()
    gq = qa.grad if qa.grad is not None else torch.zeros_like(q)
    gk = ka.grad if ka.grad is not None else torch.zeros_like(k)
    gv = va.grad if va.grad is not None else torch.zeros_like(v)
    assert torch.allclose(o, oa.detach(), atol=1e-12, rtol=0)
    assert torch.allclose(dq, gq, atol=1e-11, rtol=0)
    assert torch.allclose(dk, gk, atol=1e-11, rtol=0)
    assert torch.allclose(dv, gv, atol=1e-11, rtol=0)


def test_bwd_matches_finite_differences():
    cu, S = [0, 7, 15, 22], 24
    q, k, v, do = _rand(S, 2, 1, 4, seed=3)
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, do, cu)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd(q_, k_, v_, cu)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = torch.zeros_like(x)
        flat = x.view(-1)
        for idx in range(flat.numel()):
            old = float(flat[idx])
            flat[idx] = old + eps
            lp = loss(q, k, v)
            flat[idx] = old - eps
            lm = loss(q, k, v)
            flat[idx] = old
            num.view(-1)[idx] = (lp - lm) / (2 * eps)
        err = (num - g).norm() / g.norm()
        assert err < 1e-6, (name, float(err))


@pytest.mark.parametrize("cu,S,cp", LAYOUTS)
def test_chunks_concatenate_to_full_and_partials_sum(cu, S, cp):
    q, k, v, do = _rand(S, 4, 2, 8, seed=5 * S)
    o, lse = oracle.attention_fwd(q, k, v, cu)
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, do, cu)
    L = S // cp
    sk = torch.zeros_like(dk)
    sv = torch.zeros_like(dv)
    for r in range(cp):
        rows = slice(r * L, (r + 1) * L)
        oc, lc = oracle.chunk_fwd(q[rows], k, v, cu, S, r * L)
        assert torch.allclose(oc, o[rows], atol=1e-12, rtol=0)
        assert torch.equal(torch.isinf(lc), torch.isinf(lse[:, rows]))
        fin = torch.isfinite(lc)
        assert torch.allclose(lc[fin], lse[:, rows][fin], atol=1e-12, rtol=0)
        dqc, dkc, dvc = oracle.chunk_bwd(q[rows], k, v, do[rows], cu, S, r * L)
        assert torch.allclose(dqc, dq[rows], atol=1e-12, rtol=0)
        sk += dkc
        sv += dvc
    assert torch.allclose(sk, dk, atol=1e-12, rtol=0)
    assert torch.allclose(sv, dv, atol=1e-12, rtol=0)


@pytest.mark.parametrize("cu,S,cp", LAYOUTS)
def test_window_equals_gather(cu, S, cp):
    """The needed-only window [kv_start, kv_end) gives identical results to full K/V."""
    q, k, v, do = _rand(S, 4, 2, 8, seed=9 * S)
    L = S // cp
    for r in range(cp):
        seg = oracle.segment_chunk(cu, S, cp, r)["hdr"]
        a, b = seg["kv_start"], seg["kv_end"]
        rows = slice(r * L, (r + 1) * L)
        og, lg = oracle.chunk_fwd(q[rows], k, v, cu, S, r * L)
        ow, lw = oracle.chunk_fwd(q[rows], k[a:b], v[a:b], cu, S, r * L, kv_base=a)
        # same values up to the summation order of the longer masked rows
        assert torch.allclose(og, ow, atol=1e-13, rtol=0)
        assert torch.equal(torch.isinf(lg), torch.isinf(lw))
        assert torch.allclose(lg[torch.isfinite(lg)], lw[torch.isfinite(lw)], atol=1e-13, rtol=0)
        dqg, dkg, dvg = oracle.chunk_bwd(q[rows], k, v, do[rows], cu, S, r * L)
        dqw, dkw, dvw = oracle.chunk_bwd(q[rows], k[a:b], v[a:b], do[rows], cu, S, r * L, kv_base=a)
        assert torch.allclose(dqg, dqw, atol=1e-13, rtol=0)
        assert torch.allclose(dkg[a:b], dkw, atol=1e-13, rtol=0)
        assert torch.allclose(dvg[a:b], dvw, atol=1e-13, rtol=0)
        assert not dkg[:a].any() and not dkg[b:].any()


def test_padding_rows_are_zero_and_ignored():
    cu, S = [0, 9, 20], 28
    q, k, v, do = _rand(S, 4, 2, 8, seed=1)
    k2, v2 = k.clone(), v.clone()
    k2[20:] = 1e3
    v2[20:] = -1e3
    do2 = do.clone()
    do2[20:] = 77.0
    o, lse = oracle.attention_fwd(q, k2, v2, cu)
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k2, v2, do2, cu)
    assert not o[20:].any() and torch.isneginf(lse[:, 20:]).all()
    assert not dq[20:].any() and not dk[20:].any() and not dv[20:].any()
    o_ref, _ = oracle.attention_fwd(q, k, v, cu)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_bwd(q, k, v, do, cu)
    assert torch.equal(o[:20], o_ref[:20])
    assert torch.allclose(dq, dq_ref, atol=0, rtol=0)
    assert torch.equal(dk[:20], dk_ref[:20]) and torch.equal(dv[:20], dv_ref[:20])


def test_single_document_is_plain_causal():
    S, H, Hkv, d = 96, 4, 1, 16
    q, k, v, do = _rand(S, H, Hkv, d, seed=2)
    o, lse = oracle.attention_fwd(q, k, v, [0, S])
    ref = F.scaled_dot_product_attention(q.transpose(0, 1), k.repeat_interleave(4, 1).transpose(0, 1),
                                         v.repeat_interleave(4, 1).transpose(0, 1), is_causal=True)
    assert torch.allclose(o, ref.transpose(0, 1), atol=1e-12, rtol=0)
    # LSE of row 0 is just its own scaled self-score
    assert torch.allclose(lse[:, 0], (q[0] * k[0, 0]).sum(-1) / math.sqrt(d), atol=1e-12)


def test_sampled_rows_and_cols_match_full():
    cu, S = [0, 13, 40, 41, 60], 64
    q, k, v, do = _rand(S, 4, 2, 8, seed=4)
    dq, dk, dv, o, lse = oracle.attention_bwd(q, k, v, do, cu)
    rows = [0, 12, 13, 39, 40, 59, 60, 63]
    orow, lrow = oracle.attention_fwd(q, k, v, cu, rows=rows)
    assert torch.allclose(orow, o[rows], atol=1e-12)
    assert torch.equal(torch.isinf(lrow), torch.isinf(lse[:, rows]))
    assert torch.allclose(oracle.attention_bwd_rows(q, k, v, do, cu, rows), dq[rows], atol=1e-12)
    cols = [0, 5, 12, 13, 40, 58, 59, 62]
    dkc, dvc = oracle.attention_bwd_cols(q, k, v, do, cu, cols)
    assert torch.allclose(dkc, dk[cols], atol=1e-12)
    assert torch.allclose(dvc, dv[cols], atol=1e-12)


def test_gradient_sum_identities():
    """Per document: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 (rows of P sum to 1,
    rows of dS sum to 0); these hold at any size and are used on the GPU too."""
    cu, S = [0, 17, 30, 48], 50
    q, k, v, do = _rand(S, 4, 2, 8, seed=8)
    _, dk, dv, _, _ = oracle.attention_bwd(q, k, v, do, cu)
    for doc in range(3):
        a, b = cu[doc], cu[doc + 1]
        for g in range(2):
            assert torch.allclose(dv[a:b, g].sum(0), do[a:b, 2 * g:2 * g + 2].sum((0, 1)), atol=1e-11)
            assert torch.allclose(dk[a:b, g].sum(0), torch.zeros(8, dtype=torch.float64), atol=1e-11)


# ---- planted mistakes: each slip in the oracle must fail a pin ------------------

def _mask_strict(cu, S, rows=None, cols=None):          # j < i instead of j <= i
    m = _orig_mask(cu, S, rows, cols)
    r = torch.arange(S) if rows is None else torch.as_tensor(rows)
    c = torch.arange(S) if cols is None else torch.as_tensor(cols)
    return m & (c[None, :] != r[:, None])


def _mask_no_docs(cu, S, rows=None, cols=None):         # forgets the document boundary
    ids = torch.from_numpy(oseg.doc_ids(cu, S))
    r = torch.arange(S) if rows is None else torch.as_tensor(rows)
    c = torch.arange(S) if cols is None else torch.as_tensor(cols)
    return (ids[r][:, None] >= 0) & (ids[c][None, :] >= 0) & (c[None, :] <= r[:, None])


_orig_mask = oatt.block_causal_mask


def _softmax_no_scale(q, k, mask, scale):
    return _orig_softmax(q, k, mask, 1.0)


_orig_softmax = oatt._softmax_block


@pytest.mark.parametrize("name,patch", [("mask", _mask_strict), ("mask", _mask_no_docs),
                                        ("_softmax_block", _softmax_no_scale)])
def test_planted_forward_mistakes_are_caught(monkeypatch, name, patch):
    monkeypatch.setattr(oatt, "block_causal_mask" if name == "mask" else name, patch)
    cu, S = [0, 10, 24], 24
    q, k, v, _ = _rand(S, 2, 1, 4, seed=S + len(cu))
    o, _ = oracle.attention_fwd(q, k, v, cu)
    ob, _ = _brute(q, k, v, cu, S)
    assert not torch.allclose(o, ob, atol=1e-6)


def test_planted_backward_mistake_is_caught(monkeypatch):
    """Dropping the -D_i term of dS must break agreement with autograd."""
    cu, S = [0, 10, 24], 24
    q, k, v, do = _rand(S, 4, 2, 8, seed=11 * S)
    src = oatt.attention_bwd

    def bad_bwd(q, k, v, do, cu, scale=None, dtype=torch.float64):
        zero_do = torch.zeros_like(do)
        dq, dk, dv, o, lse = src(q, k, v, do, cu, scale, dtype)
        # recompute dQ without the D term: dS = P * dP
        S_, H, d = q.shape
        G = H // k.shape[1]
        mask = oatt.block_causal_mask(cu, S_)
        for h in range(H):
            _, p = oatt._softmax_block(q[:, h], k[:, h // G], mask, 1 / math.sqrt(d))
            dq[:, h] = (p * (do[:, h] @ v[:, h // G].T)) @ k[:, h // G] / math.sqrt(d)
        del zero_do
        return dq, dk, dv, o, lse

    dq, _, _, _, _ = bad_bwd(q, k, v, do, cu)
    qa = q.clone().requires_grad_(True)
    (_sdpa_per_doc(qa, k, v, cu, S) * do).sum().backward()
    assert not torch.allclose(dq, qa.grad, atol=1e-6)


def test_planted_head_mapping_mistake_is_caught(monkeypatch):
    """Interleaved GQA mapping (h % Hkv) instead of grouped (h // G) must fail the SDPA pin."""
    cu, S = [0, 10, 24], 24
    q, k, v, _ = _rand(S, 4, 2, 8, seed=21)
    o, _ = oracle.attention_fwd(q, k[:, [0, 1]], v[:, [0, 1]], cu)
    o_bad = torch.zeros_like(o)
    mask = oracle.block_causal_mask(cu, S)
    for h in range(4):
        _, p = oatt._softmax_block(q[:, h], k[:, h % 2], mask, 1 / math.sqrt(8))
        o_bad[:, h] = p @ v[:, h % 2]
    ref = _sdpa_per_doc(q, k, v, cu, S)
    assert torch.allclose(o, ref, atol=1e-12)
    assert not torch.allclose(o_bad, ref, atol=1e-6)
