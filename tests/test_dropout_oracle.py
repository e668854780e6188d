"""Dropout oracle against what pins it: the generator's published known-answer
vectors, the p = 0 special case, the keep rate, autograd through an explicit
masked forward, and chunk/full consistency (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

# Known-answer vectors distributed with the reference implementation of the
# Philox generator (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
# SC 2011): Philox4x32, 10 rounds, (counter words, key words) -> output words.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    got = oracle.philox4x32_10(np.array([ctr], dtype=np.uint64), key)[0]
    assert tuple(int(x) for x in got) == want


def test_philox_vectorised_rows_are_independent_calls():
    ctrs = np.array([c for c, _, _ in PHILOX_KAT[:1]] * 3, dtype=np.uint64)
    got = oracle.philox4x32_10(ctrs, (0, 0))
    assert (got == got[0]).all()


def _inputs(S, H, Hkv, d, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(S, H, d, generator=g, dtype=torch.float64)
    k = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(S, Hkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(S, H, d, generator=g, dtype=torch.float64)
    return q, k, v, do


def _eq_inf(a, b):
    return torch.equal(torch.nan_to_num(a, neginf=-1e300), torch.nan_to_num(b, neginf=-1e300))


def test_zero_probability_is_plain_attention():
    cu, S = [0, 10, 24, 30], 32
    q, k, v, do = _inputs(S, 4, 2, 8)
    o, lse = oracle.attention_fwd_dropout(q, k, v, cu, 0.0, 7)
    o0, lse0 = oracle.attention_fwd(q, k, v, cu)
    assert torch.equal(o, o0) and _eq_inf(lse, lse0)
    g = oracle.attention_bwd_dropout(q, k, v, do, cu, 0.0, 7)
    g0 = oracle.attention_bwd(q, k, v, do, cu)
    for a, b in zip(g[:3], g0[:3]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_rate(p):
    n = 1024
    m = oracle.keep_mask(3, 5, np.arange(n), np.arange(n), 0x123456789, p)
    rate = m.double().mean().item()
    sigma = (p * (1 - p) / n ** 2) ** 0.5
    assert abs(rate - (1 - p)) < 6 * sigma


def test_threshold_edges():
    assert oracle.keep_threshold(0.0) == 0
    assert oracle.keep_threshold(0.5) == 2 ** 31
    assert oracle.keep_threshold(1 - 2 ** -40) == 2 ** 32 - 1
    with pytest.raises(ValueError):
        oracle.keep_threshold(1.0)


def test_mask_depends_on_every_counter_and_key_word():
    base = oracle.keep_mask(0, 0, np.arange(64), np.arange(64), 11, 0.5)
    for kw in ({"b": 1}, {"h": 1}, {"seed": 12}, {"seed": 11 + (1 << 32)}):
        args = dict(b=0, h=0, seed=11)
        args.update(kw)
        other = oracle.keep_mask(args["b"], args["h"], np.arange(64), np.arange(64), args["seed"], 0.5)
        assert not torch.equal(base, other), kw
    # neighbouring rows and key blocks draw different words
    assert not torch.equal(base[0], base[1]) and not torch.equal(base[0], base[2])
    assert not torch.equal(base[:, :2], base[:, 2:4])


def test_mask_layout_is_the_documented_counter_and_word():
    """keep[i, j] uses word 2 (i mod 2) + (j mod 2) of the call at counter (j // 2, i // 2, h, b)."""
    seed, p, b, h = 0xABCDEF0123, 0.5, 3, 7
    rows, cols = np.array([0, 1, 5, 6, 1000]), np.array([0, 1, 2, 9, 4097])
    m = oracle.keep_mask(b, h, rows, cols, seed, p)
    t = oracle.keep_threshold(p)
    for a, i in enumerate(rows):
        for c, j in enumerate(cols):
            w = oracle.philox4x32_10(np.array([[j // 2, i // 2, h, b]], dtype=np.uint64),
                                     (seed & 0xFFFFFFFF, seed >> 32))[0]
            assert bool(m[a, c]) == (int(w[2 * (i % 2) + j % 2]) >= t)


def _autograd_reference(cu, S, H, Hkv, p, seed, b, d=8):
    q, k, v, do = _inputs(S, H, Hkv, d, seed=1)
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    mask = oracle.block_causal_mask(cu, S)
    G = H // Hkv
    outs = []
    for h in range(H):
        s = (q[:, h] @ k[:, h // G].T) / d ** 0.5
        s = s.masked_fill(~mask, float("-inf"))
        pr = torch.softmax(s, dim=-1).nan_to_num(0.0)
        z = oracle.keep_mask(b, h, np.arange(S), np.arange(S), seed, p).double() / (1 - p)
        outs.append((pr * z) @ v[:, h // G])
    o_ref = torch.stack(outs, dim=1)
    (o_ref * do).sum().backward()
    return (q.detach(), k.detach(), v.detach(), do), o_ref.detach(), (q.grad, k.grad, v.grad)


def _max_grad_err(cu, S, H, Hkv, p, seed, b):
    (q, k, v, do), o_ref, ref = _autograd_reference(cu, S, H, Hkv, p, seed, b)
    dq, dk, dv, o, _ = oracle.attention_bwd_dropout(q, k, v, do, cu, p, seed, b=b)
    return max((o - o_ref).abs().max().item(), *[(g - w).abs().max().item() for g, w in zip((dq, dk, dv), ref)])


@pytest.mark.parametrize("cu,S,H,Hkv,p", [
    ([0, 10, 24, 30], 32, 4, 2, 0.3),
    ([0, 3, 29], 32, 2, 2, 0.6),
    ([0, 17], 20, 4, 1, 0.1),
])
def test_backward_matches_autograd(cu, S, H, Hkv, p):
    """The analytic backward against autograd through an explicit forward that
    applies the same (constant) keep mask to the softmax probabilities."""
    assert _max_grad_err(cu, S, H, Hkv, p, seed=99, b=2) < 1e-10


def test_planted_mistake_in_the_oracle_is_caught(monkeypatch):
    """An oracle that forgets the 1/(1-p) rescale fails the autograd pin."""
    import oracle.dropout as od
    monkeypatch.setattr(od, "_dropout_block",
                        lambda b, h, rows, cols, p, seed, dtype: od.keep_mask(b, h, rows, cols, seed, p).to(dtype))
    assert _max_grad_err([0, 12, 20], 20, 2, 1, 0.5, seed=3, b=0) > 1e-3


@pytest.mark.parametrize("world,cu,S", [(2, [0, 10, 24, 30], 32), (4, [0, 3, 29], 32)])
def test_chunks_with_global_indices_equal_full(world, cu, S):
    H, Hkv, d, p, seed, b = 4, 2, 8, 0.4, 5, 1
    q, k, v, do = _inputs(S, H, Hkv, d, seed=3)
    o_full, lse_full = oracle.attention_fwd_dropout(q, k, v, cu, p, seed, b=b)
    dq_full, dk_full, dv_full, _, _ = oracle.attention_bwd_dropout(q, k, v, do, cu, p, seed, b=b)
    L = S // world
    dk_sum = torch.zeros_like(dk_full)
    dv_sum = torch.zeros_like(dv_full)
    for r in range(world):
        a = oracle.segment_chunk(cu, S, world, r)["hdr"]["kv_start"]
        rows = slice(r * L, (r + 1) * L)
        o, lse = oracle.chunk_fwd_dropout(q[rows], k[a:], v[a:], cu, S, r * L, p, seed, b=b, kv_base=a)
        assert (o - o_full[rows]).abs().max() < 1e-12
        assert _eq_inf(lse, lse_full[:, rows]) or (lse - lse_full[:, rows]).nan_to_num(0).abs().max() < 1e-12
        dq, dkw, dvw = oracle.chunk_bwd_dropout(q[rows], k[a:], v[a:], do[rows], cu, S, r * L, p, seed, b=b,
                                                kv_base=a)
        assert (dq - dq_full[rows]).abs().max() < 1e-12
        dk_sum[a:] += dkw
        dv_sum[a:] += dvw
    assert (dk_sum - dk_full).abs().max() < 1e-12 and (dv_sum - dv_full).abs().max() < 1e-12


def test_workload_shapes_run():
    wl = workloads.config(1)
    q, k, v, do = workloads.tensors(wl)
    o, lse = oracle.chunk_fwd_dropout(q[0, :wl.L], k[0], v[0], wl.cu[0], wl.S, 0, 0.1, 42)
    assert torch.isfinite(o).all()


def test_sampled_rows_and_columns_equal_the_full_oracle():
    cu, S, H, Hkv, p, seed, b = [0, 10, 24, 30], 32, 4, 2, 0.35, 77, 1
    q, k, v, do = _inputs(S, H, Hkv, 8, seed=4)
    dq, dk, dv, o, lse = oracle.attention_bwd_dropout(q, k, v, do, cu, p, seed, b=b)
    rows = [0, 5, 9, 10, 23, 29, 30, 31]
    o_r, lse_r, dq_r = oracle.attention_rows_dropout(q, k, v, do, cu, rows, p, seed, b=b)
    assert (o_r - o[rows]).abs().max() < 1e-12 and (dq_r - dq[rows]).abs().max() < 1e-12
    ref = lse[:, rows]
    assert torch.equal(torch.isneginf(lse_r), torch.isneginf(ref))
    fin = torch.isfinite(ref)
    assert (lse_r[fin] - ref[fin]).abs().max() < 1e-12
    cols = [0, 3, 9, 12, 23, 24, 29, 31]
    dk_c, dv_c = oracle.attention_bwd_cols_dropout(q, k, v, do, cu, cols, p, seed, b=b)
    assert (dk_c - dk[cols]).abs().max() < 1e-12 and (dv_c - dv[cols]).abs().max() < 1e-12
