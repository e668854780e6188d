"""Oracle varlen segmentation of one context-parallel chunk.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the NeMo Automodel page "block-diagonal varlen CP for packed
sequences": batch.py pads to a multiple of cp and gives rank r the contiguous
rows [r*L, (r+1)*L) (Design overview); kernels.py turns the packed layout into
per-rank varlen segments (Design overview); a document that straddles the
chunk's left edge yields an asymmetric first segment whose keys reach back to
the document start, aligned bottom-right (Key correctness property 2); the
needed-only halo exchange delivers K/V from the start of the first document the
chunk overlaps (Summary).

This version deliberately works from the per-token document-id array (runs of
equal ids), not from cu_seqlens arithmetic, so that it is an independent check
of the library's segmentation.

Readings where the page is silent:
* rows at or past S_valid = cu[-1] are padding and belong to no segment;
* an all-padding chunk has no segment and kv_start = kv_end = min(row_offset, S_valid);
* zero-length documents (repeated cu entries) produce no segment;
* kv_end = min(row_offset + L, S_valid).
"""
from __future__ import annotations

import numpy as np


def doc_ids(cu, S: int) -> np.ndarray:
    """Per-token document index; -1 on padding rows (>= cu[-1])."""
    ids = np.full(S, -1, dtype=np.int64)
    for doc in range(len(cu) - 1):
        for t in range(cu[doc], cu[doc + 1]):
            ids[t] = doc
    return ids


def segment_chunk(cu, S: int, cp: int, rank: int) -> dict:
    """Header and segment list for chunk ``rank`` of ``cp``.

    Each segment is (doc, q_start, q_len, k_start, k_len, diag_off) in global
    rows, where the keys of the segment are [k_start, q_start + q_len) and
    local query row i may see local key j iff j <= i + diag_off.
    """
    if S % cp != 0:
        raise ValueError("S must be a multiple of cp")
    if not (0 <= rank < cp):
        raise ValueError("rank out of range")
    ids = doc_ids(cu, S)
    L = S // cp
    row0 = rank * L
    s_valid = int(np.count_nonzero(ids >= 0))
    segs = []
    t = row0
    while t < row0 + L:
        doc = int(ids[t])
        if doc < 0:
            t += 1
            continue
        run_end = t
        while run_end < row0 + L and ids[run_end] == doc:
            run_end += 1
        k_start = int(np.flatnonzero(ids == doc)[0])      # first token of this doc anywhere
        q_len = run_end - t
        k_len = run_end - k_start
        segs.append((doc, t, q_len, k_start, k_len, k_len - q_len))
        t = run_end
    n_pad = int(np.count_nonzero(ids[row0:row0 + L] < 0))
    if segs:
        kv_start = segs[0][3]
        kv_end = segs[-1][1] + segs[-1][2]
    else:
        kv_start = kv_end = min(row0, s_valid)
    hdr = dict(S=S, cp=cp, rank=rank, L=L, row_offset=row0, s_valid=s_valid,
               n_pad=n_pad, kv_start=kv_start, kv_end=kv_end, nseg=len(segs))
    return {"hdr": hdr, "segs": segs}


def useful_pairs(cu, S: int, cp: int) -> int:
    """Number of unmasked (query, key) pairs per head over all chunks,
    counted by brute force over the document-id array."""
    ids = doc_ids(cu, S)
    n = 0
    for i in range(S):
        if ids[i] < 0:
            continue
        n += int(np.count_nonzero(ids[: i + 1] == ids[i]))
    return n
