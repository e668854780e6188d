"""Oracle for the 1-D document-id input and the needed-only K/V exchange plan.

TEST INFRASTRUCTURE ONLY (see the package docstring).

NeMo Automodel page "block-diagonal varlen CP for packed sequences":
* "1-D document ids" are an alternative to cu_seqlens (Proof, CPU tests): a
  document is a maximal run of equal ids; reading taken here: ids are
  non-decreasing over valid tokens and negative ids mark a padding suffix;
* the needed-only exchanges deliver to each rank the K/V rows from the start of
  the first document its chunk overlaps, by a left-neighbour halo or, when a
  document spans more than two ranks, an all-to-all-v whose backward is an
  index_add at the owners (Summary; Design overview, exchange.py).
Works token by token from the document-id array.
"""
from __future__ import annotations

from .segment import segment_chunk


def doc_ids_to_cu(ids) -> list:
    """cu_seqlens from per-token document ids (runs of equal ids)."""
    ids = [int(x) for x in ids]
    valid = [x for x in ids if x >= 0]
    if any(x >= 0 for x in ids[len(valid):]) or any(x < 0 for x in ids[:len(valid)]):
        raise ValueError("padding must be a suffix")
    if any(b < a for a, b in zip(valid, valid[1:])):
        raise ValueError("document ids must be non-decreasing")
    cu = [0]
    for t in range(1, len(valid) + 1):
        if t == len(valid) or valid[t] != valid[t - 1]:
            cu.append(t)
    return cu


def exchange_plan(cu, S: int, cp: int, rank: int):
    """(kind, transfers) for rank's window; kind 0 local, 1 halo, 2 all-to-all-v.

    Walks the window's rows one by one and groups runs of equal owner rank.
    """
    hdr = segment_chunk(cu, S, cp, rank)["hdr"]
    L = S // cp
    a, e = hdr["kv_start"], hdr["kv_end"]
    xfers = []
    for row in range(a, e):
        owner = row // L
        if xfers and xfers[-1][0] == owner:
            src_rank, src_row, n, dst = xfers[-1]
            xfers[-1] = (src_rank, src_row, n + 1, dst)
        else:
            xfers.append((owner, row, 1, row - a))
    remote = sorted({x[0] for x in xfers} - {rank})
    if not remote:
        kind = 0
    elif remote == [rank - 1]:
        kind = 1
    else:
        kind = 2
    return kind, xfers
