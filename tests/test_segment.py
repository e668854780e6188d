"""Segmentation: the oracle against a hand-worked fixture and closed forms, then
the library's bd_segment / plan against the oracle, bit-exact (CPU only)."""
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "segment_tiny_3docs.txt")


def _read_golden():
    chunks, layout = [], None
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "layout":
            S, cp, *cu = map(int, f[1:])
            layout = (cu, S, cp)
        elif f[0] == "chunk":
            rank, row0, sv, npad, ks, ke, nseg, useful = map(int, f[1:])
            chunks.append(dict(rank=rank, row_offset=row0, s_valid=sv, n_pad=npad, kv_start=ks, kv_end=ke,
                               nseg=nseg, useful=useful, segs=[]))
        elif f[0] == "seg":
            chunks[-1]["segs"].append(tuple(map(int, f[1:])))
    return layout, chunks


def _useful(segs):
    return sum(ql * (kl - ql) + ql * (ql + 1) // 2 for _, _, ql, _, kl, _ in segs)


def test_oracle_segmentation_matches_hand_worked_fixture():
    (cu, S, cp), chunks = _read_golden()
    for ch in chunks:
        got = oracle.segment_chunk(cu, S, cp, ch["rank"])
        h = got["hdr"]
        for key in ("row_offset", "s_valid", "n_pad", "kv_start", "kv_end", "nseg"):
            assert h[key] == ch[key], key
        assert got["segs"] == ch["segs"]
        assert _useful(got["segs"]) == ch["useful"]
    assert sum(c["useful"] for c in chunks) == oracle.useful_pairs(cu, S, cp)


def test_oracle_single_document_closed_form():
    """One document of S rows in cp chunks: chunk r is one segment with queries
    [rL, (r+1)L), keys [0, (r+1)L) and diagonal offset rL."""
    S, cp = 1536, 8
    L = S // cp
    for r in range(cp):
        got = oracle.segment_chunk([0, S], S, cp, r)
        assert got["segs"] == [(0, r * L, L, 0, (r + 1) * L, r * L)]
        assert got["hdr"]["kv_start"] == 0 and got["hdr"]["kv_end"] == (r + 1) * L
    assert sum(_useful(oracle.segment_chunk([0, S], S, cp, r)["segs"]) for r in range(cp)) == S * (S + 1) // 2


@pytest.mark.parametrize("seed", range(12))
def test_oracle_useful_pairs_closed_form(seed):
    rng = np.random.default_rng(seed)
    S, cp = 96, int(rng.choice([1, 2, 3, 4]))
    cu = workloads.random_layout(rng, S, cp)
    total = sum(_useful(oracle.segment_chunk(cu, S, cp, r)["segs"]) for r in range(cp))
    lens = np.diff(cu)
    assert total == int((lens * (lens + 1) // 2).sum()) == oracle.useful_pairs(cu, S, cp)


# ---- the library against the oracle ------------------------------------------------

lib = pytest.importorskip("block_causal_varlen_gb300")


def _lib_ok():
    try:
        lib.load()
        return True
    except RuntimeError:
        return False


pytestmark_lib = pytest.mark.skipif(not _lib_ok(), reason="libbd.so not built")


def _compare(cu, S, cp):
    for r in range(cp):
        want = oracle.segment_chunk(cu, S, cp, r)
        hdr, segs = lib.bd_segment(cu, S, cp, r)
        assert segs == want["segs"], (cu, S, cp, r)
        for key, val in want["hdr"].items():
            assert hdr[key] == val, (key, cu, S, cp, r)


@pytestmark_lib
def test_library_matches_fixture_and_oracle():
    (cu, S, cp), chunks = _read_golden()
    _compare(cu, S, cp)
    for ch in chunks:
        _, segs = lib.bd_segment(cu, S, cp, ch["rank"])
        assert segs == ch["segs"]


@pytestmark_lib
@pytest.mark.parametrize("seed", range(40))
def test_library_matches_oracle_random(seed):
    rng = np.random.default_rng(1000 + seed)
    cp = int(rng.choice([1, 2, 3, 4, 8]))
    S = cp * int(rng.integers(1, 40))
    cu = workloads.random_layout(rng, S, cp, max_docs=int(rng.integers(1, 10)))
    _compare(cu, S, cp)


@pytestmark_lib
@pytest.mark.parametrize("i", [1, 2, 3, 4, 5])
def test_library_matches_oracle_on_workloads(i):
    wl = workloads.config(i)
    for cu in wl.cu:
        _compare(cu, wl.S, wl.cp)


@pytestmark_lib
@pytest.mark.parametrize("i", [1, 2, 3, 5])
def test_plan_items_match_oracle_and_useful_pairs(i):
    wl = workloads.config(i)
    for mode in (lib.BD_KV_GATHER, lib.BD_KV_WINDOW):
        plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode)
        useful = 0
        for b, cu in enumerate(wl.cu):
            for r in range(wl.cp):
                hdr, segs = plan.chunk(b * wl.cp + r)
                want = oracle.segment_chunk(cu, wl.S, wl.cp, r)
                assert segs == want["segs"]
                assert {k: hdr[k] for k in want["hdr"]} == want["hdr"]
                useful += _useful(want["segs"])
        assert plan.useful_pairs() == useful
        lens = np.concatenate([np.diff(c) for c in wl.cu]) if any(len(c) > 1 for c in wl.cu) else np.zeros(0)
        assert useful == int((lens * (lens + 1) // 2).sum())


@pytestmark_lib
def test_plan_is_deterministic_bytes():
    wl = workloads.config(3)
    a = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=lib.BD_KV_WINDOW)
    b = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=lib.BD_KV_WINDOW)
    assert np.array_equal(a.host, b.host)


@pytestmark_lib
@pytest.mark.parametrize("cu,S,cp,rank,status", [
    ([1, 5], 8, 2, 0, lib.BDError),          # cu[0] != 0
    ([0, 5, 3], 8, 2, 0, lib.BDError),       # decreasing
    ([0, 9], 8, 2, 0, lib.BDError),          # beyond S
    ([0, 5], 9, 2, 0, lib.BDError),          # S not a multiple of cp
    ([0, 5], 8, 2, 2, lib.BDError),          # rank out of range
    ([0, 5], 8, 2, -1, lib.BDError),
    ([0, 5], 8, 0, 0, lib.BDError),          # cp = 0
])
def test_library_rejects_bad_metadata(cu, S, cp, rank, status):
    with pytest.raises(status) as e:
        lib.bd_segment(cu, S, cp, rank)
    assert e.value.status in (lib._abi.BD_ERR_CU_SEQLENS, lib._abi.BD_ERR_NOT_DIVISIBLE, lib._abi.BD_ERR_RANK,
                              lib._abi.BD_ERR_ARG)


@pytestmark_lib
def test_library_reports_capacity():
    import ctypes as C
    L = lib.load()
    cu = (C.c_int32 * 4)(0, 3, 6, 8)
    hdr = lib.bd_chunk_hdr()
    segs = (lib.bd_segment_t * 1)()
    st = L.bd_segment(cu, 3, 8, 1, 0, C.byref(hdr), segs, 1)
    assert st == lib._abi.BD_ERR_CAPACITY and hdr.nseg == 3
    assert b"capacity" in L.bd_last_error()


@pytestmark_lib
def test_plan_rejects_bad_desc():
    with pytest.raises(lib.BDError):
        lib.Plan([[0, 100]], 100, 3, 4, 4, 64)            # S % cp
    with pytest.raises(lib.BDError):
        lib.Plan([[0, 100]], 100, 2, 6, 4, 64)            # H % Hkv
    with pytest.raises(lib.BDError):
        lib.Plan([[0, 100]], 100, 2, 4, 4, 96)            # head dim
    with pytest.raises(lib.BDError):
        lib.Plan([[0, 100]], 100, 2, 4, 4, 64, ranks=[0, 2])  # rank out of range


@pytestmark_lib
@pytest.mark.parametrize("i", [1, 2, 3, 5])
def test_plan_row_doc_starts_match_oracle(i):
    """The per-row document starts the kernels read from the plan equal the
    first index of each row's document id (padding rows: 2**31 - 1)."""
    wl = workloads.config(i)
    plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d)
    got = plan.row_doc_starts()
    for b, cu in enumerate(wl.cu):
        ids = oracle.doc_ids(cu, wl.S)
        first = {}
        for t, x in enumerate(ids):
            if x >= 0 and x not in first:
                first[x] = t
        want = np.array([first[x] if x >= 0 else 2 ** 31 - 1 for x in ids], dtype=np.int64)
        assert np.array_equal(got[b * wl.cp:(b + 1) * wl.cp].reshape(-1).astype(np.int64), want)


# plan blob words read below (the layout of block_causal_varlen_gb300/csrc/plan_layout.h)
_H_NITEMS, _H_OFF_ITEMS, _H_OFF_BWD, _H_NBWD, _H_CK, _H_OFF_BWDO, _H_NBWDO = 13, 14, 19, 20, 23, 36, 37
_ITEM_WORDS, _I_B, _I_ROW0, _I_SVALID, _I_KVSTART, _I_KVEND, _I_KVBASE = 16, 0, 3, 4, 6, 7, 10
# load buffer, load row, K/V head, item_lo, item_hi, steps, q_lo, q_hi, first key row, output buffer,
# output row, pad
_BWD_WORDS = 12


def _check_unit_queries(wl, items, doc, it_lo, it_hi, c0, c1, nq, q_lo, q_hi, qstep):
    """The unit's query range is exactly the rows attending to a key in [c0, c1)
    and its step count the (query step, query head) pairs that touch them."""
    G = wl.H // wl.Hkv
    attend = np.zeros(wl.S, dtype=bool)
    for x in sorted(set(doc[c0:c1].tolist()) - {-1}):   # earliest key of each document in the tile
        jmin = c0 + int(np.argmax(doc[c0:c1] == x))
        attend |= (doc == x) & (np.arange(wl.S) >= jmin)
    rows_att = np.flatnonzero(attend)
    if len(rows_att) == 0:
        assert nq == 0 and q_lo == q_hi
        return
    assert (q_lo, q_hi) == (int(rows_att[0]), int(rows_att[-1]) + 1)
    assert len(rows_att) == q_hi - q_lo            # contiguous
    steps = 0
    for it in range(it_lo, it_hi):
        r0 = int(items[it][_I_ROW0])
        for t in range(-(-wl.L // qstep)):
            lo, hi = r0 + t * qstep, min(r0 + (t + 1) * qstep, r0 + wl.L)
            steps += bool(attend[lo:hi].any())
    assert nq == G * steps


def _units(h, off, n):
    return h[h[off]:h[off] + h[n] * _BWD_WORDS].reshape(-1, _BWD_WORDS)


@pytestmark_lib
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("i", [1, 2, 3, 5])
def test_plan_backward_units_match_brute_force(i, d):
    """Every backward work unit (one 128-key tile of a K/V buffer, one K/V head)
    against a brute force over document ids: its query range is exactly the rows
    that attend to a key of the tile, and its step count is the number of
    (query step, query head) pairs that touch those rows, with steps of 128 rows
    (64 at head dim 256). Every (buffer, tile, head) appears once, and its dK / dV
    rows go back to the same buffer rows."""
    wl = workloads.config(i)
    qstep = 64 if d == 256 else 128
    for mode in (lib.BD_KV_GATHER, lib.BD_KV_WINDOW):
        plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, d, kv_mode=mode)
        h = plan.host
        items = h[h[_H_OFF_ITEMS]:h[_H_OFF_ITEMS] + h[_H_NITEMS] * _ITEM_WORDS].reshape(-1, _ITEM_WORDS)
        units = _units(h, _H_OFF_BWD, _H_NBWD)
        ids = [oracle.doc_ids(cu, wl.S) for cu in wl.cu]
        seen = set()
        for buf, lrow, g, it_lo, it_hi, nq, q_lo, q_hi, key0, obuf, orow, _ in units.tolist():
            assert lrow % 128 == 0 and (obuf, orow) == (buf, lrow)
            kt = lrow // 128
            assert (buf, kt, g) not in seen
            seen.add((buf, kt, g))
            I0 = items[it_lo]
            b, kv_base, svalid = int(I0[_I_B]), int(I0[_I_KVBASE]), int(I0[_I_SVALID])
            assert key0 == kv_base + lrow
            rows = wl.S if mode == lib.BD_KV_GATHER else int(I0[_I_KVEND] - I0[_I_KVSTART])
            c0, c1 = kv_base + kt * 128, min(kv_base + kt * 128 + 128, kv_base + rows, svalid)
            _check_unit_queries(wl, items, ids[b], it_lo, it_hi, c0, c1, nq, q_lo, q_hi, qstep)
        nbuf = wl.B if mode == lib.BD_KV_GATHER else wl.B * wl.cp
        assert len(seen) == len(units) and {u[0] for u in seen} <= set(range(nbuf))
        for nb in range(nbuf):   # every key tile of every buffer, for every K/V head
            I0 = items[nb * wl.cp if mode == lib.BD_KV_GATHER else nb]
            rows = wl.S if mode == lib.BD_KV_GATHER else int(I0[_I_KVEND] - I0[_I_KVSTART])
            want = {(nb, kt, g) for kt in range(-(-rows // 128)) for g in range(wl.Hkv)}
            assert {u for u in seen if u[0] == nb} == want
        # the owner-keyed list exists for needed-only windows over every chunk (L % 128 == 0 here)
        assert (plan.owner_units() > 0) == (mode == lib.BD_KV_WINDOW)


@pytestmark_lib
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("i", [1, 2, 3, 5])
def test_plan_owner_units_match_brute_force(i, d):
    """The owner-keyed backward list of a needed-only-window plan: one unit per
    (sequence, 128-row tile of the global row grid, K/V head), every one exactly
    once; K / V come from the window of the chunk that owns the tile, at the rows
    that hold the tile's global rows; every chunk of the sequence contributes and
    the result goes to the owner rows; the query range and step count match the
    brute force over document ids."""
    wl = workloads.config(i)
    qstep = 64 if d == 256 else 128
    plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, d, kv_mode=lib.BD_KV_WINDOW)
    h = plan.host
    items = h[h[_H_OFF_ITEMS]:h[_H_OFF_ITEMS] + h[_H_NITEMS] * _ITEM_WORDS].reshape(-1, _ITEM_WORDS)
    units = _units(h, _H_OFF_BWDO, _H_NBWDO)
    assert len(units) == wl.B * (wl.S // 128) * wl.Hkv
    ids = [oracle.doc_ids(cu, wl.S) for cu in wl.cu]
    seen = set()
    for buf, lrow, g, it_lo, it_hi, nq, q_lo, q_hi, key0, obuf, orow, _ in units.tolist():
        b = obuf
        assert (it_lo, it_hi) == (b * wl.cp, (b + 1) * wl.cp)
        assert orow == key0 and key0 % 128 == 0
        assert (b, key0, g) not in seen
        seen.add((b, key0, g))
        own = b * wl.cp + key0 // wl.L
        assert buf == own
        svalid = int(items[own][_I_SVALID])
        c1 = min(key0 + 128, svalid)
        if c1 > key0:   # the owner's window holds the tile's valid rows at lrow..
            kvs, kve = int(items[own][_I_KVSTART]), int(items[own][_I_KVEND])
            assert lrow == key0 - kvs and kvs <= key0 and c1 <= kve
        _check_unit_queries(wl, items, ids[b], it_lo, it_hi, key0, max(c1, key0), nq, q_lo, q_hi, qstep)
    assert seen == {(b, kt * 128, g) for b in range(wl.B) for kt in range(wl.S // 128) for g in range(wl.Hkv)}
    # the same work as the per-window list, tile by tile (both count every attending
    # (query step, head) pair of every chunk once per key tile of their own grids)
    steps_owner = int(units[:, 5].sum())
    assert steps_owner > 0


@pytestmark_lib
def test_owner_units_only_for_whole_window_plans():
    """No owner list (the owner-row backward refuses the plan) for all-gathered K/V,
    a subset of the chunks, or L not a multiple of 128."""
    cu = [[0, 300, 700, 1000]]
    assert lib.Plan(cu, 1024, 4, 4, 4, 64, kv_mode=lib.BD_KV_WINDOW).owner_units() == 8 * 4  # L = 256
    assert lib.Plan(cu, 1024, 2, 4, 4, 64, kv_mode=lib.BD_KV_WINDOW).owner_units() > 0     # L = 512
    assert lib.Plan(cu, 1024, 2, 4, 4, 64, kv_mode=lib.BD_KV_GATHER).owner_units() == 0
    assert lib.Plan(cu, 1024, 2, 4, 4, 64, kv_mode=lib.BD_KV_WINDOW, ranks=[1]).owner_units() == 0
    assert lib.Plan(cu, 1200, 4, 4, 4, 64, kv_mode=lib.BD_KV_WINDOW).owner_units() == 0   # L = 300


@pytestmark_lib
@pytest.mark.parametrize("i", [1, 2, 3, 4, 5])
def test_visited_tiles_match_brute_force(i):
    """The forward visits exactly the 128 x 128 (query tile, key tile) pairs that
    hold at least one unmasked (row, key): query tiles on each chunk's row grid,
    key tiles on the global 128-row grid, counted by brute force over every row's
    key interval [document start, row] (from the document ids)."""
    wl = workloads.config(i)
    for mode in (lib.BD_KV_GATHER, lib.BD_KV_WINDOW):
        plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode)
        want = 0
        for b, cu in enumerate(wl.cu):
            ids = oracle.doc_ids(cu, wl.S)
            start = np.full(wl.S, -1, dtype=np.int64)
            for x in range(len(cu) - 1):
                start[cu[x]:cu[x + 1]] = cu[x]
            for c in range(wl.cp):
                for t in range(-(-wl.L // 128)):
                    lo, hi = c * wl.L + t * 128, min(c * wl.L + (t + 1) * 128, (c + 1) * wl.L)
                    rows = np.arange(lo, hi)
                    rows = rows[ids[rows] >= 0]
                    if len(rows) == 0:
                        continue
                    tiles = set()
                    for r in rows:   # key tiles met by [start(r), r]
                        tiles.update(range(start[r] // 128, r // 128 + 1))
                    want += len(tiles)
        assert plan.fwd_tiles() * plan.slots() == want * wl.H, (i, mode)


_H_OFF_FWD, _H_NFWD, _H_SLOTS, _FWD_WORDS = 17, 18, 24, 8


@pytestmark_lib
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("i", [1, 2, 3, 4, 5])
def test_plan_forward_list_order(i, d):
    """The forward work list holds every (item, query tile, head pair) once and runs
    longest unit first; lists whose units visit at most 5 key tiles on average (per
    unit that visits any) run in length bands instead (band = the key-tile total
    over 152 x 8, longest band first) with the units of a band in position order
    (item, query tile, first head). Ties always keep position order."""
    wl = workloads.config(i)
    plan = lib.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, d, kv_mode=lib.BD_KV_WINDOW)
    h = plan.host
    fw = h[h[_H_OFF_FWD]:h[_H_OFF_FWD] + h[_H_NFWD] * _FWD_WORDS].reshape(-1, _FWD_WORDS)
    slots = int(h[_H_SLOTS])
    keys = [tuple(int(x) for x in u[:3]) for u in fw]
    want = {(it, t, h0) for it in range(wl.B * wl.cp) for t in range(-(-wl.L // 128))
            for h0 in range(0, wl.H, slots)}
    assert len(keys) == len(set(keys)) and set(keys) == want
    nt = fw[:, 4].astype(np.int64)
    live = int((nt > 0).sum())
    band = max(1, int(nt.sum()) // (152 * 8)) if live and nt.sum() <= 5 * live else 1
    b = nt // band
    assert (np.diff(b) <= 0).all(), "bands must not grow along the list"
    for j in range(1, len(keys)):
        if b[j] == b[j - 1]:
            assert keys[j] > keys[j - 1], f"unit {j} breaks position order inside its band"
    # the short-document layout is the one that takes bands here
    assert (band > 1) == (i == 5)
