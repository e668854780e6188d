"""1-D document-id input and needed-only exchange plans: oracle pins, then the
library against the oracle (bit-exact), then the exchange itself over gloo."""
import numpy as np
import pytest

import oracle
import workloads

lib = pytest.importorskip("block_causal_varlen_gb300")


def test_oracle_doc_ids_roundtrip_and_rejects():
    for cu, S in (([0, 3, 5, 6], 8), ([0, 10], 10), ([0], 4), ([0, 1, 2, 3], 3)):
        ids = list(oracle.doc_ids(cu, S))
        assert oracle.doc_ids_to_cu(ids) == cu
    with pytest.raises(ValueError):
        oracle.doc_ids_to_cu([0, 0, -1, 1])       # padding not a suffix
    with pytest.raises(ValueError):
        oracle.doc_ids_to_cu([0, 1, 1, 0])        # decreasing


def test_oracle_exchange_plan_hand_cases():
    # one document over all four ranks of 8 rows: rank 3 needs every rank's rows
    kind, xs = oracle.exchange_plan([0, 3, 29], 32, 4, 3)
    assert kind == 2 and xs == [(0, 3, 5, 0), (1, 8, 8, 5), (2, 16, 8, 13), (3, 24, 5, 21)]
    # straddling document reaching back one rank: halo
    kind, xs = oracle.exchange_plan([0, 10, 24, 30], 32, 2, 1)
    assert kind == 1 and xs == [(0, 10, 6, 0), (1, 16, 14, 6)]
    # boundary on the chunk edge: local only
    kind, xs = oracle.exchange_plan([0, 8, 16], 16, 2, 1)
    assert kind == 0 and xs == [(1, 8, 8, 0)]
    # all-padding chunk: empty window
    assert oracle.exchange_plan([0, 7, 12], 32, 2, 1) == (0, [])


@pytest.mark.parametrize("seed", range(30))
def test_library_doc_ids_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 64))
    cu = workloads.random_layout(rng, S, 1)
    cu = [cu[0]] + [c for i, c in enumerate(cu[1:], 1) if c > cu[i - 1]]   # drop empty documents
    ids = list(oracle.doc_ids(cu, S))
    assert lib.bd_doc_ids_to_cu(ids) == oracle.doc_ids_to_cu(ids) == cu


def test_library_doc_ids_rejects():
    for bad in ([0, 0, -1, 1], [0, 1, 1, 0]):
        with pytest.raises(lib.BDError):
            lib.bd_doc_ids_to_cu(bad)


@pytest.mark.parametrize("i", [1, 2, 3, 4, 5])
def test_library_exchange_plan_matches_oracle_on_workloads(i):
    wl = workloads.config(i)
    kinds = set()
    for cu in wl.cu:
        for r in range(wl.cp):
            got = lib.bd_exchange_plan(cu, wl.S, wl.cp, r)
            assert got == oracle.exchange_plan(cu, wl.S, wl.cp, r)
            kinds.add(got[0])
    if i == 3:
        assert 2 in kinds       # a document spans more than two chunks
    if i == 4:
        assert kinds == {0, 1, 2}


@pytest.mark.parametrize("seed", range(30))
def test_library_exchange_plan_matches_oracle_random(seed):
    rng = np.random.default_rng(500 + seed)
    cp = int(rng.choice([1, 2, 3, 4, 8]))
    S = cp * int(rng.integers(1, 30))
    cu = workloads.random_layout(rng, S, cp, max_docs=int(rng.integers(1, 8)))
    for r in range(cp):
        assert lib.bd_exchange_plan(cu, S, cp, r) == oracle.exchange_plan(cu, S, cp, r)
