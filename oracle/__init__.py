"""Oracle for block-causal (per-document) varlen chunked attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``block_causal_varlen_gb300``) never imports it and shares no code with it.

It is a plain, slow, obviously correct CPU restatement of what the method
computes, written from the NeMo Automodel page "block-diagonal varlen CP for
packed sequences":

* attention is exactly block-causal per document: a token attends to the
  tokens of its own document at or before its own position, and nothing
  across a document boundary (Summary; Motivation; Key correctness property 1);
* the varlen kernel and a dense masked attention over a materialised mask give
  the same numbers (Summary: "dense masked-SDPA fallback ... numerically
  identical"; Design overview, kernels.py "dense [B,1,L,S] mask builder"), so
  the oracle IS the dense masked form;
* each context-parallel rank owns a contiguous slice of rows, and per-rank
  results concatenated over ranks equal full attention (Design overview,
  batch.py; Key correctness property 1);
* a document straddling a rank's left edge gives an asymmetric first segment,
  K longer than Q, aligned bottom-right (Key correctness property 2);
* the backward of the fused K/V all-gather is a reduce-scatter SUM, i.e. the
  per-chunk dK/dV partials add up at their owners (Design overview,
  exchange.py);
* attention dropout, which the page forwards to the native kernels (Proof,
  GPU varlen tests), is standard dropout on the normalised probabilities with a
  counter-based keep mask (``dropout.py``).

Floating point runs in float64 unless a caller asks for another dtype. The
pieces are pinned by ``tests/test_oracle.py`` and ``tests/test_segment.py``
against brute force, library special cases, closed forms and invariants.
"""
from .segment import doc_ids, segment_chunk, useful_pairs  # noqa: F401
from .exchange import doc_ids_to_cu, exchange_plan  # noqa: F401
from .attention import (  # noqa: F401
    block_causal_mask, attention_fwd, attention_bwd, chunk_fwd, chunk_bwd,
    attention_bwd_cols, attention_bwd_rows,
)
from .dropout import (  # noqa: F401
    philox4x32_10, keep_threshold, keep_mask, attention_fwd_dropout, attention_bwd_dropout,
    chunk_fwd_dropout, chunk_bwd_dropout, attention_rows_dropout, attention_bwd_cols_dropout,
)
