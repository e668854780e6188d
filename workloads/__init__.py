"""Seeded synthetic workloads for block-causal varlen attention.

This module is shared by the tests, ``bench.py`` and the oracle's checks. It
holds none of the attention arithmetic: it only draws document lengths
(packed into ``cu_seqlens``) and random bf16 tensors.

The five layouts follow the packed multi-document shapes that the NeMo
Automodel page "block-diagonal varlen CP for packed sequences" (Summary,
Motivation and Proof sections) describes: documents of mixed lengths packed into
one sequence, padded to a multiple of the context-parallel size, split into
contiguous per-rank query chunks, with GQA heads.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = ["Workload", "pack_lengths", "config", "tensors", "NAMES"]


@dataclass
class Workload:
    name: str
    B: int
    S: int          # padded sequence length (multiple of cp)
    cp: int         # number of contiguous query chunks
    H: int          # query heads
    Hkv: int        # key/value heads
    d: int          # head dim
    cu: list        # per sequence: python list of cu_seqlens over valid tokens
    seed: int       # tensor seed
    kv_mode: str    # exchange mode the throughput run uses: "gather" | "window"
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def L(self) -> int:
        return self.S // self.cp

    @property
    def G(self) -> int:
        return self.H // self.Hkv


def pack_lengths(lengths, total: int) -> list:
    """Concatenate document lengths until ``total`` tokens; the last is truncated."""
    cu = [0]
    for ln in lengths:
        if cu[-1] >= total:
            break
        cu.append(min(total, cu[-1] + int(ln)))
    return cu


def _draw_until(draw, total):
    out, s = [], 0
    while s < total:
        ln = int(draw())
        out.append(ln)
        s += ln
    return out


def _max_chunk_span(cu, L):
    return max(((cu[i + 1] - 1) // L - cu[i] // L + 1) for i in range(len(cu) - 1) if cu[i + 1] > cu[i])


NAMES = {
    1: "tiny_s512_3docs_h4_d64_cp2",
    2: "llama8b_s4096_uniformdocs_h32kv8_d128_cp2",
    3: "lognormal_s16384_h32kv8_d128_cp4_window",
    4: "single_doc_s49152_h32kv8_d128_cp8",
    5: "qwen06b_b8_s8192_geomdocs_h16kv8_d128_cp1",
}


def config(i: int, seed: int = 0) -> Workload:
    """Return workload ``i`` (1..5) drawn from ``seed``."""
    if i == 1:
        return Workload(NAMES[1], B=1, S=512, cp=2, H=4, Hkv=4, d=64,
                        cu=[[0, 200, 350, 512]], seed=seed, kv_mode="gather",
                        note="hand-built 3-document layout 200/150/162")
    if i == 2:
        rng = np.random.default_rng(seed)
        lens = _draw_until(lambda: rng.integers(64, 2049), 4096)
        return Workload(NAMES[2], B=1, S=4096, cp=2, H=32, Hkv=8, d=128,
                        cu=[pack_lengths(lens, 4096)], seed=seed, kv_mode="gather",
                        note="doc lengths ~ U{64..2048}, last truncated")
    if i == 3:
        # Lognormal lengths (median 1500), S_valid = 16381 so that the last 3 rows
        # of S = 16384 are masked padding; search seeds upward until one document
        # overlaps at least three of the four chunks.
        s_valid, S, cp = 16381, 16384, 4
        s = seed
        while True:
            rng = np.random.default_rng(s)
            lens = _draw_until(lambda: max(1, int(np.rint(rng.lognormal(np.log(1500.0), 1.0)))), s_valid)
            cu = pack_lengths(lens, s_valid)
            if _max_chunk_span(cu, S // cp) >= 3:
                break
            s += 1
        return Workload(NAMES[3], B=1, S=S, cp=cp, H=32, Hkv=8, d=128, cu=[cu], seed=s,
                        kv_mode="window",
                        note=f"doc lengths max(1, rint(lognormal(ln 1500, 1))), layout seed {s}",
                        extra={"layout_seed": s})
    if i == 4:
        return Workload(NAMES[4], B=1, S=49152, cp=8, H=32, Hkv=8, d=128,
                        cu=[[0, 49152]], seed=seed, kv_mode="gather",
                        note="one document, pure causal")
    if i == 5:
        rng = np.random.default_rng(seed)
        cus = []
        for b in range(8):
            if b == 7:
                cus.append([0])   # a sequence with no documents: its only chunk is all padding
            else:
                lens = _draw_until(lambda: rng.geometric(1.0 / 300.0), 8192)
                cus.append(pack_lengths(lens, 8192))
        return Workload(NAMES[5], B=8, S=8192, cp=1, H=16, Hkv=8, d=128, cu=cus, seed=seed,
                        kv_mode="gather",
                        note="doc lengths ~ geometric(p=1/300); sequence 7 all padding")
    raise ValueError(f"no workload {i}")


def tensors(wl: Workload, heads: slice | None = None):
    """Q, K, V, dO as bf16 CPU tensors, drawn in that order from ``wl.seed``.

    Shapes: Q, dO [B, S, H, d]; K, V [B, S, Hkv, d]; values ~ N(0, 1) rounded
    to bf16.
    """
    g = torch.Generator(device="cpu").manual_seed(wl.seed)
    q = torch.randn(wl.B, wl.S, wl.H, wl.d, generator=g).to(torch.bfloat16)
    k = torch.randn(wl.B, wl.S, wl.Hkv, wl.d, generator=g).to(torch.bfloat16)
    v = torch.randn(wl.B, wl.S, wl.Hkv, wl.d, generator=g).to(torch.bfloat16)
    do = torch.randn(wl.B, wl.S, wl.H, wl.d, generator=g).to(torch.bfloat16)
    return q, k, v, do


def random_layout(rng: np.random.Generator, S: int, cp: int, max_docs: int = 6,
                  pad_max: int | None = None) -> list:
    """A random cu_seqlens over at most S tokens (some trailing padding, some
    zero-length documents allowed) for property tests."""
    pad_max = S // 4 if pad_max is None else pad_max
    s_valid = S - int(rng.integers(0, pad_max + 1))
    n = int(rng.integers(1, max_docs + 1))
    cuts = sorted(int(x) for x in rng.integers(0, s_valid + 1, size=n - 1))
    return [0] + cuts + [s_valid]
