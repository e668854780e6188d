"""block_causal_varlen_gb300 -- block-causal (per-document) varlen attention over
packed sequences, one contiguous context-parallel query chunk at a time, on
GB300 (sm_103a).

The compute lives in libbd.so (CUDA kernels behind a C ABI, see
include/bd_attn.h). This module is the thin Python binding with the same
names: it marshals torch tensors into the ABI's plain pointers and strides.

Tensor layouts (all strided views are accepted; the head dim is contiguous):
    q, out, dout  bf16 [B, nchunks, L, H, d]        dq fp32, same shape
    k, v          bf16 [B, Ck, rows, Hkv, d]        dk, dv fp32, same shape
                  Ck = 1 with all-gathered K/V (row = global row),
                  Ck = nchunks with needed-only windows (row 0 = kv_start)
    lse           fp32 [B, nchunks, H, L]
A whole packed sequence [B, S, H, d] is the view [B, cp, L, H, d].
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _abi
from ._abi import (BD_BWD_DQ_ZEROED, BD_BWD_OWNER_ROWS, BD_KV_GATHER, BD_KV_WINDOW, BDError,  # noqa: F401
                   bd_chunk_hdr, bd_rowstat, bd_segment_t, bd_tensor, check, load)

__all__ = ["Plan", "bd_segment", "bd_doc_ids_to_cu", "bd_exchange_plan", "bd_attn_fwd", "bd_attn_fwd_ex", "bd_attn_bwd",
           "bd_attn_bwd_ex", "bd_attn_bwd_pre", "bd_attn_bwd_main", "bd_attn_bwd_main_ex", "bd_owner_sum",
           "bd_check_status", "bd_attn_bwd_workspace", "attn_fwd", "attn_bwd", "BD_KV_GATHER", "BD_KV_WINDOW",
           "BD_BWD_OWNER_ROWS", "BD_BWD_DQ_ZEROED", "BDError", "load"]

_HDR_FIELDS = ("S", "cp", "rank", "L", "row_offset", "s_valid", "n_pad", "kv_start", "kv_end", "nseg")
_SEG_FIELDS = ("doc", "q_start", "q_len", "k_start", "k_len", "diag_off")


def _i32(arr):
    a = np.ascontiguousarray(np.asarray(arr, dtype=np.int32))
    return a, a.ctypes.data_as(C.POINTER(C.c_int32))


def bd_segment(cu_seqlens, S: int, cp: int, rank: int):
    """Varlen metadata of chunk ``rank``: (header dict, list of segment tuples)."""
    lib = load()
    cu, pcu = _i32(cu_seqlens)
    hdr = bd_chunk_hdr()
    check(lib.bd_segment(pcu, len(cu) - 1, S, cp, rank, C.byref(hdr), None, 0))
    segs = (bd_segment_t * max(1, hdr.nseg))()
    check(lib.bd_segment(pcu, len(cu) - 1, S, cp, rank, C.byref(hdr), segs, hdr.nseg))
    return ({f: getattr(hdr, f) for f in _HDR_FIELDS},
            [tuple(getattr(segs[i], f) for f in _SEG_FIELDS) for i in range(hdr.nseg)])


def bd_doc_ids_to_cu(doc_ids):
    """cu_seqlens (list) from a 1-D per-token document-id array (negative = padding suffix)."""
    lib = load()
    ids, pids = _i32(doc_ids)
    nd = C.c_int32()
    st = lib.bd_doc_ids_to_cu(pids, len(ids), None, 0, C.byref(nd))
    if st not in (0, _abi.BD_ERR_CAPACITY):
        check(st)
    out = (C.c_int32 * (nd.value + 1))()
    check(lib.bd_doc_ids_to_cu(pids, len(ids), out, nd.value + 1, C.byref(nd)))
    return list(out)


def bd_exchange_plan(cu_seqlens, S: int, cp: int, rank: int):
    """Needed-only K/V exchange of chunk ``rank``: (kind, [(src_rank, src_row, n_rows, dst_row), ...])."""
    lib = load()
    cu, pcu = _i32(cu_seqlens)
    kind, n = C.c_int32(), C.c_int32()
    check(lib.bd_exchange_plan(pcu, len(cu) - 1, S, cp, rank, C.byref(kind), None, 0, C.byref(n)))
    xs = (_abi.bd_xfer_t * max(1, n.value))()
    check(lib.bd_exchange_plan(pcu, len(cu) - 1, S, cp, rank, C.byref(kind), xs, n.value, C.byref(n)))
    return kind.value, [(x.src_rank, x.src_row, x.n_rows, x.dst_row) for x in xs[:n.value]]


class Plan:
    """Host plan blob (built once per step) and its device copy.

    ``cu_list``: one cu_seqlens list per sequence; ``ranks``: the chunks the
    plan covers (default: all cp chunks, i.e. the batched single-GPU grid).
    """

    def __init__(self, cu_list, S, cp, H, Hkv, d, kv_mode=BD_KV_GATHER, ranks=None):
        lib = load()
        self.B, self.S, self.cp, self.H, self.Hkv, self.d = len(cu_list), S, cp, H, Hkv, d
        self.L = S // cp if cp > 0 and S % cp == 0 else None
        self.kv_mode = kv_mode
        self.ranks = list(range(cp)) if ranks is None else list(ranks)
        self.nchunks = len(self.ranks)
        self.Ck = 1 if kv_mode == BD_KV_GATHER else self.nchunks
        offs = np.cumsum([0] + [len(c) for c in cu_list]).astype(np.int32)
        self._cu, pcu = _i32(np.concatenate([np.asarray(c, dtype=np.int32) for c in cu_list]))
        self._offs, poffs = _i32(offs)
        self._ranks, pranks = _i32(self.ranks)
        self._desc = _abi.bd_plan_desc(self.B, S, cp, self.nchunks, pranks, H, Hkv, d, kv_mode, pcu, poffs)
        nbytes = C.c_size_t()
        check(lib.bd_plan_bytes(C.byref(self._desc), C.byref(nbytes)))
        self.nbytes = nbytes.value
        raw = np.zeros(self.nbytes // 4 + 16, dtype=np.int32)
        off = (-raw.ctypes.data % 64) // 4
        self.host = raw[off:off + self.nbytes // 4]
        self._raw = raw
        check(lib.bd_plan_build(C.byref(self._desc), C.c_void_p(self.host.ctypes.data), self.nbytes))
        self.dev = None

    @property
    def host_ptr(self):
        return C.c_void_p(self.host.ctypes.data)

    @property
    def dev_ptr(self):
        if self.dev is None:
            raise RuntimeError("plan not uploaded: call .upload(device)")
        return C.c_void_p(self.dev.data_ptr())

    def upload(self, device="cuda", non_blocking=False):
        """Copy the plan blob to device memory (once per step)."""
        src = torch.from_numpy(self.host)
        if self.dev is None or self.dev.device != torch.device(device):
            self.dev = torch.empty_like(src, device=device)
        self.dev.copy_(src, non_blocking=non_blocking)
        return self

    def set_dropout(self, p: float, seed: int):
        """Attention dropout with probability p (0 turns it off) and a 64-bit seed,
        written into the host blob: upload the plan again before the next launch."""
        check(load().bd_plan_set_dropout(self.host_ptr, float(p), int(seed) & (2 ** 64 - 1)))
        return self

    def useful_pairs(self) -> int:
        """Unmasked (query, key) pairs per head over the whole plan."""
        return int(load().bd_plan_useful_pairs(self.host_ptr))

    def chunk(self, item: int):
        lib = load()
        hdr = bd_chunk_hdr()
        check(lib.bd_plan_chunk(self.host_ptr, item, C.byref(hdr), None, 0))
        segs = (bd_segment_t * max(1, hdr.nseg))()
        check(lib.bd_plan_chunk(self.host_ptr, item, C.byref(hdr), segs, hdr.nseg))
        return ({f: getattr(hdr, f) for f in _HDR_FIELDS},
                [tuple(getattr(segs[i], f) for f in _SEG_FIELDS) for i in range(hdr.nseg)])

    def header(self, field: int) -> int:
        return int(self.host[field])

    # index of a few header words (see csrc/plan_layout.h)
    H_NFWD, H_NBWD, H_KV_ROWS, H_SLOTS, H_FWD_TILES_LO, H_FWD_TILES_HI, H_NBWDO = 18, 20, 22, 24, 29, 30, 37

    def slots(self) -> int:
        """Query heads per forward work unit (2 when GQA heads are paired, else 1)."""
        return int(self.host[self.H_SLOTS])

    def fwd_tiles(self) -> int:
        """Key tiles visited by the forward over all work units (each for `slots` heads)."""
        return (int(self.host[self.H_FWD_TILES_HI]) << 31) | int(self.host[self.H_FWD_TILES_LO])

    def row_doc_starts(self):
        """Per chunk item, the global start row of each row's document (int32;
        2**31 - 1 on padding rows), as the kernels read it from the plan."""
        off = int(self.host[31])
        return self.host[off:off + self.B * self.nchunks * self.L].reshape(self.B * self.nchunks, self.L)

    def kv_rows(self) -> int:
        return int(self.host[self.H_KV_ROWS])

    def owner_units(self) -> int:
        """Backward work units of the plan's owner-keyed list (0 when the plan has
        none: it needs BD_KV_WINDOW, every chunk 0..cp-1 in order, L % 128 == 0)."""
        return int(self.host[self.H_NBWDO])


def _tensor(t: torch.Tensor, name: str) -> bd_tensor:
    if t.dim() != 5:
        raise ValueError(f"{name}: expected a 5-D tensor [B, C, rows, heads, d], got {tuple(t.shape)}")
    if t.stride(4) != 1:
        raise ValueError(f"{name}: head dim must be contiguous")
    s = t.stride()
    return bd_tensor(t.data_ptr(), s[0], s[1], s[2], s[3], t.shape[2], 0)


def _rowstat(t: torch.Tensor, name: str) -> bd_rowstat:
    if t.dim() != 4 or t.stride(3) != 1 or t.dtype != torch.float32:
        raise ValueError(f"{name}: expected fp32 [B, C, H, L] with L contiguous")
    s = t.stride()
    return bd_rowstat(t.data_ptr(), s[0], s[1], s[2])


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check_args(plan: Plan, bf16=(), fp32=(), other=()):
    """The C ABI carries no dtypes, so the binding checks them (a wrong one would
    make a kernel read or write past a buffer): bf16 / fp32 tensors as named, every
    tensor on the plan's device."""
    for group, dtype in ((bf16, torch.bfloat16), (fp32, torch.float32)):
        for t, n in group:
            if t.dtype != dtype:
                raise TypeError(f"{n}: dtype {t.dtype}, expected {dtype}")
    dev = plan.dev.device if plan.dev is not None else None
    for t, n in (*bf16, *fp32, *other):
        if not t.is_cuda:
            raise TypeError(f"{n}: must be a CUDA tensor")
        if dev is not None and t.device != dev:
            raise ValueError(f"{n}: on {t.device}, the plan was uploaded to {dev}")


def bd_attn_fwd(plan: Plan, q, k, v, out, lse, row_offset: int = -1, stream=None):
    """Forward of every chunk item in ``plan`` (see include/bd_attn.h)."""
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (out, "out")), fp32=((lse, "lse"),))
    tq, tk, tv, to = _tensor(q, "q"), _tensor(k, "k"), _tensor(v, "v"), _tensor(out, "out")
    tl = _rowstat(lse, "lse")
    check(load().bd_attn_fwd(plan.host_ptr, plan.dev_ptr, C.byref(tq), C.byref(tk), C.byref(tv), row_offset,
                             C.byref(to), C.byref(tl), _stream(stream)))


def bd_attn_fwd_ex(plan: Plan, q, k, v, out, lse, dq_zero=None, row_offset: int = -1, stream=None):
    """bd_attn_fwd that also zeroes ``dq_zero`` (fp32, the backward's dq
    accumulator) while the forward runs; see include/bd_attn.h."""
    fp32 = ((lse, "lse"),) + (((dq_zero, "dq_zero"),) if dq_zero is not None else ())
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (out, "out")), fp32=fp32)
    tq, tk, tv, to = _tensor(q, "q"), _tensor(k, "k"), _tensor(v, "v"), _tensor(out, "out")
    tl = _rowstat(lse, "lse")
    tz = C.byref(_tensor(dq_zero, "dq_zero")) if dq_zero is not None else None
    check(load().bd_attn_fwd_ex(plan.host_ptr, plan.dev_ptr, C.byref(tq), C.byref(tk), C.byref(tv), row_offset,
                                C.byref(to), C.byref(tl), tz, _stream(stream)))


def bd_attn_bwd_workspace(plan: Plan) -> int:
    n = C.c_size_t()
    check(load().bd_attn_bwd_workspace(plan.host_ptr, C.byref(n)))
    return n.value


def bd_attn_bwd(plan: Plan, q, k, v, out, dout, lse, dq, dk, dv, workspace, accumulate_dkv=False,
                stream=None):
    """Backward of every chunk item in ``plan`` (see include/bd_attn.h)."""
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")),
                fp32=((lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")), other=((workspace, "workspace"),))
    ts = [_tensor(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"))]
    tl = _rowstat(lse, "lse")
    tdq, tdk, tdv = _tensor(dq, "dq"), _tensor(dk, "dk"), _tensor(dv, "dv")
    check(load().bd_attn_bwd(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts], C.byref(tl), C.byref(tdq),
                             C.byref(tdk), C.byref(tdv), int(bool(accumulate_dkv)),
                             C.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                             _stream(stream)))


def bd_attn_bwd_ex(plan: Plan, q, k, v, out, dout, lse, dq, dk, dv, workspace, flags: int, accumulate_dkv=False,
                   stream=None):
    """bd_attn_bwd with flags: BD_BWD_OWNER_ROWS (dk, dv are owner-row tensors
    [B, 1, S, Hkv, d] summed over chunks), BD_BWD_DQ_ZEROED (dq already zero)."""
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")),
                fp32=((lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")), other=((workspace, "workspace"),))
    ts = [_tensor(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"))]
    tl = _rowstat(lse, "lse")
    tdq, tdk, tdv = _tensor(dq, "dq"), _tensor(dk, "dk"), _tensor(dv, "dv")
    check(load().bd_attn_bwd_ex(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts], C.byref(tl),
                                C.byref(tdq), C.byref(tdk), C.byref(tdv), int(bool(accumulate_dkv)), int(flags),
                                C.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                                _stream(stream)))


def bd_attn_bwd_pre(plan: Plan, out, dout, lse, dq, workspace, stream=None, clear_dq=True):
    """First backward step only: D, log2 LSE, document starts; zeroes dq unless
    clear_dq is False (the caller then zeroes it before bd_attn_bwd_main)."""
    _check_args(plan, bf16=((out, "out"), (dout, "dout")), fp32=((lse, "lse"), (dq, "dq")),
                other=((workspace, "workspace"),))
    to, tg, tq = _tensor(out, "out"), _tensor(dout, "dout"), _tensor(dq, "dq")
    tl = _rowstat(lse, "lse")
    check(load().bd_attn_bwd_pre_ex(plan.host_ptr, plan.dev_ptr, C.byref(to), C.byref(tg), C.byref(tl),
                                    C.byref(tq), C.c_void_p(workspace.data_ptr()),
                                    workspace.numel() * workspace.element_size(), int(bool(clear_dq)),
                                    _stream(stream)))


def bd_attn_bwd_main(plan: Plan, q, k, v, dout, dq, dk, dv, workspace, accumulate_dkv=False, stream=None):
    """Second backward step only: dq, dk, dv from the workspace bd_attn_bwd_pre filled."""
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (dout, "dout")), fp32=((dq, "dq"), (dk, "dk"), (dv, "dv")),
                other=((workspace, "workspace"),))
    ts = [_tensor(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout"), (dq, "dq"), (dk, "dk"),
                                      (dv, "dv"))]
    check(load().bd_attn_bwd_main(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts],
                                  int(bool(accumulate_dkv)), C.c_void_p(workspace.data_ptr()),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def bd_attn_bwd_main_ex(plan: Plan, q, k, v, dout, dq, dk, dv, workspace, flags: int, accumulate_dkv=False,
                        stream=None):
    """bd_attn_bwd_main with flags (BD_BWD_OWNER_ROWS: dk, dv at owner rows)."""
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (dout, "dout")), fp32=((dq, "dq"), (dk, "dk"), (dv, "dv")),
                other=((workspace, "workspace"),))
    ts = [_tensor(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout"), (dq, "dq"), (dk, "dk"),
                                      (dv, "dv"))]
    check(load().bd_attn_bwd_main_ex(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts],
                                     int(bool(accumulate_dkv)), int(flags), C.c_void_p(workspace.data_ptr()),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def bd_owner_sum(plan: Plan, dk_win, dv_win, dk, dv, stream=None, accumulate=True):
    """Sum needed-only-window dK/dV partials at their owner rows, added into dk/dv
    (accumulate=True) or stored there (accumulate=False: every owner row is
    written); see include/bd_attn.h."""
    _check_args(plan, fp32=((dk_win, "dk_win"), (dv_win, "dv_win"), (dk, "dk"), (dv, "dv")))
    ts = [_tensor(x, n) for x, n in ((dk_win, "dk_win"), (dv_win, "dv_win"), (dk, "dk"), (dv, "dv"))]
    check(load().bd_owner_sum_ex(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts], int(bool(accumulate)),
                                 _stream(stream)))


def bd_attn_bwd_pre_ex(plan: Plan, out, dout, lse, dq, workspace, clear_dq: bool, stream=None):
    """bd_attn_bwd_pre with an explicit clear_dq (the C entry point's form)."""
    bd_attn_bwd_pre(plan, out, dout, lse, dq, workspace, stream=stream, clear_dq=clear_dq)


def bd_owner_sum_ex(plan: Plan, dk_win, dv_win, dk, dv, accumulate: bool, stream=None):
    """bd_owner_sum with an explicit accumulate (the C entry point's form)."""
    bd_owner_sum(plan, dk_win, dv_win, dk, dv, stream=stream, accumulate=accumulate)


def bd_attn_bwd_noalloc(plan: Plan, q, k, v, out, dout, lse, dq, dk, dv, accumulate_dkv=False, stream=None):
    """bd_attn_bwd with the library's fixed device workspace instead of a caller
    buffer, for callers that cannot allocate (see include/bd_attn.h)."""
    _check_args(plan, bf16=((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")),
                fp32=((lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")))
    ts = [_tensor(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"))]
    tl = _rowstat(lse, "lse")
    tdq, tdk, tdv = _tensor(dq, "dq"), _tensor(dk, "dk"), _tensor(dv, "dv")
    check(load().bd_attn_bwd_noalloc(plan.host_ptr, plan.dev_ptr, *[C.byref(t) for t in ts], C.byref(tl),
                                     C.byref(tdq), C.byref(tdk), C.byref(tdv), int(bool(accumulate_dkv)),
                                     _stream(stream)))


def bd_attn_bwd_noalloc_capacity() -> int:
    """Bytes of the fixed workspace bd_attn_bwd_noalloc draws on."""
    return int(load().bd_attn_bwd_noalloc_capacity())


def bd_padded_len(s: int, cp: int) -> int:
    """Smallest multiple of cp that is >= s."""
    n = int(load().bd_padded_len(int(s), int(cp)))
    check(min(n, 0))
    return n


def bd_version() -> int:
    return int(load().bd_version())


def bd_last_error() -> str:
    """Message of this thread's last failed call."""
    m = load().bd_last_error()
    return m.decode() if m else ""


def bd_check_status(plan: Plan, reset: bool = True, stream=None):
    check(load().bd_check_status(plan.dev_ptr, int(reset), _stream(stream)))


# ---------------------------------------------------------------- conveniences

def attn_fwd(plan: Plan, q, k, v, stream=None):
    """Allocate O and LSE and run the forward; returns (out, lse)."""
    B, Cn, L, H, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty(B, Cn, H, L, dtype=torch.float32, device=q.device)
    bd_attn_fwd(plan, q, k, v, out, lse, stream=stream)
    return out, lse


def attn_bwd(plan: Plan, q, k, v, out, dout, lse, stream=None):
    """Allocate gradients and run the backward; returns (dq, dk, dv)."""
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    ws = torch.empty(max(1, bd_attn_bwd_workspace(plan)), dtype=torch.uint8, device=q.device)
    bd_attn_bwd(plan, q, k, v, out, dout, lse, dq, dk, dv, ws, stream=stream)
    return dq, dk, dv
