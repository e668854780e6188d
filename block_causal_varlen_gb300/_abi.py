"""ctypes binding of libbd (the C ABI declared in include/bd_attn.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels. PyTorch provides device memory and streams.
Loading fails loudly when libbd.so has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbd.so")

BD_OK = 0
BD_ERR_ARG = -1
BD_ERR_CU_SEQLENS = -2
BD_ERR_NOT_DIVISIBLE = -3
BD_ERR_RANK = -4
BD_ERR_CAPACITY = -5
BD_ERR_ALIGN = -6
BD_ERR_UNSUPPORTED = -7
BD_ERR_CUDA = -8
BD_ERR_DEVICE_TIMEOUT = -9
BD_ERR_PLAN = -10

BD_KV_GATHER = 0
BD_KV_WINDOW = 1

BD_BWD_OWNER_ROWS = 1
BD_BWD_DQ_ZEROED = 2


class bd_segment_t(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("doc", "q_start", "q_len", "k_start", "k_len", "diag_off")]


class bd_chunk_hdr(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("S", "cp", "rank", "L", "row_offset", "s_valid", "n_pad",
                                          "kv_start", "kv_end", "nseg")]


class bd_xfer_t(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("src_rank", "src_row", "n_rows", "dst_row")]


BD_XCHG_LOCAL, BD_XCHG_HALO, BD_XCHG_A2A = 0, 1, 2


class bd_plan_desc(C.Structure):
    _fields_ = [("B", C.c_int32), ("S", C.c_int32), ("cp", C.c_int32), ("nchunks", C.c_int32),
                ("ranks", C.POINTER(C.c_int32)), ("H", C.c_int32), ("Hkv", C.c_int32), ("d", C.c_int32),
                ("kv_mode", C.c_int32), ("cu_seqlens", C.POINTER(C.c_int32)),
                ("cu_offsets", C.POINTER(C.c_int32))]


class bd_tensor(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("stride_b", C.c_int64), ("stride_c", C.c_int64),
                ("stride_row", C.c_int64), ("stride_head", C.c_int64), ("rows", C.c_int32),
                ("reserved", C.c_int32)]


class bd_rowstat(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("stride_b", C.c_int64), ("stride_c", C.c_int64),
                ("stride_head", C.c_int64)]


EXPORTS = {
    "bd_segment": (C.c_int32, [C.POINTER(C.c_int32), C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                               C.POINTER(bd_chunk_hdr), C.POINTER(bd_segment_t), C.c_int32]),
    "bd_padded_len": (C.c_int32, [C.c_int32, C.c_int32]),
    "bd_doc_ids_to_cu": (C.c_int32, [C.POINTER(C.c_int32), C.c_int32, C.POINTER(C.c_int32), C.c_int32,
                                     C.POINTER(C.c_int32)]),
    "bd_exchange_plan": (C.c_int32, [C.POINTER(C.c_int32), C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                     C.POINTER(C.c_int32), C.POINTER(bd_xfer_t), C.c_int32,
                                     C.POINTER(C.c_int32)]),
    "bd_plan_bytes": (C.c_int32, [C.POINTER(bd_plan_desc), C.POINTER(C.c_size_t)]),
    "bd_plan_build": (C.c_int32, [C.POINTER(bd_plan_desc), C.c_void_p, C.c_size_t]),
    "bd_plan_chunk": (C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(bd_chunk_hdr), C.POINTER(bd_segment_t),
                                  C.c_int32]),
    "bd_plan_useful_pairs": (C.c_int64, [C.c_void_p]),
    "bd_plan_set_dropout": (C.c_int32, [C.c_void_p, C.c_double, C.c_uint64]),
    "bd_attn_fwd": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                C.POINTER(bd_tensor), C.c_int32, C.POINTER(bd_tensor), C.POINTER(bd_rowstat),
                                C.c_void_p]),
    "bd_attn_fwd_ex": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                   C.POINTER(bd_tensor), C.c_int32, C.POINTER(bd_tensor), C.POINTER(bd_rowstat),
                                   C.POINTER(bd_tensor), C.c_void_p]),
    "bd_attn_bwd_workspace": (C.c_int32, [C.c_void_p, C.POINTER(C.c_size_t)]),
    "bd_attn_bwd_ex": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                   C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                   C.POINTER(bd_rowstat), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                   C.POINTER(bd_tensor), C.c_int32, C.c_int32, C.c_void_p, C.c_size_t,
                                   C.c_void_p]),
    "bd_attn_bwd_main_ex": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                        C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                        C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.c_int32, C.c_int32,
                                        C.c_void_p, C.c_size_t, C.c_void_p]),
    "bd_attn_bwd": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                C.POINTER(bd_rowstat), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                C.POINTER(bd_tensor), C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p]),
    "bd_attn_bwd_pre": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                    C.POINTER(bd_rowstat), C.POINTER(bd_tensor), C.c_void_p, C.c_size_t,
                                    C.c_void_p]),
    "bd_attn_bwd_pre_ex": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                       C.POINTER(bd_rowstat), C.POINTER(bd_tensor), C.c_void_p, C.c_size_t,
                                       C.c_int32, C.c_void_p]),
    "bd_attn_bwd_main": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                     C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                     C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.c_int32, C.c_void_p,
                                     C.c_size_t, C.c_void_p]),
    "bd_attn_bwd_noalloc": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                        C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                        C.POINTER(bd_rowstat), C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                        C.POINTER(bd_tensor), C.c_int32, C.c_void_p]),
    "bd_attn_bwd_noalloc_capacity": (C.c_size_t, []),
    "bd_owner_sum": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                 C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.c_void_p]),
    "bd_owner_sum_ex": (C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(bd_tensor), C.POINTER(bd_tensor),
                                    C.POINTER(bd_tensor), C.POINTER(bd_tensor), C.c_int32, C.c_void_p]),
    "bd_check_status": (C.c_int32, [C.c_void_p, C.c_int32, C.c_void_p]),
    "bd_selftest_bounded_wait": (C.c_int32, [C.c_void_p, C.c_uint32, C.c_void_p]),
    "bd_last_error": (C.c_char_p, []),
    "bd_version": (C.c_int32, []),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libbd.so (once) and declare every exported function's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libbd.so not built at {path}: run `python -m block_causal_varlen_gb300.build`")
    lib = C.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class BDError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libbd status {status}: {msg}")
        self.status = status


def check(status: int) -> int:
    if status < 0:
        raise BDError(status, load().bd_last_error().decode())
    return status
