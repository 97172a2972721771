"""ctypes mirror of include/ep.h and the loader of libep_gb300.so.

Argument marshalling only. There is no fallback: if the library is missing or
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_CAPACITY = 2
EP_ERR_ALIGNMENT = 3
EP_ERR_WORKSPACE = 4
EP_ERR_CAPTURE_HOST_SYNC = 5
EP_ERR_CUDA = 6
EP_ERR_NO_LAYOUT = 7
EP_ERR_HOST_ALLOC = 8

EP_BF16 = 0
EP_F32 = 1

EP_PERMUTE_DEFAULT = 0
EP_PERMUTE_VEC = 1
EP_PERMUTE_BULK = 2

EP_LAYOUT_STRIDED = 0
EP_LAYOUT_PACKED = 1

EP_DEVERR_BAD_ID = 0x1
EP_DEVERR_ROW_OOB = 0x2
EP_DEVERR_TIMEOUT = 0x4
EP_DEVERR_DEBUG_UNWRITTEN = 0x8   # EP_DEBUG=1 only
EP_DEVERR_DEBUG_STRAY = 0x10      # EP_DEBUG=1 only

EP_NOALLOC_SCRATCH_BYTES = 4 << 20

EP_PATTERN_READ = 0
EP_PATTERN_WRITE = 1
EP_PATTERN_COPY = 2
EP_PATTERN_FANOUT = 3
EP_PATTERN_GATHER = 4


class EpConfig(C.Structure):
    _fields_ = [
        ("num_max_tokens_per_rank", C.c_int64),
        ("hidden", C.c_int64),
        ("num_experts", C.c_int32),
        ("num_ranks", C.c_int32),
        ("topk", C.c_int32),
        ("dtype", C.c_int32),
        ("num_sms", C.c_int32),
        ("permute_impl", C.c_int32),
        ("layout_mode", C.c_int32),
    ]


class EpLayout(C.Structure):
    _fields_ = [
        ("tokens_per_expert", C.c_void_p),
        ("expert_offset", C.c_void_p),
        ("rows_per_rank", C.c_void_p),
        ("rank_prefix", C.c_void_p),
        ("tokens_in_rank", C.c_void_p),
        ("pos", C.c_void_p),
        ("num_tokens", C.c_int64),
        ("padded_tokens", C.c_int64),
        ("rank_stride", C.c_int64),
        ("packed", C.c_int32),
    ]


class EpDispatchOut(C.Structure):
    _fields_ = [
        ("recv_x", C.c_void_p),
        ("recv_scores", C.c_void_p),
        ("recv_src", C.c_void_p),
        ("layout", EpLayout),
    ]


class EpDedupOut(C.Structure):
    _fields_ = [
        ("recv_x", C.c_void_p),
        ("recv_tok_src", C.c_void_p),
        ("recv_topk_idx", C.c_void_p),
        ("recv_topk_w", C.c_void_p),
        ("tok_pos", C.c_void_p),
        ("rows_per_rank_stride", C.c_int64),
        ("layout", EpLayout),
    ]


class EpBufferInfo(C.Structure):
    _fields_ = [
        ("workspace_bytes", C.c_int64),
        ("max_rank_stride", C.c_int64),
        ("kernel_launches", C.c_int64),
        ("device", C.c_int32),
        ("num_sms", C.c_int32),
        ("permute_impl", C.c_int32),
        ("permute_grid", C.c_int32),
        ("combine_grid", C.c_int32),
        ("bulk_stages", C.c_int32),
        ("gemm_kernel", C.c_int32),
        ("gemm_grid", C.c_int32),
    ]


# name -> (restype, argtypes), in the order of include/ep.h
SIGNATURES = {
    "ep_buffer_required_bytes": (C.c_size_t, [C.POINTER(EpConfig)]),
    "ep_buffer_init": (C.c_int, [C.POINTER(EpConfig), C.c_void_p, C.c_size_t,
                                 C.POINTER(C.c_void_p)]),
    "ep_buffer_destroy": (C.c_int, [C.c_void_p]),
    "ep_dispatch_layout": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                     C.POINTER(EpLayout), C.c_void_p]),
    "ep_dispatch": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                              C.c_int64, C.c_void_p, C.POINTER(EpDispatchOut)]),
    "ep_dispatch_permute": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.POINTER(EpDispatchOut)]),
    "ep_combine": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p,
                             C.c_int32, C.c_void_p]),
    "ep_combine_backward": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "ep_dispatch_backward": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                       C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "ep_dispatch_dedup": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                    C.c_int64, C.c_void_p, C.POINTER(EpDedupOut)]),
    "ep_dedup_expand": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "ep_expert_gemm": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                 C.c_void_p, C.c_void_p]),
    "ep_get_device_error": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(C.c_uint32)]),
    "ep_buffer_query": (C.c_int, [C.c_void_p, C.POINTER(EpBufferInfo)]),
    "ep_dispatch_layout_noalloc": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_int32,
                                             C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                             C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                             C.c_void_p, C.c_void_p]),
    "ep_dispatch_layout_noalloc_scratch_bytes": (C.c_size_t, [C.c_int64, C.c_int32, C.c_int32,
                                                           C.c_int32]),
    "ep_pad_tokens": (C.c_int64, [C.c_int64]),
    "ep_derive_max_tokens_pretrain": (C.c_int64, [C.c_int64, C.c_int64, C.c_int64, C.c_int64]),
    "ep_derive_max_tokens_inference": (C.c_int64, [C.c_int64, C.c_int64, C.c_int64]),
    "ep_validate_max_tokens": (C.c_int, [C.c_int64, C.c_int64]),
    "ep_pattern_probe": (C.c_int, [C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                   C.c_int32, C.c_void_p]),
    "ep_status_string": (C.c_char_p, [C.c_int]),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m combine_topk_ids_expert_gb300.build` (needs nvcc). "
                "There is no fallback implementation.")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class EpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().ep_status_string(status).decode()
        super().__init__(f"{what}: {msg} (status {status})")


def check(status: int, what: str) -> None:
    if status != EP_OK:
        raise EpError(status, what)
