"""ctypes declarations of the C-ABI in include/spec_verify.h.

The functions keep the C names (``sv_verify_chain`` ...).  Loading fails
loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# SPEC_VERIFY_LIBRARY selects another build of the same C-ABI, e.g. the
# bounds-checked debug build libspec_verify_debug.so (its index checks
# report through sv_debug_flags).
LIB_PATH = os.environ.get("SPEC_VERIFY_LIBRARY") or os.path.join(_HERE, "libspec_verify.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libspec_verify_debug.so")

SV_OK = 0
SV_ERR_INVALID_ARGUMENT = 1
SV_ERR_UNSUPPORTED = 2
SV_ERR_CUDA = 3
SV_ERR_WORKSPACE_TOO_SMALL = 4

SV_F32 = 0
SV_BF16 = 1

SV_ROW_BAD_DRAFT_ID = 1
SV_ROW_BAD_PARENT = 2
SV_ROW_DEPTH_EXCEEDED = 4
SV_ROW_BAD_TOKEN = 8
SV_ROW_EMPTY = 16
SV_ROW_RESAMPLE_FALLBACK = 32

SV_MAX_GAMMA = 64
SV_MAX_VOCAB = 16777216
SV_MAX_TREE_NODES = 1024
SV_MAX_TREE_DEPTH = 64

SV_DEBUG_INDEX = 1


class ChainDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("gamma", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("draft_vocab", ctypes.c_int32), ("target_dtype", ctypes.c_int32),
                ("draft_dtype", ctypes.c_int32), ("temperature", ctypes.c_float),
                ("top_p", ctypes.c_float), ("target_row_stride", ctypes.c_int64),
                ("draft_row_stride", ctypes.c_int64)]


class TreeDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("nodes", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("max_depth", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("row_stride", ctypes.c_int64)]


class SampleDesc(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("vocab", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
                ("row_stride", ctypes.c_int64)]


class TreeSampleDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("nodes", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("max_depth", ctypes.c_int32), ("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("target_row_stride", ctypes.c_int64),
                ("draft_row_stride", ctypes.c_int64)]


class TopkDesc(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("vocab", ctypes.c_int32), ("k", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("row_stride", ctypes.c_int64)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

SIGNATURES = {
    "sv_chain_workspace_size": (_SZ, [ctypes.POINTER(ChainDesc)]),
    "sv_verify_chain": (_I32, [ctypes.POINTER(ChainDesc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, _P, _SZ, _P]),
    "sv_verify_chain_static": (_I32, [ctypes.POINTER(ChainDesc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, _P]),
    "sv_static_scratch_bytes": (_SZ, []),
    "sv_tree_workspace_size": (_SZ, [ctypes.POINTER(TreeDesc)]),
    "sv_verify_tree": (_I32, [ctypes.POINTER(TreeDesc), _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sv_tree_path_workspace_size": (_SZ, [ctypes.POINTER(TreeDesc)]),
    "sv_topk": (_I32, [ctypes.POINTER(TopkDesc), _P, _P, _P, _P]),
    "sv_tree_sample_workspace_size": (_SZ, [ctypes.POINTER(TreeSampleDesc)]),
    "sv_verify_tree_sample": (_I32, [ctypes.POINTER(TreeSampleDesc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                     _P, _SZ, _P]),
    "sv_verify_tree_path": (_I32, [ctypes.POINTER(TreeDesc), _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sv_d2t_scatter": (_I32, [_P, _I64, _P, _P, _I32, _I32, _I32, _I32, _F, _P, _I64, _P]),
    "sv_build_t2d": (_I32, [_P, _I32, _I32, _P, _P, _P]),
    "sv_sample_workspace_size": (_SZ, [ctypes.POINTER(SampleDesc)]),
    "sv_sample": (_I32, [ctypes.POINTER(SampleDesc), _P, _P, _P, _P, _P, _SZ, _P]),
    "sv_softmax_topp": (_I32, [ctypes.POINTER(SampleDesc), _P, _P, _I64, _P, _SZ, _P]),
    "sv_status_string": (ctypes.c_char_p, [_I32]),
    "sv_version": (_I32, []),
    "sv_set_phase_events": (None, [_P, _I32]),
    "sv_launch_count": (ctypes.c_uint64, []),
    "sv_debug_flags": (ctypes.c_uint32, [_I32]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -m draft_token_verification_sv_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class SVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().sv_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def check(status: int, where: str) -> None:
    if status != SV_OK:
        raise SVError(status, where)
