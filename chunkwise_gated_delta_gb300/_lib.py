"""ctypes view of the C ABI declared in include/kda.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_WORKSPACE = -3
KDA_ERR_CUDA = -4
KDA_ERR_TIMEOUT = -5
KDA_ERR_RANGE = -6

KDA_BF16 = 0
KDA_F32 = 1

KDA_GATE_NONE = 0
KDA_GATE_SCALAR = 1
KDA_GATE_CHANNEL = 2

KDA_FLAG_BETA_SCALES_V = 1

# Every symbol include/kda.h declares.
EXPORTS = ("kda_chunk_fwd_workspace", "kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_status_read",
           "kda_status_string", "kda_chunk_bwd_workspace", "kda_chunk_bwd", "dplr_chunk_fwd_workspace",
           "dplr_chunk_fwd", "dplr_factor_norms", "dplr_chunk_bwd_workspace", "dplr_chunk_bwd")

DPLR_FLAG_CLIP_GATE = 1


class KdaFwdArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("gate_kind", ctypes.c_int), ("g_dtype", ctypes.c_int),
        ("flags", ctypes.c_uint),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("ht", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("cu_seqlens", ctypes.c_void_p),
    ]


class KdaBwdArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("gate_kind", ctypes.c_int), ("g_dtype", ctypes.c_int),
        ("flags", ctypes.c_uint),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("grad_o", ctypes.c_void_p), ("grad_ht", ctypes.c_void_p),
        ("grad_q", ctypes.c_void_p), ("grad_k", ctypes.c_void_p), ("grad_v", ctypes.c_void_p),
        ("grad_g", ctypes.c_void_p), ("grad_beta", ctypes.c_void_p), ("grad_h0", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("cu_seqlens", ctypes.c_void_p),
    ]


class DplrFwdArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("gate_kind", ctypes.c_int), ("g_dtype", ctypes.c_int),
        ("flags", ctypes.c_uint),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("h0", ctypes.c_void_p), ("o", ctypes.c_void_p), ("ht", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("cu_seqlens", ctypes.c_void_p),
    ]


class DplrBwdArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("gate_kind", ctypes.c_int), ("g_dtype", ctypes.c_int),
        ("flags", ctypes.c_uint),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("h0", ctypes.c_void_p), ("grad_o", ctypes.c_void_p), ("grad_ht", ctypes.c_void_p),
        ("grad_q", ctypes.c_void_p), ("grad_k", ctypes.c_void_p), ("grad_v", ctypes.c_void_p),
        ("grad_a", ctypes.c_void_p), ("grad_b", ctypes.c_void_p), ("grad_g", ctypes.c_void_p),
        ("grad_h0", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("cu_seqlens", ctypes.c_void_p),
    ]


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


_lib = None


def load() -> ctypes.CDLL:
    """Load libkda.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        lib.kda_chunk_fwd_workspace.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_workspace.argtypes = [ctypes.POINTER(KdaFwdArgs)]
        lib.kda_chunk_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd.argtypes = [ctypes.POINTER(KdaFwdArgs), ctypes.c_void_p]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(KdaFwdArgs), ctypes.c_void_p]
        lib.kda_chunk_bwd_workspace.restype = ctypes.c_size_t
        lib.kda_chunk_bwd_workspace.argtypes = [ctypes.POINTER(KdaBwdArgs)]
        lib.kda_chunk_bwd.restype = ctypes.c_int
        lib.kda_chunk_bwd.argtypes = [ctypes.POINTER(KdaBwdArgs), ctypes.c_void_p]
        lib.dplr_chunk_fwd_workspace.restype = ctypes.c_size_t
        lib.dplr_chunk_fwd_workspace.argtypes = [ctypes.POINTER(DplrFwdArgs)]
        lib.dplr_chunk_fwd.restype = ctypes.c_int
        lib.dplr_chunk_fwd.argtypes = [ctypes.POINTER(DplrFwdArgs), ctypes.c_void_p]
        lib.dplr_factor_norms.restype = ctypes.c_int
        lib.dplr_factor_norms.argtypes = [ctypes.POINTER(DplrFwdArgs), ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]
        lib.dplr_chunk_bwd_workspace.restype = ctypes.c_size_t
        lib.dplr_chunk_bwd_workspace.argtypes = [ctypes.POINTER(DplrBwdArgs)]
        lib.dplr_chunk_bwd.restype = ctypes.c_int
        lib.dplr_chunk_bwd.argtypes = [ctypes.POINTER(DplrBwdArgs), ctypes.c_void_p]
        lib.kda_status_read.restype = ctypes.c_int
        lib.kda_status_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().kda_status_string(code).decode()
