"""ctypes bindings of liboracle.so (test infrastructure only)."""
import ctypes
import threading

import numpy as np

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def lib():
    """Loads (building first if needed) the oracle library."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            L.or_rne_bf16.argtypes = [ctypes.c_float]
            L.or_rne_bf16.restype = ctypes.c_uint16
            L.or_rne_f16.argtypes = [ctypes.c_float]
            L.or_rne_f16.restype = ctypes.c_uint16
            L.or_bf16_f32.argtypes = [ctypes.c_uint16]
            L.or_bf16_f32.restype = ctypes.c_float
            L.or_f16_f32.argtypes = [ctypes.c_uint16]
            L.or_f16_f32.restype = ctypes.c_float
            L.or_cvt_f32_bf16.argtypes = [_f32p, _u16p, _i64]
            L.or_cvt_f32_f16.argtypes = [_f32p, _u16p, _i64]
            L.or_cvt_f16_f32.argtypes = [_u16p, _f32p, _i64]
            L.or_leaf.argtypes = [_vp, _i64, _vp, _i64, _i64, ctypes.c_int, ctypes.c_int]
            L.or_leaf.restype = ctypes.c_float
            L.or_tree_from_leaves.argtypes = [_f32p, _i64]
            L.or_tree_from_leaves.restype = ctypes.c_uint16
            L.or_tree_node.argtypes = [_f32p, _i64, _i64]
            L.or_tree_node.restype = ctypes.c_float
            L.or_tree_gemm.argtypes = [_vp, _i64, _i64, _vp, _i64, _i64,
                                       _i64, _i64, _i64, _vp, _i64, _i64, _vp,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int]
            L.or_tree_replay.argtypes = [_f32p, _i64, _i64, _u16p]
            L.or_silu_tables.argtypes = [_u16p, _f32p]
            L.or_silu_mul.argtypes = [_u16p, _u16p, _i64, _u16p]
            L.or_silu_bwd.argtypes = [_u16p, _u16p, _u16p, _i64, _vp, _vp, _vp]
            L.or_add_bf16.argtypes = [_u16p, _u16p, _i64, _u16p]
            L.or_rank_tree.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _i64,
                                       ctypes.c_int, _vp]
            L.or_rank_tree.restype = ctypes.c_int
            _LIB = L
    return _LIB
