"""ctypes declarations of libgdr's C ABI (include/gdr.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_BF16, GDR_F32, GDR_I32 = 1, 2, 3
PATHS = {"auto": 0, "fused": 1, "staged": 2, "fused_whole": 3}

STATUS = {
    0: "GDR_OK", -1: "GDR_ERR_NULL", -2: "GDR_ERR_DTYPE", -3: "GDR_ERR_SHAPE",
    -4: "GDR_ERR_STRIDE", -5: "GDR_ERR_DIM", -6: "GDR_ERR_HEADS", -7: "GDR_ERR_NSEQ",
    -8: "GDR_ERR_WORKSPACE", -9: "GDR_ERR_PATH", -10: "GDR_ERR_CUDA", -11: "GDR_ERR_ALIGN",
    -12: "GDR_ERR_DEVICE", -13: "GDR_ERR_SCRATCH_LIMIT", -14: "GDR_ERR_CKPT",
}

# Every function the header declares, with its ctypes signature.
_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                              ctypes.c_float, ctypes.c_size_t)


class GdrTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("strides", ctypes.POINTER(ctypes.c_int64))]


_T = ctypes.POINTER(GdrTensor)

SIGNATURES = {
    "gdr_chunk_fwd": (ctypes.c_int, [_T, _T, _T, _T, _T, _f32, _T, _vp, _i32, _T, _T, _vp]),
    "gdr_chunk_fwd_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32]),
    "gdr_chunk_fwd_ws": (ctypes.c_int, [_T, _T, _T, _T, _T, _f32, _T, _vp, _i32, _T, _T, _i32,
                                        _vp, _sz, _vp]),
    "gdr_chunk_fwd_ckpt": (ctypes.c_int, [_T, _T, _T, _T, _T, _f32, _T, _vp, _i32, _T, _T, _T,
                                          _vp, _i32, _i32, _vp, _sz, _vp]),
    "gdr_chunk_bwd": (ctypes.c_int, [_T, _T, _T, _T, _T, _f32, _T, _vp, _i32, _T, _T, _T, _T,
                                     _T, _T, _T, _T, _vp, _sz, _vp]),
    "gdr_chunk_bwd_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32]),
    "gdr_ckpt_count_bound": (_i64, [_i64, _i32]),
    "gdr_fused_split_pieces": (_i32, [_i64, _i32, _i32]),
    "gdr_split_plan": (_i32, [_i64, _i32, _vp]),
    "gdr_chunk_count_bound": (_i64, [_i64, _i32]),
    "gdr_stage_workspace_bytes": (_sz, [_i64, _i32]),
    "gdr_chunk_index": (ctypes.c_int, [_vp, _i32, _i64, _vp, _vp, _vp, _vp]),
    "gdr_chunk_prep": (ctypes.c_int, [_T, _T, _T, _T, _vp, _i32, _T, _T, _T, _vp, _sz, _vp]),
    "gdr_state_scan": (ctypes.c_int, [_T, _T, _T, _T, _T, _vp, _i32, _T, _T, _T, _vp, _sz, _vp]),
    "gdr_chunk_out": (ctypes.c_int, [_T, _T, _T, _T, _T, _f32, _vp, _i32, _T, _vp, _sz, _vp]),
    "gdr_chunk_out_noalloc": (ctypes.c_int, [_T, _T, _T, _T, _T, _f32, _vp, _i32, _T, _vp]),
    "gdr_debug_check_cu_seqlens": (ctypes.c_int, [_vp, _i32, _i64, _vp, _vp, _vp]),
    "gdr_device_status": (ctypes.c_int, [_vp]),
    "gdr_debug_wait_selftest": (ctypes.c_int, [ctypes.c_uint32, _vp]),
    "gdr_clear_device_status": (ctypes.c_int, []),
    "gdr_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gdr_version": (ctypes.c_int, []),
}

_lock = threading.Lock()
_lib = None


def lib():
    """Load libgdr.so (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libgdr.so is missing at {LIB_PATH}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` or "
                    "`python -m chunked_gated_delta_gdr_gb300.build`")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = lib().gdr_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


def check(status: int, where: str) -> None:
    if status != 0:
        raise GdrError(status, where)
