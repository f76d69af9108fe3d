"""ctypes declarations of the C ABI in include/dgemm.h.

Loading fails loudly (ImportError-like RuntimeError) when libdgemm.so is not
built: there is no fallback path of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

OK = 0
STATUS = {
    0: "DGEMM_OK", 1: "DGEMM_ERR_INVALID_VALUE", 2: "DGEMM_ERR_NOT_SUPPORTED", 3: "DGEMM_ERR_MISALIGNED",
    4: "DGEMM_ERR_WORKSPACE_TOO_SMALL", 5: "DGEMM_ERR_CUDA", 6: "DGEMM_ERR_DEVICE_TIMEOUT", 7: "DGEMM_ERR_ARCH",
}
F32, BF16, E4M3 = 0, 1, 2
B_KN, B_NK = 0, 1
ACT = {"none": 0, "relu": 1, "gelu": 2, "silu": 3}
QUANT = {"none": 0, "e4m3_row_amax": 1}

# Every symbol the header declares, with (restype, argtypes).
_vp, _i64, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class Epilogue(ctypes.Structure):
    _fields_ = [("bias", _vp), ("act", _i32), ("out_quant", _i32), ("out_row_scale", _vp)]


class Overrides(ctypes.Structure):
    _fields_ = [("tile_n", _i32), ("cta_pair", _i32), ("tail_split", _i32), ("tail_halves", _i32),
                ("cluster_split", _i32), ("seg_first", _i32), ("raster_group", _i32), ("cooperative", _i32),
                ("kslices", _i32), ("wait_limit_ns", _i64), ("stall_after_loads", _i64)]


class Plan(ctypes.Structure):
    _fields_ = [("swap_ab", _i32), ("tile_m", _i32), ("tile_n", _i32), ("cta_group", _i32), ("stages", _i32),
                ("num_tiles", _i32), ("grid", _i32), ("cooperative", _i32), ("raster_group", _i32), ("k_groups", _i32),
                ("tail_tiles", _i32), ("tail_split", _i32), ("cluster_split", _i32),
                ("tail_halves", _i32), ("tail_units", _i32), ("k_slices", _i32),
                ("smem_bytes", _sz), ("workspace_bytes", _sz)]


SIGNATURES = {
    "dgemm_bf16": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp, _i32, _i64, _i64, _i64, _f32, _f32,
                          ctypes.POINTER(Epilogue), _vp, _sz, _vp]),
    "dgemm_fp8_scaled": (_i32, [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _i64, _i64, _i64, _f32,
                                _f32, ctypes.POINTER(Epilogue), _vp, _sz, _vp]),
    "dgemm_fp8_blockscaled": (_i32, [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _i64, _i64, _i64,
                                     _f32, _f32, ctypes.POINTER(Epilogue), _vp, _sz, _vp]),
    "dgemm_workspace_size": (_sz, [_i32, _i64, _i64, _i64, _i32, ctypes.POINTER(Epilogue)]),
    "dgemm_plan": (_i32, [_i32, _i64, _i64, _i64, _i32, _i32, ctypes.POINTER(Epilogue), _i32, _i32,
                          ctypes.POINTER(Plan)]),
    "dgemm_status_string": (ctypes.c_char_p, [_i32]),
    "dgemm_query_device_status": (_i32, [_vp, _vp]),
    "dgemm_overrides_init": (None, [ctypes.POINTER(Overrides)]),
    "dgemm_set_overrides": (_i32, [ctypes.POINTER(Overrides)]),
    "dgemm_get_overrides": (_i32, [ctypes.POINTER(Overrides)]),
    "dgemm_fp8_rowquant_noalloc": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _i64, _i64, _i64, _f32, _f32,
                                          ctypes.POINTER(Epilogue), _vp]),
}
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
WS_STATUS_BYTES = 256

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded libdgemm.so. Raises RuntimeError if it is not built (unless
    build_if_missing, which runs nvcc)."""
    global _lib
    lib = _lib
    if lib is not None:   # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libdgemm.so is not built ({path}); run "
                                   "`python -m dense_gemm_persistent_gb300.build`")
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (rt, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = rt
            fn.argtypes = args
        _lib = lib
        return lib


class DgemmError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        msg = load().dgemm_status_string(code).decode()
        super().__init__(f"{where}: {STATUS.get(code, code)} ({msg})")
        self.code = code
