"""GB300 (sm_103a) dense GEMM: Python binding of the C ABI in include/dgemm.h.

The functions here only marshal arguments -- torch tensors to device pointers,
shapes to M/N/K, strings to enums, the current torch stream to a cudaStream_t --
and call libdgemm.so. Every step of the computation runs in the library's CUDA
kernels; there is no other path. PyTorch supplies device memory and streams.

    D = dgemm_bf16(A, B, D, b_layout="kn", C=None, alpha=1.0, beta=0.0, ...)
    D = dgemm_fp8_scaled(Aq, Bq, a_scale, b_scale, D, b_layout="nk", ...)
"""
from __future__ import annotations

import ctypes

from ._lib import (ACT, B_KN, B_NK, BF16, E4M3, F32, QUANT, DgemmError, Epilogue, Overrides, Plan, load,
                   lib_path)

__all__ = ["dgemm_bf16", "dgemm_fp8_scaled", "dgemm_fp8_rowquant_noalloc", "dgemm_workspace_size", "dgemm_plan",
           "dgemm_status_string", "dgemm_query_device_status", "set_overrides", "get_overrides", "overrides",
           "DgemmError", "load", "lib_path"]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    # plain ints: ctypes converts them for the c_void_p parameters
    return None if t is None else t.data_ptr()


def _on_device(t) -> bool:
    return t.is_cuda


def _require(t, name, shape=None, dtypes=None):
    """The C ABI takes dense row-major device buffers and trusts their sizes, so
    a tensor that is not one (a CPU tensor, a transposed or sliced view, a wrong
    shape or element type) is refused here instead of being read as one."""
    if t is None:
        return
    if not _on_device(t):
        raise ValueError(f"{name} must be a CUDA tensor (it is on {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major); pass {name}.contiguous()")
    if shape is not None and tuple(t.shape) != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")


def _require_common(M, N, C, beta, D, bias, out_row_scale, ws):
    torch = _torch()
    _require(D, "D", (M, N), (torch.float32, torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    if beta != 0.0:   # C is read only then (and may be None otherwise)
        _require(C, "C", (M, N), (torch.float32, torch.bfloat16))
    _require(bias, "bias", (N,), (torch.float32,))
    _require(out_row_scale, "out_row_scale", (M,), (torch.float32,))
    _require(ws, "ws")


def _require_fp8(Aq, Bq, a_scale, b_scale):
    torch = _torch()
    codes = (torch.float8_e4m3fn, torch.uint8)
    _require(Aq, "Aq", None, codes)
    _require(Bq, "Bq", None, codes)
    # the scale tables' shapes depend on k_group and b_block: the library checks those
    _require(a_scale, "a_scale", None, (torch.float32,))
    _require(b_scale, "b_scale", None, (torch.float32,))


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(A, B, b_layout):
    M, K = A.shape
    if b_layout == "kn":
        K2, N = B.shape
    elif b_layout == "nk":
        N, K2 = B.shape
    else:
        raise ValueError(f"b_layout must be 'kn' or 'nk', not {b_layout!r}")
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A has K={K}, B has K={K2}")
    return M, N, K


def _epilogue(bias, act, out_quant, out_row_scale):
    if bias is None and act == "none" and out_quant == "none":
        return None
    return Epilogue(None if bias is None else bias.data_ptr(), ACT[act], QUANT[out_quant],
                    None if out_row_scale is None else out_row_scale.data_ptr())


def _check(code, where):
    if code != 0:
        raise DgemmError(code, where)


def dgemm_bf16(A, B, D, *, b_layout="kn", C=None, alpha=1.0, beta=0.0, bias=None, act="none",
               out_quant="none", out_row_scale=None, ws=None, stream=None):
    """D = epilogue(alpha * A . op(B) + beta * C) with BF16 A, B and FP32 accumulation.

    A [M,K] bf16; B [K,N] ("kn") or [N,K] ("nk") bf16; C, D [M,N]; bias [N] fp32;
    act in none/relu/gelu/silu; out_quant "e4m3_row_amax" writes E4M3 codes to D
    and per-row scales to out_row_scale [M]. ws: workspace tensor (uint8) of at
    least dgemm_workspace_size(...) bytes. Returns D.
    """
    M, N, K = _dims(A, B, b_layout)
    torch = _torch()
    _require(A, "A", None, (torch.bfloat16,))
    _require(B, "B", None, (torch.bfloat16,))
    _require_common(M, N, C, beta, D, bias, out_row_scale, ws)
    epi = _epilogue(bias, act, out_quant, out_row_scale)
    code = load().dgemm_bf16(_ptr(A), _ptr(B), B_KN if b_layout == "kn" else B_NK, _ptr(C),
                             _dtype_code(C) if C is not None else F32, _ptr(D), _dtype_code(D),
                             M, N, K, float(alpha), float(beta),
                             ctypes.byref(epi) if epi is not None else None,
                             _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(code, "dgemm_bf16")
    return D


def dgemm_fp8_scaled(Aq, Bq, a_scale, b_scale, D, *, b_layout="nk", k_group=0, b_block=1, C=None, alpha=1.0,
                     beta=0.0, bias=None, act="none", out_quant="none", out_row_scale=None, ws=None,
                     stream=None):
    """D = epilogue(alpha * diag(a_scale) (Aq . op(Bq)) diag(b_scale) + beta * C), E4M3 inputs.

    Aq [M,K] and Bq [N,K] ("nk") or [K,N] ("kn") are float8_e4m3fn (or uint8 codes);
    a_scale [M] and b_scale [N] fp32. k_group = g > 0: per-K-group scales,
    a_scale [G,M] and b_scale [G,N]; with b_block=128 as well, one weight scale
    per 128 output channels, b_scale [G, ceil(N/128)] (dgemm_fp8_blockscaled).
    Other arguments as for dgemm_bf16. Returns D.
    """
    M, N, K = _dims(Aq, Bq, b_layout)
    _require_fp8(Aq, Bq, a_scale, b_scale)
    _require_common(M, N, C, beta, D, bias, out_row_scale, ws)
    epi = _epilogue(bias, act, out_quant, out_row_scale)
    if b_block != 1:
        if b_block != 128:
            raise ValueError("b_block must be 1 or 128")
        entry, name = load().dgemm_fp8_blockscaled, "dgemm_fp8_blockscaled"
    else:
        entry, name = load().dgemm_fp8_scaled, "dgemm_fp8_scaled"
    code = entry(_ptr(Aq), _ptr(Bq), B_KN if b_layout == "kn" else B_NK, _ptr(a_scale),
                                   _ptr(b_scale), int(k_group), _ptr(C),
                                   _dtype_code(C) if C is not None else F32, _ptr(D), _dtype_code(D),
                                   M, N, K, float(alpha), float(beta),
                                   ctypes.byref(epi) if epi is not None else None,
                                   _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                   _stream(stream))
    _check(code, name)
    return D


def dgemm_fp8_rowquant_noalloc(Aq, Bq, a_scale, b_scale, Dq, out_row_scale, *, b_layout="nk", C=None,
                               alpha=1.0, beta=0.0, bias=None, act="none", stream=None):
    """The requantising FP8 GEMM without a workspace, for callers that cannot
    allocate device memory at call time: its scratch is a static 32 MiB device
    array inside the library (M*N up to about 16.7 million; calls that overlap
    on the GPU race on it). Dq [M,N] uint8 E4M3 codes, out_row_scale [M] fp32."""
    M, N, K = _dims(Aq, Bq, b_layout)
    _require_fp8(Aq, Bq, a_scale, b_scale)
    _require_common(M, N, C, beta, Dq, bias, out_row_scale, None)
    epi = _epilogue(bias, act, "e4m3_row_amax", out_row_scale)
    code = load().dgemm_fp8_rowquant_noalloc(_ptr(Aq), _ptr(Bq), B_KN if b_layout == "kn" else B_NK,
                                             _ptr(a_scale), _ptr(b_scale), _ptr(C),
                                             _dtype_code(C) if C is not None else F32, _ptr(Dq),
                                             M, N, K, float(alpha), float(beta), ctypes.byref(epi),
                                             _stream(stream))
    _check(code, "dgemm_fp8_rowquant_noalloc")
    return Dq


def dgemm_workspace_size(is_fp8, M, N, K, b_layout="nk", *, out_quant="none", act="none") -> int:
    epi = Epilogue(None, ACT[act], QUANT[out_quant], None)
    return int(load().dgemm_workspace_size(int(bool(is_fp8)), M, N, K, B_KN if b_layout == "kn" else B_NK,
                                           ctypes.byref(epi)))


def dgemm_plan(is_fp8, M, N, K, b_layout="nk", d_dtype="bf16", *, out_quant="none", act="none",
               k_group=0, num_sms=152) -> dict:
    """The plan the library would use (host-only; no GPU needed). k_group as for
    dgemm_fp8_scaled."""
    epi = Epilogue(None, ACT[act], QUANT[out_quant], None)
    plan = Plan()
    d = {"f32": F32, "bf16": BF16, "e4m3": E4M3}[d_dtype]
    code = load().dgemm_plan(int(bool(is_fp8)), M, N, K, B_KN if b_layout == "kn" else B_NK, d,
                             ctypes.byref(epi), int(k_group), int(num_sms), ctypes.byref(plan))
    _check(code, "dgemm_plan")
    return {name: getattr(plan, name) for name, _ in Plan._fields_}


def dgemm_status_string(code: int) -> str:
    return load().dgemm_status_string(int(code)).decode()


def dgemm_query_device_status(ws=None, stream=None) -> int:
    """Synchronises the stream and returns (and clears) a status word: the one
    at the start of workspace ws (errors of the calls given that workspace), or
    with ws=None the per-device word (calls without a workspace)."""
    if ws is not None:
        _require(ws, "ws")
    return int(load().dgemm_query_device_status(_ptr(ws), _stream(stream)))


_OVR_FIELDS = [name for name, _ in Overrides._fields_]


def get_overrides() -> dict:
    """The planner overrides in force (see dgemm_set_overrides in dgemm.h)."""
    o = Overrides()
    _check(load().dgemm_get_overrides(ctypes.byref(o)), "dgemm_get_overrides")
    return {name: getattr(o, name) for name in _OVR_FIELDS}


def set_overrides(**fields) -> None:
    """Sets the planner overrides for later calls: the named fields, every other
    one at its default (the planner's choice). set_overrides() restores all."""
    o = Overrides()
    lib = load()
    lib.dgemm_overrides_init(ctypes.byref(o))
    for name, value in fields.items():
        if name not in _OVR_FIELDS:
            raise ValueError(f"unknown override {name!r}; known: {_OVR_FIELDS}")
        setattr(o, name, int(value))
    _check(lib.dgemm_set_overrides(ctypes.byref(o)), "dgemm_set_overrides")


class overrides:
    """Context manager: ``with overrides(tile_n=128): ...`` sets the named
    overrides and restores the previous ones on exit."""

    def __init__(self, **fields):
        self.fields = fields
        self.saved = None

    def __enter__(self):
        self.saved = get_overrides()
        merged = dict(self.saved)
        merged.update(self.fields)
        o = Overrides(**{k: int(v) for k, v in merged.items()})
        _check(load().dgemm_set_overrides(ctypes.byref(o)), "dgemm_set_overrides")
        return self

    def __exit__(self, *exc):
        o = Overrides(**{k: int(v) for k, v in self.saved.items()})
        _check(load().dgemm_set_overrides(ctypes.byref(o)), "dgemm_set_overrides")
        return False
