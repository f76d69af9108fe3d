"""The oracle: a plain float64 CPU restatement of the dense GEMM hot path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The GPU library never imports it and shares no code with it; the two
meet only through the seeded inputs of ``workloads.py``.

The arithmetic lives in ``dgemm_oracle.c`` (plain loops, float64). This module
compiles it with gcc on first use and wraps each C function for numpy arrays.

Sources (cited by page title and section):
  [W1] DeepGEMM write-up, czchanglian.com/news/51329 -- C = alpha*A*B + beta*C
       (§1.1); fused bias + activation (§6.1); per-token output quantisation
       (§6.2).
  [W3] "DeepGEMM: FP8 Tensor Core GEMM", bjdmk.com.cn/news/6078902 -- E4M3
       (§1.2); per-token x per-channel scales applied to the accumulated result
       (§1.2, §3.2).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, identities, closed forms, library special cases); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

F64, F32, BF16, E4M3 = 0, 1, 2, 3
ACT = {"none": 0, "relu": 1, "gelu": 2, "silu": 3}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d, i64, i32, vp = ctypes.c_double, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.orc_bf16_to_f64.restype = d
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_e4m3_to_f64.restype = d
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_f64_to_e4m3.restype = ctypes.c_uint8
            lib.orc_f64_to_e4m3.argtypes = [d]
            lib.orc_round_bf16.restype = d
            lib.orc_round_bf16.argtypes = [d]
            lib.orc_silu.restype = d
            lib.orc_silu.argtypes = [d]
            lib.orc_gelu.restype = d
            lib.orc_gelu.argtypes = [d]
            lib.orc_decode.restype = i32
            lib.orc_decode.argtypes = [vp, i32, i64, vp]
            lib.orc_dequant.restype = i32
            lib.orc_dequant.argtypes = [vp, i32, i64, i64, vp, i32, vp]
            lib.orc_dequant_grouped.restype = i32
            lib.orc_dequant_grouped.argtypes = [vp, i64, i64, vp, i32, i64, vp]
            lib.orc_gemm.restype = i32
            lib.orc_gemm.argtypes = [vp, vp, i32, vp, d, d, i64, i64, i64, i64, i64, vp, i32]
            lib.orc_epilogue.restype = i32
            lib.orc_epilogue.argtypes = [vp, i64, i64, vp, i32]
            lib.orc_requant_rows.restype = i32
            lib.orc_requant_rows.argtypes = [vp, i64, i64, vp, vp]
            for name, rt in (("orc_encode_e4m3_array", None), ("orc_round_bf16_array", None),
                             ("orc_encode_bf16_array", None)):
                getattr(lib, name).restype = rt
                getattr(lib, name).argtypes = [vp, i64, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _threads(nthreads: int | None) -> int:
    if nthreads:
        return int(nthreads)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---- codecs -----------------------------------------------------------------

def decode(raw: np.ndarray, kind: int) -> np.ndarray:
    """Exact widening of raw F32 / BF16-bits (uint16) / E4M3-codes (uint8) to float64."""
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.shape, dtype=np.float64)
    if _load().orc_decode(_ptr(raw), kind, raw.size, _ptr(out)) != 0:
        raise ValueError("unknown element type")
    return out


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return decode(np.asarray(codes, dtype=np.uint8), E4M3)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    return decode(np.asarray(bits, dtype=np.uint16), BF16)


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to E4M3 (nearest, ties to even, saturating at +-448); returns codes."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().orc_encode_e4m3_array(_ptr(x), x.size, _ptr(q))
    return q


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest BF16 value (ties to even), as float64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.float64)
    _load().orc_round_bf16_array(_ptr(x), x.size, _ptr(y))
    return y


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) of round_bf16(x)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().orc_encode_bf16_array(_ptr(x), x.size, _ptr(y))
    return y


def silu(y: float) -> float:
    return _load().orc_silu(float(y))


def gelu(y: float) -> float:
    return _load().orc_gelu(float(y))


# ---- the GEMM ---------------------------------------------------------------

def gemm(A: np.ndarray, B: np.ndarray, b_layout: str = "kn", C: np.ndarray | None = None,
         alpha: float = 1.0, beta: float = 0.0, rows=None, nthreads: int | None = None) -> np.ndarray:
    """alpha * A @ op(B) + beta * C in float64 ([W1] §1.1).

    A is M x K; B is K x N (``b_layout="kn"``) or N x K (``"nk"``); C is M x N and
    is read only when beta != 0. ``rows`` = (row0, row1) restricts the result to
    those rows of D (the full-size parity checks sample rows this way).
    """
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    if b_layout == "kn":
        K2, N = B.shape
    elif b_layout == "nk":
        N, K2 = B.shape
    else:
        raise ValueError(b_layout)
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        C = np.ascontiguousarray(C, dtype=np.float64)
        if C.shape != (M, N):
            raise ValueError("C shape")
    else:
        C = None
    r0, r1 = (0, M) if rows is None else rows
    out = np.empty((r1 - r0, N), dtype=np.float64)
    rc = _load().orc_gemm(_ptr(A), _ptr(B), 1 if b_layout == "nk" else 0, _ptr(C),
                          float(alpha), float(beta), M, N, K, r0, r1, _ptr(out), _threads(nthreads))
    if rc != 0:
        raise ValueError("bad row range")
    return out


def dequant(codes: np.ndarray, scale: np.ndarray, axis: int) -> np.ndarray:
    """Decode E4M3 codes and multiply by a float32 scale per row (axis 0) or column (axis 1)
    ([W3] §3.2)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    rows, cols = codes.shape
    if scale.shape != ((rows,) if axis == 0 else (cols,)):
        raise ValueError("scale shape")
    out = np.empty((rows, cols), dtype=np.float64)
    _load().orc_dequant(_ptr(codes), E4M3, rows, cols, _ptr(scale), axis, _ptr(out))
    return out


def dequant_grouped(codes: np.ndarray, scale: np.ndarray, k_axis: int, group: int) -> np.ndarray:
    """Decode E4M3 codes and multiply each by the scale of its K group ([W3] §3.2,
    per-group granularity). ``k_axis`` is the index of ``codes`` that runs along K;
    ``scale`` is [ceil(K / group), L], L the extent of the other index."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    rows, cols = codes.shape
    K, L = (cols, rows) if k_axis == 1 else (rows, cols)
    if scale.shape != (-(-K // group), L):
        raise ValueError("scale shape")
    out = np.empty((rows, cols), dtype=np.float64)
    if _load().orc_dequant_grouped(_ptr(codes), rows, cols, _ptr(scale), int(k_axis), int(group), _ptr(out)) != 0:
        raise ValueError("bad group or axis")
    return out


def epilogue(X: np.ndarray, bias: np.ndarray | None = None, act: str = "none") -> np.ndarray:
    """y = x + bias[n], then the activation ([W1] §6.1). Returns a new array."""
    X = np.array(X, dtype=np.float64, order="C", copy=True)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rows, N = X.shape
    if b is not None and b.shape != (N,):
        raise ValueError("bias shape")
    if _load().orc_epilogue(_ptr(X), rows, N, _ptr(b), ACT[act]) != 0:
        raise ValueError("activation")
    return X


def requant_rows(Z: np.ndarray):
    """Per-row E4M3 quantisation: (codes, scales) with s = amax/448 ([W1] §6.2)."""
    Z = np.ascontiguousarray(Z, dtype=np.float64)
    rows, N = Z.shape
    q = np.empty((rows, N), dtype=np.uint8)
    s = np.empty(rows, dtype=np.float64)
    _load().orc_requant_rows(_ptr(Z), rows, N, _ptr(q), _ptr(s))
    return q, s


# ---- whole-path references for the five workloads ------------------------------

def _row_select(X, rows):
    """Rows of X picked by a (row0, row1) range or an index array (None: all)."""
    if X is None or rows is None:
        return X
    X = np.asarray(X)
    if isinstance(rows, tuple):
        return X[rows[0]:rows[1]]
    return X[np.asarray(rows, dtype=np.int64)]


def _rows_index(rows, n):
    """The row indices a (row0, row1) range or an index array selects (None: all n)."""
    if rows is None:
        return np.arange(n)
    if isinstance(rows, tuple):
        return np.arange(rows[0], rows[1])
    return np.asarray(rows, dtype=np.int64)


def bf16_gemm_ref(A_bits, B_bits, b_layout, C=None, alpha=1.0, beta=0.0, rows=None,
                  nthreads=None) -> np.ndarray:
    """Reference for the BF16 form: inputs are the raw BF16 bit patterns (uint16) the
    GPU receives; C is float32 or BF16 bits. ``rows`` ((row0, row1) or an index
    array) restricts the result to those rows of D: the same GEMM on those rows of A."""
    A = decode_bf16(_row_select(A_bits, rows))
    B = decode_bf16(B_bits)
    Cd = None
    if beta != 0.0:
        Cs = _row_select(C, rows)
        Cd = decode_bf16(Cs) if Cs.dtype == np.uint16 else decode(np.asarray(Cs, np.float32), F32)
    return gemm(A, B, b_layout, Cd, alpha, beta, None, nthreads)


def block_scales_per_channel(b_scale: np.ndarray, N: int, block: int) -> np.ndarray:
    """A weight-block scale table [G, ceil(N / block)] written out per output
    channel, [G, N]: channel n takes the scale of block n // block ([W3] §3.2,
    one scale per group of weights)."""
    b_scale = np.asarray(b_scale, dtype=np.float32)
    if b_scale.ndim != 2 or b_scale.shape[1] != -(-N // block):
        raise ValueError("block scale shape")
    return np.ascontiguousarray(b_scale[:, np.arange(N) // block])


def fp8_gemm_ref(Aq, Bq, b_layout, a_scale, b_scale, C=None, alpha=1.0, beta=0.0,
                 bias=None, act="none", rows=None, nthreads=None, k_group=0, b_block=1) -> np.ndarray:
    """Reference for the FP8 form: D = alpha * diag(sa) (Aq Bq) diag(sb) + beta*C,
    then + bias and the activation, on the dequantised E4M3 values ([W3] §3.2).
    With k_group > 0 the scales are per K group: a_scale [G, M] and b_scale
    [G, N] (G = ceil(K / k_group)), and each code is dequantised with its own
    group's scale before the plain GEMM. b_block = 128 (with k_group > 0): one
    weight scale per block of 128 output channels, b_scale [G, ceil(N / 128)]."""
    if b_block != 1 and not k_group:
        raise ValueError("weight blocks need k_group")
    if k_group:
        if np.shape(a_scale) != (-(-Aq.shape[1] // k_group), Aq.shape[0]):
            raise ValueError("a_scale shape")
        Ad = dequant_grouped(_row_select(Aq, rows), np.asarray(a_scale)[:, _rows_index(rows, Aq.shape[0])],
                             1, k_group)
        N = Bq.shape[0] if b_layout == "nk" else Bq.shape[1]
        if b_block != 1:
            b_scale = block_scales_per_channel(b_scale, N, b_block)
        Bd = dequant_grouped(Bq, b_scale, 1 if b_layout == "nk" else 0, k_group)
    else:
        Ad = dequant(_row_select(Aq, rows), _row_select(a_scale, rows), 0)
        Bd = dequant(Bq, b_scale, 0 if b_layout == "nk" else 1)
    Cs = _row_select(C, rows)
    Cd = None
    if beta != 0.0:
        Cd = decode_bf16(Cs) if Cs.dtype == np.uint16 else decode(np.asarray(Cs, np.float32), F32)
    D = gemm(Ad, Bd, b_layout, Cd, alpha, beta, None, nthreads)
    if bias is not None or act != "none":
        D = epilogue(D, bias, act)
    return D
