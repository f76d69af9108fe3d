"""The per-workload tolerances, written out.

  1  BF16, FP32 output:  max|err| <= 1e-4 * sqrt(K) * max|ref|
  2,4 BF16 output:      |gpu - bf16(ref)| <= ulp_bf16(bf16(ref)) + 1e-6, with
                         ulp = 2^(floor(log2|v|) - 7): one BF16 unit in the last place
                         of the correctly rounded reference (a flip of a rounding
                         tie between FP32 and exact accumulation is one ulp).
  3  FP8 -> BF16:        relative Frobenius error <= 2e-3.
  5  E4M3 requant:       dequantised outputs dec(q) * s against the exact y:
                         >= 99.9% within 1 E4M3 ulp and all within 2, where
                         ulp(y) = s_ref * 2^(max(floor(log2(|y| / s_ref)), -6) - 3)
                         (the subnormal spacing below 2^-6); and s within 1e-5
                         relative of max|y| / 448.
"""
from __future__ import annotations

import numpy as np

import oracle


def c1_ok(gpu: np.ndarray, ref: np.ndarray, K: int):
    err = np.abs(gpu.astype(np.float64) - ref).max() if ref.size else 0.0
    bound = 1e-4 * np.sqrt(max(K, 1)) * (np.abs(ref).max() if ref.size else 0.0)
    return err <= bound, f"max|err| {err:.3e} bound {bound:.3e}"


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a > 0, np.exp2(e - 7), np.exp2(-133.0))


def bf16_ulp_ok(gpu: np.ndarray, ref: np.ndarray):
    r = oracle.round_bf16(ref)
    err = np.abs(gpu.astype(np.float64) - r)
    bound = bf16_ulp(r) + 1e-6
    bad = int(np.count_nonzero(err > bound))
    strict = int(np.count_nonzero(np.abs(gpu - ref) > np.abs(ref) * 2.0 ** -8 + 1e-6))
    return bad == 0, f"{bad} of {ref.size} beyond 1 ulp (strict 2^-8-relative reading: {strict})"


def frob_ok(gpu: np.ndarray, ref: np.ndarray, tol: float = 2e-3):
    num = np.linalg.norm((gpu.astype(np.float64) - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    rel = num / den if den > 0 else num
    return rel <= tol, f"relative Frobenius error {rel:.3e} (tol {tol:g})"


def e4m3_spacing(y: np.ndarray, s_ref: np.ndarray) -> np.ndarray:
    x = np.abs(y) / s_ref[:, None]
    e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    e = np.where(x > 0, np.maximum(e, -6), -6)
    return s_ref[:, None] * np.exp2(e - 3)


def requant_ok(q: np.ndarray, s_gpu: np.ndarray, y: np.ndarray):
    """q: E4M3 codes from the GPU, s_gpu: its row scales, y: exact pre-quant values."""
    _, s_ref = oracle.requant_rows(y)
    dq = oracle.decode_e4m3(q) * s_gpu.astype(np.float64)[:, None]
    ulp = e4m3_spacing(y, s_ref)
    err = np.abs(dq - y) / ulp
    frac1 = float(np.mean(err <= 1.0)) if err.size else 1.0
    worst = float(err.max()) if err.size else 0.0
    srel = float(np.max(np.abs(s_gpu.astype(np.float64) - s_ref) / s_ref)) if s_ref.size else 0.0
    ok = frac1 >= 0.999 and worst <= 2.0 and srel <= 1e-5
    return ok, f"within 1 ulp {frac1:.5f}, worst {worst:.3f} ulp, scale rel err {srel:.2e}"
