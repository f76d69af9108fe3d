"""Seeded synthetic inputs for the five GEMM workloads.

This module is the one place both sides of a parity check get their inputs
from: the GPU library (through the tests, the smoke check and the benchmark)
and the oracle. It draws random numbers and converts them to the storage types
the GEMM consumes (BF16, and E4M3 codes with their FP32 scales); it holds none
of the GEMM's own arithmetic. The E4M3 input quantisation (one FP32 scale per
row / per output channel = amax / 448) is the caller-side preparation that the
workloads specify, done here with torch's own float8 cast.

Every workload is generated from ``numpy.random.default_rng(seed)`` with
``seed = 1000 + workload number`` unless a seed is given; shapes can be shrunk
for the small parity cases, keeping the same value recipe.

  1  BF16 512^3, A KxN-layout B, alpha 1.5, beta 0.5, FP32 C0 -> FP32 D
  2  BF16 4096^3, entries N(0,1)/sqrt(K) -> BF16 D
  3  FP8 E4M3 4096 x 11008 x 4096 (FFN projection) -> BF16 D
  4  decode-shaped BF16 16 x 18432 x 7168, weights stored N x K -> BF16 D
  5  FP8 E4M3 8192^3 + bias -> SiLU -> per-row E4M3 requantisation
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclass
class Workload:
    number: int
    name: str
    form: str                    # "bf16" | "fp8"
    M: int
    N: int
    K: int
    b_layout: str                # "kn": B is K x N row-major; "nk": B is N x K row-major
    alpha: float = 1.0
    beta: float = 0.0
    A: torch.Tensor = None       # bf16 [M,K] or float8_e4m3fn [M,K]
    B: torch.Tensor = None       # [K,N] or [N,K], same dtype as A
    C: Optional[torch.Tensor] = None        # float32 [M,N], read when beta != 0
    a_scale: Optional[torch.Tensor] = None  # float32 [M] (per token)
    b_scale: Optional[torch.Tensor] = None  # float32 [N] (per output channel)
    bias: Optional[torch.Tensor] = None     # float32 [N]
    act: str = "none"
    d_dtype: str = "bf16"        # "f32" | "bf16" | "e4m3"
    out_quant: str = "none"      # "none" | "e4m3_row_amax"
    k_group: int = 0             # FP8: 0 = one scale per row / channel; g > 0 = one per K group of g
    b_block: int = 1             # FP8 with k_group: output channels per weight scale (1 or 128)
    seed: int = 0
    extras: dict = field(default_factory=dict)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def tensors(self):
        return {k: getattr(self, k) for k in ("A", "B", "C", "a_scale", "b_scale", "bias")
                if getattr(self, k) is not None}

    def to(self, device) -> "Workload":
        """A copy whose tensors live on ``device``."""
        w = Workload(**{**self.__dict__})
        for k, t in self.tensors().items():
            setattr(w, k, t.to(device))
        return w


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def quantize_e4m3_rows(X: np.ndarray):
    """E4M3 codes of X with one FP32 scale per row, s = amax_row / 448."""
    X32 = np.ascontiguousarray(X, dtype=np.float32)
    amax = np.abs(X32).max(axis=1, initial=0.0)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    s[s == 0] = 1.0
    q = torch.from_numpy(X32 / s[:, None]).to(torch.float8_e4m3fn)
    return q, torch.from_numpy(s)


def quantize_e4m3_groups(X: np.ndarray, group: int):
    """E4M3 codes of X [rows, K] with one FP32 scale per (row, K group of
    ``group`` columns), s = amax / 448 over that slice. Scales come back
    group-major, [ceil(K / group), rows]."""
    X32 = np.ascontiguousarray(X, dtype=np.float32)
    rows, K = X32.shape
    G = -(-K // group)
    s = np.empty((G, rows), dtype=np.float32)
    Y = np.empty_like(X32)
    for j in range(G):
        sl = X32[:, j * group:(j + 1) * group]
        sj = (np.abs(sl).max(axis=1, initial=0.0) / np.float32(E4M3_MAX)).astype(np.float32)
        sj[sj == 0] = 1.0
        s[j] = sj
        Y[:, j * group:(j + 1) * group] = sl / sj[:, None]
    return torch.from_numpy(Y).to(torch.float8_e4m3fn), torch.from_numpy(s)


def quantize_e4m3_blocks(W: np.ndarray, group: int, block: int):
    """E4M3 codes of W [N, K] with one FP32 scale per (block of ``block`` rows,
    K group of ``group`` columns), s = amax / 448 over that block. Scales come
    back group-major, [ceil(K / group), ceil(N / block)]."""
    W32 = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W32.shape
    G, NB = -(-K // group), -(-N // block)
    s = np.empty((G, NB), dtype=np.float32)
    Y = np.empty_like(W32)
    for j in range(G):
        for b in range(NB):
            blk = W32[b * block:(b + 1) * block, j * group:(j + 1) * group]
            sb = np.float32(np.abs(blk).max(initial=0.0) / np.float32(E4M3_MAX))
            sb = np.float32(1.0) if sb == 0 else sb
            s[j, b] = sb
            Y[b * block:(b + 1) * block, j * group:(j + 1) * group] = blk / sb
    return torch.from_numpy(Y).to(torch.float8_e4m3fn), torch.from_numpy(s)


def _log_uniform_rows(rng, M, lo=0.1, hi=10.0):
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=(M, 1))).astype(np.float32)


def config1(M=512, N=512, K=512, seed=None) -> Workload:
    seed = 1001 if seed is None else seed
    rng = np.random.default_rng(seed)
    A = _bf16(rng.uniform(-1, 1, size=(M, K)))
    B = _bf16(rng.uniform(-1, 1, size=(K, N)))
    C = torch.from_numpy(rng.uniform(-1, 1, size=(M, N)).astype(np.float32))
    return Workload(1, f"bf16 {M}x{N}x{K} alpha1.5 beta0.5 f32-out", "bf16", M, N, K, "kn",
                    alpha=1.5, beta=0.5, A=A, B=B, C=C, d_dtype="f32", seed=seed)


def config2(M=4096, N=4096, K=4096, seed=None) -> Workload:
    seed = 1002 if seed is None else seed
    rng = np.random.default_rng(seed)
    sd = 1.0 / math.sqrt(K)
    A = _bf16(rng.standard_normal((M, K), dtype=np.float32) * sd)
    B = _bf16(rng.standard_normal((K, N), dtype=np.float32) * sd)
    return Workload(2, f"bf16 {M}x{N}x{K} bf16-out", "bf16", M, N, K, "kn", A=A, B=B,
                    d_dtype="bf16", seed=seed)


def _fp8_inputs(rng, M, N, K):
    X = rng.standard_normal((M, K), dtype=np.float32) * _log_uniform_rows(rng, M)
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    Xq, sx = quantize_e4m3_rows(X)
    Wq, sw = quantize_e4m3_rows(W)       # one scale per output channel (row of W)
    return Xq, sx, Wq, sw


def config3(M=4096, N=11008, K=4096, seed=None) -> Workload:
    seed = 1003 if seed is None else seed
    rng = np.random.default_rng(seed)
    Xq, sx, Wq, sw = _fp8_inputs(rng, M, N, K)
    return Workload(3, f"fp8 {M}x{N}x{K} per-token x per-channel -> bf16", "fp8", M, N, K, "nk",
                    A=Xq, B=Wq, a_scale=sx, b_scale=sw, d_dtype="bf16", seed=seed)


def config4(M=16, N=18432, K=7168, seed=None) -> Workload:
    seed = 1004 if seed is None else seed
    rng = np.random.default_rng(seed)
    X = _bf16(rng.standard_normal((M, K), dtype=np.float32))
    W = _bf16(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    return Workload(4, f"decode bf16 {M}x{N}x{K} weights NxK", "bf16", M, N, K, "nk",
                    A=X, B=W, d_dtype="bf16", seed=seed)


def config5(M=8192, N=8192, K=8192, seed=None) -> Workload:
    seed = 1005 if seed is None else seed
    rng = np.random.default_rng(seed)
    Xq, sx, Wq, sw = _fp8_inputs(rng, M, N, K)
    bias = torch.from_numpy(rng.standard_normal(N, dtype=np.float32) * np.float32(0.1))
    return Workload(5, f"fp8 {M}x{N}x{K} + bias -> SiLU -> E4M3 row requant", "fp8", M, N, K,
                    "nk", A=Xq, B=Wq, a_scale=sx, b_scale=sw, bias=bias, act="silu",
                    d_dtype="e4m3", out_quant="e4m3_row_amax", seed=seed)


def fp8_grouped(M=4096, N=11008, K=4096, k_group=128, b_layout="nk", seed=None, d_dtype="bf16",
                b_block=1) -> Workload:
    """FP8 GEMM with per-K-group scales: the workload 3 recipe, with an extra
    log-uniform magnitude per (token, K group) in [0.1, 10] on the activations
    and per (channel, K group) in [0.5, 2] on the weights (per block of b_block
    channels when b_block > 1), so neighbouring groups and blocks get different
    scales. a_scale [G, M], b_scale [G, N] (b_block > 1: [G, ceil(N / b_block)],
    one scale per block of weights)."""
    seed = 1003 if seed is None else seed
    rng = np.random.default_rng(seed)
    G = -(-K // k_group)
    tx = np.exp(rng.uniform(math.log(0.1), math.log(10.0), size=(M, G))).astype(np.float32)
    tw = np.exp(rng.uniform(math.log(0.5), math.log(2.0), size=(-(-N // b_block), G))).astype(np.float32)
    cols = np.arange(K) // k_group
    X = rng.standard_normal((M, K), dtype=np.float32) * _log_uniform_rows(rng, M) * tx[:, cols]
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02) * tw[np.arange(N) // b_block][:, cols]
    Xq, sx = quantize_e4m3_groups(X, k_group)
    Wq, sw = quantize_e4m3_groups(W, k_group) if b_block == 1 else quantize_e4m3_blocks(W, k_group, b_block)
    if b_layout == "kn":
        Wq = Wq.t().contiguous()
    what = f"per-{k_group}-K-group scales" + (f", {b_block}-channel weight blocks" if b_block > 1 else "")
    return Workload(3, f"fp8 {M}x{N}x{K} {what} -> {d_dtype}", "fp8", M, N, K,
                    b_layout, A=Xq, B=Wq, a_scale=sx, b_scale=sw, d_dtype=d_dtype, k_group=k_group,
                    b_block=b_block, seed=seed)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def make(number: int, **kw) -> Workload:
    return CONFIGS[number](**kw)


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """Raw BF16 bit patterns of a (CPU) bf16 tensor, as uint16."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def codes_u8(t: torch.Tensor) -> np.ndarray:
    """Raw E4M3 codes of a (CPU) float8_e4m3fn tensor, as uint8."""
    return t.contiguous().view(torch.uint8).numpy()
