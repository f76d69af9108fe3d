"""Algorithmic work and traffic models used to report measurements.

The tiled-traffic model is the one on the tiling page ("GEMM(矩阵乘)",
blog.daoxuan.cc/posts/60929, the sections on counting repeated reads and on
arithmetic intensity): an output tile of edge T reads a T x K strip of A and a
K x T strip of B, so each A row is re-read N/T times and each B column M/T
times; the reads total 2MNK/T elements (2MNK untiled), and a block's arithmetic
intensity is 2T^2 k FLOP over 2Tk elements, T/2 FLOP per byte for 2-byte types.
Rectangular BM x BN tiles generalise this to MNK (1/BN + 1/BM) elements.
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int) -> int:
    """2MNK: one multiply and one add per (m, n, k)."""
    return 2 * M * N * K


def untiled_read_elements(M: int, N: int, K: int) -> int:
    """Every output element reads a full row of A and column of B: 2MNK elements."""
    return 2 * M * N * K


def tiled_read_elements(M: int, N: int, K: int, BM: int, BN: int | None = None) -> float:
    """Operand elements read from HBM with BM x BN output tiles and no L2 reuse."""
    BN = BM if BN is None else BN
    return M * N * K * (1.0 / BN + 1.0 / BM)


def reads_per_output(K: int, T: int) -> float:
    """Reads per output element with square tiles of edge T: 2K / T."""
    return 2.0 * K / T


def tile_intensity(T: int, elem_bytes: int = 2) -> float:
    """FLOP per byte of a T x T output tile: 2 T^2 k / (2 T k elem_bytes)."""
    return T / float(elem_bytes)


def ridge_point(peak_flops: float, bandwidth_bytes: float) -> float:
    """Intensity (FLOP/B) at which the compute and bandwidth roofs meet."""
    return peak_flops / bandwidth_bytes


def compulsory_bytes(M: int, N: int, K: int, a_bytes: float, b_bytes: float,
                     c_in_bytes: float, d_bytes: float) -> float:
    """Each operand read once and the output written once."""
    return M * K * a_bytes + K * N * b_bytes + M * N * (c_in_bytes + d_bytes)
