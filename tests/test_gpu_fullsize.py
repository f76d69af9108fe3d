"""The five workloads at their full sizes, in the launch configuration the
benchmark times (the library's own plan), checked on sampled rows that the
oracle computes one by one (whole rows, so every column tile is covered; at
least one row in every 256-row tile row and the last row of every raster band,
so every tile of the output is checked), and in full where the oracle is fast
enough (workloads 1 and 4)."""
import numpy as np
import pytest

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from gpu_util import run_workload, to_f64
from test_gpu_parity import ref_of
from tolerances import bf16_ulp_ok, c1_ok, frob_ok, requant_ok

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def sample_rows(M, n=32, seed=0, tile=256, band=2048):
    """n random rows, plus one random row inside every tile row of `tile`
    rows, the last row of every raster band (`band` rows: 8 tile rows), and
    the first and last two rows."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(M, size=min(n, M), replace=False).tolist()) | {0, 1, M - 2, M - 1}
    for t0 in range(0, M, tile):
        pick.add(int(rng.integers(t0, min(M, t0 + tile))))
    for b0 in range(0, M, band):
        pick.add(min(M, b0 + band) - 1)
    return np.array(sorted(pick), dtype=np.int64)


def test_sample_rows_touch_every_tile_row_and_band_end():
    rows = sample_rows(8192, 24, seed=5)
    assert set(rows // 256) == set(range(32))
    assert {2047, 4095, 6143, 8191} <= set(rows.tolist())


def test_workload1_full():
    w = wl.make(1)
    D, _ = run_workload(w)
    ok, msg = c1_ok(to_f64(D), ref_of(w), w.K)
    assert ok, msg


def test_workload2_full_size_sampled_rows():
    w = wl.make(2)
    D, _ = run_workload(w)
    rows = sample_rows(w.M, 48, seed=2)
    ok, msg = bf16_ulp_ok(to_f64(D)[rows], ref_of(w, rows=rows))
    assert ok, msg


def test_workload3_full_size_sampled_rows():
    w = wl.make(3)
    D, _ = run_workload(w)
    rows = sample_rows(w.M, 32, seed=3)
    ok, msg = frob_ok(to_f64(D)[rows], ref_of(w, rows=rows))
    assert ok, msg


def test_workload4_full():
    w = wl.make(4)
    assert dg.dgemm_plan(0, w.M, w.N, w.K, "nk", "bf16")["swap_ab"] == 1
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


def test_workload5_full_size_sampled_rows():
    w = wl.make(5)
    q, s = run_workload(w)
    rows = sample_rows(w.M, 24, seed=5)
    ok, msg = requant_ok(q.numpy()[rows], s.numpy()[rows], ref_of(w, rows=rows))
    assert ok, msg
    # properties that hold on every row: each row's scale is positive and its
    # largest code magnitude is the E4M3 maximum (448) unless the row is zero
    qa = q.numpy() & 0x7F
    assert np.all(s.numpy() > 0)
    assert np.all(qa.max(axis=1) == 0x7E)


def test_fp8_grouped_scales_full_size_sampled_rows():
    """The FFN projection of workload 3 with one scale per 128-element K group."""
    w = wl.fp8_grouped(4096, 11008, 4096, k_group=128)
    D, _ = run_workload(w)
    rows = sample_rows(w.M, 24, seed=6)
    ok, msg = bf16_ulp_ok(to_f64(D)[rows], ref_of(w, rows=rows))
    assert ok, msg


def test_fp8_block_scaled_full_size_sampled_rows():
    """The same projection with block-scaled weights: one scale per (128-channel
    block, 128-element K group)."""
    w = wl.fp8_grouped(4096, 11008, 4096, k_group=128, b_block=128)
    D, _ = run_workload(w)
    rows = sample_rows(w.M, 24, seed=7)
    ok, msg = bf16_ulp_ok(to_f64(D)[rows], ref_of(w, rows=rows))
    assert ok, msg
