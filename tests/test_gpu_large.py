"""Maximum sizes: element offsets beyond 2^31 and very long K.

Every output tile of these problems is addressed with coordinates that fit in
32 bits, but the element offsets of C loads, transposed stores and the
requantisation stash (row * leading dimension + column) pass 2^31, so any
32-bit offset arithmetic would read or write the wrong elements. Long K runs
hundreds of thousands of pipeline phases per tile. Integer operands keep the
first four cases bit-exact (every FP32 partial sum below 2^24); the
requantising case uses the workload recipe and its tolerance. Results are
checked on sampled rows (or columns) that include the ones past 2^31.

C is built on the device from two seeded integer vectors, C[m, n] = u[m] + v[n]
(small integers, exact in FP32), so that no multi-gigabyte array is generated
on the host; the oracle receives the same values computed on the host.
"""
import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from gpu_util import dev, status_ok
from tolerances import requant_ok

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TWO31 = 2 ** 31


def int_tensor(rng, shape, lo, hi, dtype):
    """Seeded small integers as a CPU tensor of dtype (int8 on the host first, to
    keep host memory at one byte per element)."""
    return torch.from_numpy(rng.integers(lo, hi + 1, size=shape, dtype=np.int8)).to(dtype)


def outer_sum_c(rng, M, N):
    """(u, v) on the host and C = u[:, None] + v[None, :] (FP32) on the device."""
    u = rng.integers(-3, 4, size=M, dtype=np.int8)
    v = rng.integers(-3, 4, size=N, dtype=np.int8)
    C = (torch.from_numpy(u).to(dev(), torch.float32)[:, None]
         + torch.from_numpy(v).to(dev(), torch.float32)[None, :])
    return u, v, C


def release():
    """Hand the freed multi-gigabyte buffers back before the next test (a failed
    assertion's traceback would otherwise keep them alive)."""
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_tile_path_c_and_d_offsets_beyond_2_31():
    # M x N = 49152^2 = 2.42e9 elements: rows >= 43691 start past 2^31
    M = N = 49152
    K = 64
    assert (M - 1) * N > TWO31
    rng = np.random.default_rng(2101)
    A = int_tensor(rng, (M, K), -4, 4, torch.bfloat16)
    B = int_tensor(rng, (K, N), -4, 4, torch.bfloat16)
    u, v, C = outer_sum_c(rng, M, N)
    D = torch.empty(M, N, dtype=torch.float32, device=dev())
    dg.dgemm_bf16(A.to(dev()), B.to(dev()), D, b_layout="kn", C=C, alpha=1.0, beta=1.0)
    assert status_ok()
    rows = np.array(sorted({0, 1, TWO31 // N, TWO31 // N + 1, M - 2, M - 1}
                           | set(np.random.default_rng(7).choice(M, 8, replace=False).tolist())), dtype=np.int64)
    got = D[torch.from_numpy(rows).to(dev())].cpu().numpy().astype(np.float64)
    c_rows = (u[rows].astype(np.float32)[:, None] + v.astype(np.float32)[None, :]).astype(np.float32)
    ref = oracle.bf16_gemm_ref(wl.bits_u16(A)[rows], wl.bits_u16(B), "kn", c_rows, 1.0, 1.0)
    del C, D
    release()
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} mismatches"


def test_small_m_transposed_store_offsets_beyond_2_31():
    # small-M (transposed) form: D[m, n] is stored at m * N + n by direct stores;
    # with M = 64 the last rows start past 2^31
    M, K = 64, 16
    N = 2 ** 25 + 2 ** 20
    assert (M - 1) * N > TWO31
    rng = np.random.default_rng(2102)
    A = int_tensor(rng, (M, K), -4, 4, torch.bfloat16)
    B = int_tensor(rng, (N, K), -4, 4, torch.bfloat16)
    u, v, C = outer_sum_c(rng, M, N)
    D = torch.empty(M, N, dtype=torch.float32, device=dev())
    plan = dg.dgemm_plan(0, M, N, K, "nk", "f32")
    assert plan["swap_ab"] == 1
    dg.dgemm_bf16(A.to(dev()), B.to(dev()), D, b_layout="nk", C=C, alpha=1.0, beta=1.0)
    assert status_ok()
    pick = np.random.default_rng(8).choice(N, 512, replace=False)
    cols = np.array(sorted(set(pick.tolist()) | set(range(0, 64)) | set(range(N - 512, N))), dtype=np.int64)
    got = D[:, torch.from_numpy(cols).to(dev())].cpu().numpy().astype(np.float64)
    c_cols = (u.astype(np.float32)[:, None] + v[cols].astype(np.float32)[None, :]).astype(np.float32)
    ref = oracle.bf16_gemm_ref(wl.bits_u16(A), wl.bits_u16(B)[cols], "nk", c_cols, 1.0, 1.0)
    del C, D
    release()
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} mismatches"


@pytest.mark.parametrize("fp8", [0, 1])
def test_very_long_k(fp8):
    # K = 2^19: 8192 (BF16) or 4096 (E4M3) K slices per tile; entries in {-1, 0, 1}
    # keep every partial sum (|s| <= 2^19) exact in FP32
    M, N, K = 256, 384, 2 ** 19
    rng = np.random.default_rng(2103 + fp8)
    dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    A = int_tensor(rng, (M, K), -1, 1, torch.float32).to(dt)
    B = int_tensor(rng, (N, K), -1, 1, torch.float32).to(dt)
    D = torch.empty(M, N, dtype=torch.float32, device=dev())
    nbytes = dg.dgemm_workspace_size(fp8, M, N, K, "nk")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev()) if nbytes else None
    if fp8:
        ones_m = torch.ones(M, dtype=torch.float32, device=dev())
        ones_n = torch.ones(N, dtype=torch.float32, device=dev())
        dg.dgemm_fp8_scaled(A.to(dev()), B.to(dev()), ones_m, ones_n, D, b_layout="nk", ws=ws)
    else:
        dg.dgemm_bf16(A.to(dev()), B.to(dev()), D, b_layout="nk", ws=ws)
    assert status_ok(ws)
    rows = np.array([0, 1, 127, 128, 200, M - 1], dtype=np.int64)
    got = D.cpu().numpy().astype(np.float64)[rows]
    if fp8:
        ref = oracle.fp8_gemm_ref(wl.codes_u8(A), wl.codes_u8(B), "nk", np.ones(M, np.float32),
                                  np.ones(N, np.float32), rows=rows)
    else:
        ref = oracle.bf16_gemm_ref(wl.bits_u16(A), wl.bits_u16(B), "nk", rows=rows)
    del D, ws
    release()
    assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} mismatches"


def test_requant_stash_offsets_beyond_2_31():
    # FP8 + bias + SiLU + per-row E4M3 requantisation with M x N = 2.42e9: the
    # BF16 stash and the code array are indexed past 2^31 elements
    M = N = 49152
    K = 128
    w = wl.make(5, M=M, N=N, K=K, seed=2104)
    g = w.to(dev())
    q = torch.empty(M, N, dtype=torch.uint8, device=dev())
    s = torch.full((M,), -1.0, dtype=torch.float32, device=dev())
    ws = torch.empty(dg.dgemm_workspace_size(1, M, N, K, "nk", out_quant="e4m3_row_amax"),
                     dtype=torch.uint8, device=dev())
    dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, q, b_layout="nk", bias=g.bias, act="silu",
                        out_quant="e4m3_row_amax", out_row_scale=s, ws=ws)
    assert status_ok(ws)
    rows = np.array(sorted({0, TWO31 // N, TWO31 // N + 1, M - 1}
                           | set(np.random.default_rng(9).choice(M, 6, replace=False).tolist())), dtype=np.int64)
    idx = torch.from_numpy(rows).to(dev())
    q_rows = q[idx].cpu().numpy()
    s_rows = s[idx].cpu().numpy()
    del q, ws, s, g
    release()
    y = oracle.fp8_gemm_ref(wl.codes_u8(w.A), wl.codes_u8(w.B), "nk", w.a_scale.numpy(), w.b_scale.numpy(),
                            bias=w.bias.numpy(), act="silu", rows=rows)
    ok, msg = requant_ok(q_rows, s_rows, y)
    assert ok, msg
