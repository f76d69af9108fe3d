"""The allocation-free requantising FP8 GEMM, through the C ABI.

dgemm_fp8_rowquant_noalloc serves callers that cannot allocate device memory
when they run the GEMM (allocator callbacks, paths that must not synchronise
the device, runtimes with memory fixed at start-up): its scratch is a static
device array inside the library instead of a caller workspace. These tests run
it on several problems in a row and check each result against the
workspace-taking entry point dgemm_fp8_scaled on the same inputs and against
the float64 oracle, with the requantisation tolerance the other tests use:
a fault shared by both entry points, or one only in the whole-tile fallback
taken when the split area does not fit the array, shows up against the oracle.
The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from dense_gemm_persistent_gb300 import _lib
from tolerances import e4m3_spacing, requant_ok

pytestmark = pytest.mark.gpu


def c_args(g, w):
    """(C pointer, its dtype code) of workload w on the device, or none."""
    if w.beta != 0.0 and g.C is not None:
        return g.C.data_ptr(), _lib.F32
    return None, _lib.F32


def with_workspace(g, w, dev):
    q = torch.empty(w.M, w.N, dtype=torch.uint8, device=dev)
    s = torch.empty(w.M, dtype=torch.float32, device=dev)
    ws = torch.empty(dg.dgemm_workspace_size(1, w.M, w.N, w.K, "nk", out_quant="e4m3_row_amax"),
                     dtype=torch.uint8, device=dev)
    dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, q, b_layout="nk", C=g.C, alpha=w.alpha, beta=w.beta,
                        bias=g.bias, act=w.act, out_quant="e4m3_row_amax", out_row_scale=s, ws=ws)
    torch.cuda.synchronize()
    assert dg.dgemm_query_device_status(ws) == 0
    return q, s


def no_alloc(lib, g, w, dev):
    q = torch.empty(w.M, w.N, dtype=torch.uint8, device=dev)
    s = torch.empty(w.M, dtype=torch.float32, device=dev)
    epi = _lib.Epilogue(g.bias.data_ptr(), _lib.ACT[w.act], _lib.QUANT["e4m3_row_amax"], s.data_ptr())
    c_ptr, c_dt = c_args(g, w)
    code = lib.dgemm_fp8_rowquant_noalloc(g.A.data_ptr(), g.B.data_ptr(), _lib.B_NK, g.a_scale.data_ptr(),
                                          g.b_scale.data_ptr(), c_ptr, c_dt, q.data_ptr(), w.M, w.N, w.K,
                                          w.alpha, w.beta, ctypes.byref(epi),
                                          torch.cuda.current_stream().cuda_stream)
    assert code == 0, dg.dgemm_status_string(code)
    torch.cuda.synchronize()
    assert dg.dgemm_query_device_status(None) == 0   # these calls report on the per-device word
    return q, s


def close(q_new, s_new, q_ref, s_ref):
    """Dequantised outputs of the two entry points within one E4M3 step of each
    other. When the two sum in different orders (whole tiles here, split tiles
    there) their FP32 values, row maxima and scales differ by rounding, so a
    value near a rounding boundary can take neighbouring codes on the two
    slightly different grids: one step, plus the scales' relative difference."""
    s_new_np = s_new.cpu().numpy().astype(np.float64)
    s_ref_np = s_ref.cpu().numpy().astype(np.float64)
    dq_new = oracle.decode_e4m3(q_new.cpu().numpy()) * s_new_np[:, None]
    dq_ref = oracle.decode_e4m3(q_ref.cpu().numpy()) * s_ref_np[:, None]
    ulp = e4m3_spacing(dq_ref, s_ref_np)
    srel = np.abs(s_new_np - s_ref_np) / s_ref_np
    bound = ulp + np.abs(dq_ref) * srel[:, None] * 2.0
    ratio = np.abs(dq_new - dq_ref) / ulp
    assert np.all(np.abs(dq_new - dq_ref) <= bound), f"worst {ratio.max():.4f} E4M3 steps apart"
    assert np.all(srel <= 1e-5), f"row scales {srel.max():.2e} apart"


def oracle_rows(w, rows):
    """The exact pre-quantisation values y of the given rows."""
    C = None if w.C is None else w.C.numpy()
    return oracle.fp8_gemm_ref(wl.codes_u8(w.A), wl.codes_u8(w.B), "nk", w.a_scale.numpy(), w.b_scale.numpy(),
                               C, w.alpha, w.beta, w.bias.numpy(), w.act, rows=rows)


def check_against_oracle(q, s, w, rows):
    ok, msg = requant_ok(q.cpu().numpy()[rows], s.cpu().numpy()[rows], oracle_rows(w, rows))
    assert ok, msg


def with_c(w, seed):
    """Workload w with an FP32 C term: D = SiLU(alpha * acc + beta * C + bias), requantised."""
    rng = np.random.default_rng(seed)
    w.C = torch.from_numpy(rng.standard_normal((w.M, w.N)).astype(np.float32))
    w.alpha, w.beta = 0.75, -1.5
    return w


def test_no_alloc_matches_workspace_entry_point_and_oracle_twice():
    dev = torch.device("cuda:0")
    lib = dg.load(build_if_missing=True)
    # calls in a row: a larger problem, then a smaller one whose zeroed scratch
    # must not see the first call's leftovers, then one with a C term
    cases = [wl.make(5, M=512, N=2048, K=1024, seed=11),
             wl.make(5, M=130, N=528, K=384, seed=12),
             with_c(wl.make(5, M=384, N=1040, K=640, seed=13), 14)]
    for w in cases:
        g = w.to(dev)
        q_new, s_new = no_alloc(lib, g, w, dev)
        q_ref, s_ref = with_workspace(g, w, dev)
        close(q_new, s_new, q_ref, s_ref)
        rows = np.unique(np.concatenate([np.arange(0, w.M, max(1, w.M // 40)), [w.M - 1]])).astype(np.int64)
        check_against_oracle(q_new, s_new, w, rows)


def test_no_alloc_whole_tile_fallback_when_the_split_area_does_not_fit():
    """2048 x 8064 with K = 6144: the requantising scratch (33.0 MB) fits the
    32 MiB array but the split area for the last partial wave does not, so the
    allocation-free call runs every tile whole while the workspace entry point
    splits the 28 leftover tiles along K. Both match the oracle."""
    dev = torch.device("cuda:0")
    lib = dg.load(build_if_missing=True)
    M, N, K = 2048, 8064, 6144
    base = 256 + 256 + 4 * M + 2 * M * N
    assert base <= _lib.NOALLOC_SCRATCH_BYTES
    assert dg.dgemm_workspace_size(1, M, N, K, "nk", out_quant="e4m3_row_amax") > _lib.NOALLOC_SCRATCH_BYTES
    plan = dg.dgemm_plan(1, M, N, K, "nk", "e4m3", out_quant="e4m3_row_amax", act="silu", num_sms=0)
    if plan["cta_group"] != 2 or plan["grid"] != 152:
        pytest.skip("needs 76 resident CTA pairs")
    assert plan["tail_split"] == 2            # the workspace entry point splits the tail
    w = wl.make(5, M=M, N=N, K=K, seed=15)
    g = w.to(dev)
    q_new, s_new = no_alloc(lib, g, w, dev)
    q_ref, s_ref = with_workspace(g, w, dev)
    # rows of every tile row (the split tiles are tile rows 4-7 of the last
    # tile columns, the last one ragged), against the oracle for both paths
    rows = np.array(sorted({0, 1, 255, 300, 600, 1000, 1100, 1300, 1500, 1792, 1793, 2000, M - 1}),
                    dtype=np.int64)
    check_against_oracle(q_new, s_new, w, rows)
    check_against_oracle(q_ref, s_ref, w, rows)
    close(q_new, s_new, q_ref, s_ref)


def test_no_alloc_rejects_problems_beyond_its_scratch():
    lib = dg.load(build_if_missing=True)
    epi = _lib.Epilogue(None, 3, 1, 16)
    # 4096 x 8192 needs 64 MiB of scratch, more than the 32 MiB array
    code = lib.dgemm_fp8_rowquant_noalloc(16, 16, _lib.B_NK, 16, 16, None, _lib.F32, 16, 4096, 8192, 256,
                                          1.0, 0.0, ctypes.byref(epi), None)
    assert code == 4   # DGEMM_ERR_WORKSPACE_TOO_SMALL
    # 2048 x 8192 is just beyond it: the status header, counters and row maxima
    # come on top of the 32 MiB stash
    code = lib.dgemm_fp8_rowquant_noalloc(16, 16, _lib.B_NK, 16, 16, None, _lib.F32, 16, 2048, 8192, 256,
                                          1.0, 0.0, ctypes.byref(epi), None)
    assert code == 4
