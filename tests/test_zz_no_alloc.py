"""The allocation-free requantising FP8 GEMM, through the C ABI.

dgemm_fp8_rowquant_noalloc serves callers that cannot allocate device memory
when they run the GEMM (allocator callbacks, paths that must not synchronise
the device, runtimes with memory fixed at start-up): its scratch is a static
device array inside the library instead of a caller workspace. This test runs
it twice in a row on different problems and checks each result against the
workspace-taking entry point dgemm_fp8_scaled on the same inputs, with the
requantisation tolerance the other tests use. It sits in its own file, named
to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from dense_gemm_persistent_gb300 import _lib
from tolerances import e4m3_spacing

pytestmark = pytest.mark.gpu


def with_workspace(g, w, dev):
    q = torch.empty(w.M, w.N, dtype=torch.uint8, device=dev)
    s = torch.empty(w.M, dtype=torch.float32, device=dev)
    ws = torch.empty(dg.dgemm_workspace_size(1, w.M, w.N, w.K, "nk", out_quant="e4m3_row_amax"),
                     dtype=torch.uint8, device=dev)
    dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, q, b_layout="nk", bias=g.bias, act=w.act,
                        out_quant="e4m3_row_amax", out_row_scale=s, ws=ws)
    return q, s


def no_alloc(lib, g, w, dev):
    q = torch.empty(w.M, w.N, dtype=torch.uint8, device=dev)
    s = torch.empty(w.M, dtype=torch.float32, device=dev)
    epi = _lib.Epilogue(g.bias.data_ptr(), _lib.ACT[w.act], _lib.QUANT["e4m3_row_amax"], s.data_ptr())
    code = lib.dgemm_fp8_rowquant_noalloc(g.A.data_ptr(), g.B.data_ptr(), _lib.B_NK, g.a_scale.data_ptr(),
                                          g.b_scale.data_ptr(), None, _lib.F32, q.data_ptr(), w.M, w.N, w.K,
                                          1.0, 0.0, ctypes.byref(epi),
                                          torch.cuda.current_stream().cuda_stream)
    assert code == 0, dg.dgemm_status_string(code)
    return q, s


def close(q_new, s_new, q_ref, s_ref):
    dq_new = oracle.decode_e4m3(q_new.cpu().numpy()) * s_new.cpu().numpy().astype(np.float64)[:, None]
    dq_ref = oracle.decode_e4m3(q_ref.cpu().numpy()) * s_ref.cpu().numpy().astype(np.float64)[:, None]
    ulp = e4m3_spacing(dq_ref, s_ref.cpu().numpy().astype(np.float64))
    assert np.all(np.abs(dq_new - dq_ref) <= ulp)
    assert np.allclose(s_new.cpu().numpy(), s_ref.cpu().numpy(), rtol=1e-5, atol=0)


def test_no_alloc_matches_workspace_entry_point_twice():
    dev = torch.device("cuda:0")
    lib = dg.load(build_if_missing=True)
    # two calls in a row: a larger problem, then a smaller one whose zeroed
    # scratch must not see the first call's leftovers
    for shape, seed in (((512, 2048, 1024), 11), ((130, 528, 384), 12)):
        w = wl.make(5, M=shape[0], N=shape[1], K=shape[2], seed=seed)
        g = w.to(dev)
        q_new, s_new = no_alloc(lib, g, w, dev)
        torch.cuda.synchronize()
        assert dg.dgemm_query_device_status() == 0
        q_ref, s_ref = with_workspace(g, w, dev)
        torch.cuda.synchronize()
        close(q_new, s_new, q_ref, s_ref)


def test_no_alloc_rejects_problems_beyond_its_scratch():
    lib = dg.load(build_if_missing=True)
    epi = _lib.Epilogue(None, 3, 1, 16)
    # 4096 x 8192 needs 64 MiB of scratch, more than the 32 MiB array
    code = lib.dgemm_fp8_rowquant_noalloc(16, 16, _lib.B_NK, 16, 16, None, _lib.F32, 16, 4096, 8192, 256,
                                          1.0, 0.0, ctypes.byref(epi), None)
    assert code == 4   # DGEMM_ERR_WORKSPACE_TOO_SMALL
