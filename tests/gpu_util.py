"""Shared helpers of the GPU parity tests: running the library on a workload and
fetching results as numpy arrays. Nothing here computes a reference."""
from __future__ import annotations

import numpy as np
import torch

import dense_gemm_persistent_gb300 as dg
import workloads as wl


def dev():
    return torch.device("cuda:0")


def status_ok(ws=None, stream=None) -> bool:
    """No bounded device wait gave up: neither in the per-device status word nor,
    when the call was given one, in its workspace's status word."""
    dev_word = dg.dgemm_query_device_status(None, stream)
    ws_word = dg.dgemm_query_device_status(ws, stream) if ws is not None else 0
    return dev_word == 0 and ws_word == 0


def run_workload(w: wl.Workload, d_dtype: str | None = None):
    """Run the library on workload w (tensors on CPU); returns (D, row_scale or None)
    as CPU tensors, after checking the device status word."""
    g = w.to(dev())
    d_dtype = d_dtype or w.d_dtype
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}[d_dtype]
    D = torch.empty(w.M, w.N, dtype=tdt, device=dev())
    s = None
    if w.out_quant != "none":
        s = torch.full((w.M,), -1.0, dtype=torch.float32, device=dev())   # (every row must be written)
    # the workspace the library can use (tail splitting, requantisation)
    nbytes = dg.dgemm_workspace_size(w.form == "fp8", w.M, w.N, w.K, w.b_layout, out_quant=w.out_quant)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev()) if nbytes else None
    kw = dict(b_layout=w.b_layout, C=g.C, alpha=w.alpha, beta=w.beta, bias=g.bias, act=w.act,
              out_quant=w.out_quant, out_row_scale=s, ws=ws)
    if w.form == "bf16":
        dg.dgemm_bf16(g.A, g.B, D, **kw)
    else:
        dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, D, k_group=w.k_group, b_block=w.b_block, **kw)
    assert status_ok(ws)
    return D.cpu(), (None if s is None else s.cpu())


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy() if t.dtype != torch.uint8 else t.numpy()
