"""Bounded device-side waits driven to their limit, and the recovery after.

The debugging order on the DeepGEMM write-up (czchanglian.com/news/51329,
§4.2-4.3) puts the placement of synchronisation first. Here the synchronisation
code that no ordinary run reaches -- a wait that gives up, the error word it
sets, the drain of every role, the Tensor Memory release after an abort -- is
run on purpose, without any fault: a testing override makes every CTA's operand
producer stop issuing loads after a few stages, so the tensor-core issuer's
wait for the next stage runs out (after a short limit, also an override). The
call must report DGEMM_ERR_DEVICE_TIMEOUT through the status word it was given
(its workspace's, or the per-device one), and the next ordinary call on the
same device must be bit-exact and leave the status clean.
"""
import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from gpu_util import dev, status_ok
from tolerances import requant_ok

pytestmark = pytest.mark.gpu

TIMEOUT = 6              # DGEMM_ERR_DEVICE_TIMEOUT
LIMIT_NS = 20_000_000    # 20 ms per bounded wait while stalled


def int_tensor(rng, shape, dt):
    return torch.from_numpy(rng.integers(-4, 5, size=shape).astype(np.float32)).to(dt)


def bf16_call(M, N, K, seed, ws_bytes):
    rng = np.random.default_rng(seed)
    A = int_tensor(rng, (M, K), torch.bfloat16)
    B = int_tensor(rng, (N, K), torch.bfloat16)
    D = torch.empty(M, N, dtype=torch.float32, device=dev())
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev()) if ws_bytes else None
    if ws is not None:
        ws.fill_(0xA5)               # arbitrary contents on entry
    Ad, Bd = A.to(dev()), B.to(dev())
    ref = oracle.bf16_gemm_ref(wl.bits_u16(A), wl.bits_u16(B), "nk")
    return lambda: dg.dgemm_bf16(Ad, Bd, D, b_layout="nk", ws=ws), D, ws, ref


@pytest.mark.parametrize("M,N,K,pair", [(128, 512, 1024, "0"),     # single-CTA 128-row tiles
                                        (2560, 2048, 512, "1"),    # CTA pairs, 256 x 256 tiles
                                        (512, 1024, 1024, "1"),    # CTA pairs, split-K through the workspace
                                        (16, 1024, 2048, None)])   # small-M transposed form
def test_stalled_producer_reports_timeout_through_the_workspace(M, N, K, pair, knobs):
    if pair is not None:
        knobs(cta_pair=pair, tile_n="256")   # pairs exist for 256-wide tiles
    ws_bytes = max(dg.dgemm_workspace_size(0, M, N, K, "nk"), 256)
    call, D, ws, ref = bf16_call(M, N, K, seed=M + K, ws_bytes=ws_bytes)
    plan = dg.dgemm_plan(0, M, N, K, "nk", "f32", num_sms=0)
    assert plan["cta_group"] == (2 if pair == "1" else 1)
    knobs(wait_limit_ns=LIMIT_NS, stall_after_loads=3)
    call()
    assert dg.dgemm_query_device_status(ws) == TIMEOUT
    assert dg.dgemm_query_device_status(ws) == 0        # the query cleared it
    assert dg.dgemm_query_device_status(None) == 0      # the per-device word was not used
    # the next ordinary call on the same device and workspace
    knobs(wait_limit_ns=None, stall_after_loads=None)
    D.zero_()
    call()
    assert status_ok(ws)
    got = D.cpu().double().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


def test_stalled_producer_without_workspace_reports_on_the_device_word(knobs):
    M, N, K = 256, 768, 1024
    call, D, _, ref = bf16_call(M, N, K, seed=77, ws_bytes=0)
    assert dg.dgemm_plan(0, M, N, K, "nk", "f32", num_sms=0)["workspace_bytes"] == 0
    # (each K segment is 4 stages of two slices: stop below that)
    knobs(wait_limit_ns=LIMIT_NS, stall_after_loads=2)
    call()
    assert dg.dgemm_query_device_status(None) == TIMEOUT
    assert dg.dgemm_query_device_status(None) == 0
    knobs(wait_limit_ns=None, stall_after_loads=None)
    D.zero_()
    call()
    assert status_ok()
    assert np.array_equal(D.cpu().double().numpy(), ref)


def test_stalled_requantising_kernel_then_clean_call(knobs):
    """The cooperative requantising form: every role of every CTA (including
    the row-band waits) gives up and drains; the next call is within the
    requantisation tolerance of the oracle."""
    w = wl.make(5, M=512, N=1024, K=1024, seed=31)
    g = w.to(dev())
    q = torch.empty(w.M, w.N, dtype=torch.uint8, device=dev())
    s = torch.empty(w.M, dtype=torch.float32, device=dev())
    ws = torch.empty(dg.dgemm_workspace_size(1, w.M, w.N, w.K, "nk", out_quant="e4m3_row_amax"),
                     dtype=torch.uint8, device=dev())

    def call():
        dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, q, b_layout="nk", bias=g.bias, act="silu",
                            out_quant="e4m3_row_amax", out_row_scale=s, ws=ws)

    assert dg.dgemm_plan(1, w.M, w.N, w.K, "nk", "e4m3", out_quant="e4m3_row_amax", num_sms=0)["cooperative"] == 1
    knobs(wait_limit_ns=LIMIT_NS, stall_after_loads=2)
    call()
    assert dg.dgemm_query_device_status(ws) == TIMEOUT
    knobs(wait_limit_ns=None, stall_after_loads=None)
    call()
    assert status_ok(ws)
    y = oracle.fp8_gemm_ref(wl.codes_u8(w.A), wl.codes_u8(w.B), "nk", w.a_scale.numpy(), w.b_scale.numpy(),
                            bias=w.bias.numpy(), act="silu")
    ok, msg = requant_ok(q.cpu().numpy(), s.cpu().numpy(), y)
    assert ok, msg
