"""GPU vs oracle on the five workloads' value recipes, element by element, at
sizes the oracle finishes in seconds (several tiles plus ragged tails), and the
edge cases of the method: K = 0, one-row and one-column problems, in-place C,
alpha = 0, every activation, requantisation from the BF16 form, small-M
transposed path with bias and C."""
import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from gpu_util import dev, run_workload, status_ok, to_f64
from tolerances import bf16_ulp_ok, c1_ok, frob_ok, requant_ok

pytestmark = pytest.mark.gpu


def ref_of(w: wl.Workload, rows=None):
    C = None if w.C is None else w.C.numpy()
    if w.form == "bf16":
        y = oracle.bf16_gemm_ref(wl.bits_u16(w.A), wl.bits_u16(w.B), w.b_layout, C, w.alpha, w.beta, rows=rows)
        if w.bias is not None or w.act != "none":
            y = oracle.epilogue(y, None if w.bias is None else w.bias.numpy(), w.act)
        return y
    return oracle.fp8_gemm_ref(wl.codes_u8(w.A), wl.codes_u8(w.B), w.b_layout, w.a_scale.numpy(),
                               w.b_scale.numpy(), C, w.alpha, w.beta,
                               None if w.bias is None else w.bias.numpy(), w.act, rows=rows, k_group=w.k_group,
                               b_block=w.b_block)


def test_workload1_full_size():
    w = wl.make(1)
    D, _ = run_workload(w)
    ok, msg = c1_ok(to_f64(D), ref_of(w), w.K)
    assert ok, msg


@pytest.mark.parametrize("shape", [(300, 520, 1000), (1000, 1000, 1000), (129, 264, 4096), (640, 2048, 576)])
def test_workload2_recipe(shape):
    w = wl.make(2, M=shape[0], N=shape[1], K=shape[2])
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


@pytest.mark.parametrize("shape,layout", [((300, 528, 1024), "nk"), ((1000, 1008, 2048), "nk"),
                                          ((257, 512, 1024), "kn")])
def test_workload3_recipe(shape, layout):
    w = wl.make(3, M=shape[0], N=shape[1], K=shape[2])
    if layout == "kn":
        w.B = w.B.view(torch.uint8).t().contiguous().view(torch.float8_e4m3fn)
        w.b_layout = "kn"
    D, _ = run_workload(w)
    ok, msg = frob_ok(to_f64(D), ref_of(w))
    assert ok, msg


@pytest.mark.parametrize("M", [1, 5, 16, 33, 64])
def test_workload4_recipe_small_m(M):
    w = wl.make(4, M=M, N=4224, K=1024)
    plan = dg.dgemm_plan(0, w.M, w.N, w.K, "nk", "bf16")
    assert plan["swap_ab"] == 1
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


@pytest.mark.parametrize("shape", [(300, 528, 512), (256, 1024, 1024), (130, 2064, 384)])
def test_workload5_recipe(shape):
    w = wl.make(5, M=shape[0], N=shape[1], K=shape[2])
    q, s = run_workload(w)
    ok, msg = requant_ok(q.numpy(), s.numpy(), ref_of(w))
    assert ok, msg


# ------------------------------------------------------------------ edge cases

def test_k_zero_gives_beta_c_and_epilogue():
    w = wl.make(1, M=200, N=136, K=0)
    w.alpha, w.beta = 2.0, 0.5
    D, _ = run_workload(w)
    assert np.array_equal(to_f64(D), 0.5 * w.C.numpy().astype(np.float64))
    w5 = wl.make(5, M=130, N=272, K=0)       # y = SiLU(bias) on every row
    q, s = run_workload(w5)
    y = oracle.epilogue(np.zeros((130, 272)), w5.bias.numpy(), "silu")
    ok, msg = requant_ok(q.numpy(), s.numpy(), y)
    assert ok, msg


@pytest.mark.parametrize("shape", [(1, 8, 8), (1, 8, 4096), (7, 16, 64), (128, 8, 64), (1000, 8, 72)])
def test_tiny_and_one_sided_shapes(shape):
    M, N, K = shape
    w = wl.make(2, M=M, N=N, K=K)
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


def test_in_place_beta_with_bf16_c():
    w = wl.make(2, M=300, N=264, K=512)
    rng = np.random.default_rng(3)
    C = torch.from_numpy(rng.standard_normal((300, 264)).astype(np.float32)).to(torch.bfloat16)
    g = w.to(dev())
    D = C.to(dev())                         # C and D share storage
    dg.dgemm_bf16(g.A, g.B, D, b_layout="kn", C=D, alpha=0.75, beta=-1.25)
    assert status_ok()
    ref = oracle.bf16_gemm_ref(wl.bits_u16(w.A), wl.bits_u16(w.B), "kn", wl.bits_u16(C), 0.75, -1.25)
    ok, msg = bf16_ulp_ok(to_f64(D.cpu()), ref)
    assert ok, msg


def test_alpha_zero_reads_only_c():
    w = wl.make(1, M=256, N=256, K=256)
    w.alpha, w.beta = 0.0, 3.0
    D, _ = run_workload(w)
    assert np.array_equal(D.numpy(), np.float32(3.0) * w.C.numpy())   # one FP32 rounding of 3c


@pytest.mark.parametrize("act", ["relu", "gelu", "silu"])
@pytest.mark.parametrize("M", [40, 300])
def test_bias_and_activations_bf16_out(act, M):
    w = wl.make(2, M=M, N=520, K=768)
    w.bias = torch.from_numpy(np.random.default_rng(4).standard_normal(520).astype(np.float32) * 0.1)
    w.act = act
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


@pytest.mark.parametrize("M", [16, 200])
def test_fp8_with_c_bias_and_f32_output(M):
    w = wl.make(3, M=M, N=400, K=512)
    rng = np.random.default_rng(5)
    w.C = torch.from_numpy(rng.standard_normal((M, 400)).astype(np.float32))
    w.beta, w.alpha = 0.5, 1.25
    w.bias = torch.from_numpy(rng.standard_normal(400).astype(np.float32))
    w.act = "gelu"
    D, _ = run_workload(w, d_dtype="f32")
    ok, msg = c1_ok(to_f64(D), ref_of(w), w.K)
    assert ok, msg


def test_requant_tail_split(knobs):
    """The requantising epilogue with the last partial wave split along K: the
    split tiles' segments finish their units with plain stores into the stash
    and fold their row maxima in before counting their row band. 90 tiles of 256 x 256
    on 76 pairs: the last 14 (rows 2048-2559 in the banded raster) are split."""
    knobs(tail_split="force")
    knobs(tail_halves="0")
    w = wl.make(5, M=2560, N=2304, K=2048)
    plan = dg.dgemm_plan(1, w.M, w.N, w.K, "nk", "e4m3", out_quant="e4m3_row_amax", act="silu", num_sms=0)
    if plan["cta_group"] != 2 or plan["grid"] != 152:
        pytest.skip("needs 76 resident CTA pairs")
    assert plan["tail_tiles"] == 14 and plan["tail_split"] == 2
    q, s = run_workload(w)
    rows = np.array(sorted(set(range(2048, 2560, 23)) | {0, 1000, 2047, 2559}), dtype=np.int64)
    ok, msg = requant_ok(q.numpy()[rows], s.numpy()[rows], ref_of(w, rows=rows))
    assert ok, msg


def test_requant_tail_halves():
    """The same 90 tiles with the last 14 run as 28 halves of 256 x 128: each
    half stashes its columns and folds its row maxima in before counting its band."""
    w = wl.make(5, M=2560, N=2304, K=2048)
    plan = dg.dgemm_plan(1, w.M, w.N, w.K, "nk", "e4m3", out_quant="e4m3_row_amax", act="silu", num_sms=0)
    if plan["cta_group"] != 2 or plan["grid"] != 152:
        pytest.skip("needs 76 resident CTA pairs")
    assert plan["tail_tiles"] == 14 and plan["tail_halves"] == 1 and plan["tail_split"] == 1
    q, s = run_workload(w)
    rows = np.array(sorted(set(range(2048, 2560, 23)) | {0, 1000, 2047, 2559}), dtype=np.int64)
    ok, msg = requant_ok(q.numpy()[rows], s.numpy()[rows], ref_of(w, rows=rows))
    assert ok, msg


@pytest.mark.parametrize("M,N,K", [(8192, 512, 256), (130000, 64, 128)])
def test_requant_row_bands(M, N, K):
    """Row bands converted while later bands are still being multiplied: short
    K makes each tile quick, so bands finish throughout the call (32 raster
    groups of 2048 rows); 130000 rows make 64 raster groups, more than the
    header's band counters, so each band spans two groups (and N = 64 is one
    ragged quarter of a tile)."""
    w = wl.make(5, M=M, N=N, K=K)
    plan = dg.dgemm_plan(1, M, N, K, "nk", "e4m3", out_quant="e4m3_row_amax", act="silu", num_sms=0)
    assert plan["cooperative"] == 1
    q, s = run_workload(w)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([rng.integers(0, M, 200), [0, 2047, 2048, M - 1]])).astype(np.int64)
    ok, msg = requant_ok(q.numpy()[rows], s.numpy()[rows], ref_of(w, rows=rows))
    assert ok, msg
    assert np.all(s.numpy() > 0)   # every row's scale was written


def test_requant_from_bf16_form():
    w = wl.make(2, M=300, N=512, K=640)
    w.bias = torch.from_numpy(np.random.default_rng(6).standard_normal(512).astype(np.float32) * 0.01)
    w.act, w.d_dtype, w.out_quant = "silu", "e4m3", "e4m3_row_amax"
    q, s = run_workload(w)
    ok, msg = requant_ok(q.numpy(), s.numpy(), ref_of(w))
    assert ok, msg


def test_requant_zero_row_gets_unit_scale():
    w = wl.make(5, M=256, N=256, K=256)
    codes = w.A.view(torch.uint8).clone()
    codes[17] = 0                            # row 17 of A is zero -> y = 0 without bias
    w.A = codes.view(torch.float8_e4m3fn)
    w.bias, w.act = None, "none"
    q, s = run_workload(w)
    assert s[17].item() == 1.0 and not q[17].any()
    ok, msg = requant_ok(q.numpy(), s.numpy(), ref_of(w))
    assert ok, msg


def test_repeated_calls_and_streams():
    """The same problem on a side stream, twice, gives identical bits."""
    w = wl.make(3, M=512, N=1024, K=1024)
    g = w.to(dev())
    outs = []
    s = torch.cuda.Stream()
    for _ in range(2):
        D = torch.empty(512, 1024, dtype=torch.bfloat16, device=dev())
        with torch.cuda.stream(s):
            dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, D, b_layout="nk", stream=s)
        outs.append(D)
    s.synchronize()
    assert status_ok(stream=s)
    assert torch.equal(outs[0], outs[1])
