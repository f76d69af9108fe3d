"""FP8 GEMM with per-K-group scales (one FP32 scale per row of A and per output
channel of B for every K group), GPU against the oracle.

Bit-exact cases: small-integer E4M3 codes and power-of-two scales keep every
product, group sum and scaled sum exact in FP32, so the result must equal the
oracle exactly whatever the order of accumulation; they cover every kernel
variant (tile widths, CTA pairs, both B layouts, the small-M transposed form),
ragged K (a partial last K slice and a partial last group), and K segments of
split tiles that start inside a scale group. Recipe cases use the per-group
quantised workload at sizes the oracle finishes in seconds, with the BF16
one-ulp bound.
"""
import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from gpu_util import dev, run_workload, status_ok, to_f64
from test_gpu_parity import ref_of
from tolerances import bf16_ulp_ok, c1_ok

pytestmark = pytest.mark.gpu


def grouped_int_case(M, N, K, g, layout, seed, d_dtype=torch.float32, b_block=1):
    rng = np.random.default_rng(seed)
    G = -(-K // g)
    Aq = torch.from_numpy(rng.integers(-4, 5, size=(M, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    shape_b = (K, N) if layout == "kn" else (N, K)
    Bq = torch.from_numpy(rng.integers(-4, 5, size=shape_b).astype(np.float32)).to(torch.float8_e4m3fn)
    sa = torch.from_numpy(np.exp2(rng.integers(-1, 2, size=(G, M))).astype(np.float32))
    sb = torch.from_numpy(np.exp2(rng.integers(-1, 2, size=(G, -(-N // b_block)))).astype(np.float32))
    n = dg.dgemm_workspace_size(1, M, N, K, layout)
    ws = torch.empty(n, dtype=torch.uint8, device=dev()) if n else None
    D = torch.empty(M, N, dtype=d_dtype, device=dev())
    dg.dgemm_fp8_scaled(Aq.to(dev()), Bq.to(dev()), sa.to(dev()), sb.to(dev()), D, b_layout=layout, k_group=g,
                        b_block=b_block, ws=ws)
    assert status_ok(ws)
    ref = oracle.fp8_gemm_ref(wl.codes_u8(Aq), wl.codes_u8(Bq), layout, sa.numpy(), sb.numpy(), k_group=g,
                              b_block=b_block)
    return D.cpu().to(torch.float64).numpy(), ref


@pytest.mark.parametrize("g", [128, 384])
@pytest.mark.parametrize("layout,bn,pair", [("nk", 64, "0"), ("nk", 128, "0"), ("nk", 256, "0"), ("nk", 256, "1"),
                                            ("kn", 128, "0"), ("kn", 256, "0"), ("kn", 256, "1")])
def test_grouped_tile_exact(layout, bn, pair, g, knobs):
    """Every tile variant, with the plan checked to use it."""
    knobs(tile_n=str(bn))
    knobs(cta_pair=pair)
    knobs(tail_split="0")
    plan = dg.dgemm_plan(1, 300, 528, 1040, layout, "f32", k_group=g, num_sms=0)
    assert (plan["tile_n"], plan["cta_group"], plan["k_groups"]) == (bn, 2 if pair == "1" else 1, -(-1040 // g))
    # K = 1040: nine K slices, the last one partial; groups of 128 or 384
    got, ref = grouped_int_case(300, 528, 1040, g, layout, seed=bn + g + int(pair))
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("g", [128, 256])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M", [1, 16, 40, 64])
def test_grouped_small_m_exact(layout, M, g):
    assert dg.dgemm_plan(1, M, 400, 1040, layout, "f32")["swap_ab"] == 1
    got, ref = grouped_int_case(M, 400, 1040, g, layout, seed=M + g)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("cluster", ["1", "0"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 4096), (16, 1024, 4096)])
def test_grouped_split_k_segments_inside_groups_exact(M, N, K, cluster, knobs):
    """Under-filled grids split every tile into K segments of 8 slices; with
    groups of 3 slices (384 elements) most segments start inside a group."""
    knobs(cluster_split=cluster)
    plan = dg.dgemm_plan(1, M, N, K, "nk", "f32", k_group=384, num_sms=0)
    assert plan["tail_split"] > 1 and plan["cluster_split"] == int(cluster)
    got, ref = grouped_int_case(M, N, K, 384, "nk", seed=K + M)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("seg_first", ["1", "0"])
def test_grouped_tail_split_exact(seg_first, knobs):
    knobs(seg_first=seg_first)
    knobs(cta_pair="0")
    knobs(tile_n="64")
    knobs(tail_split="force")
    M, N, K = 1280, 1024, 2064     # 160 tiles of 128 x 64: the last 8 are split
    plan = dg.dgemm_plan(1, M, N, K, "nk", "f32", k_group=384, num_sms=0)
    assert plan["tail_tiles"] > 0 and plan["tail_split"] == 2
    got, ref = grouped_int_case(M, N, K, 384, "nk", seed=7)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("g", [128, 256])
@pytest.mark.parametrize("layout,bn,pair", [("nk", 64, "0"), ("nk", 128, "0"), ("nk", 256, "0"), ("nk", 256, "1"),
                                            ("kn", 128, "0"), ("kn", 256, "1")])
def test_block_scaled_tile_exact(layout, bn, pair, g, knobs):
    """Weights scaled per (128-channel block, K group): each warp's columns
    share one scale per group (one fused multiply-add per output). N = 400
    ends inside the fourth block."""
    knobs(tile_n=str(bn))
    knobs(cta_pair=pair)
    knobs(tail_split="0")
    got, ref = grouped_int_case(300, 400, 1040, g, layout, seed=bn + g + 7 * int(pair), b_block=128)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M", [1, 16, 64])
def test_block_scaled_small_m_exact(layout, M):
    """The transposed small-M form: output channels run along the MMA's rows,
    so the weight block scale is per row (one per 128 rows of the tile)."""
    assert dg.dgemm_plan(1, M, 528, 1040, layout, "f32")["swap_ab"] == 1
    got, ref = grouped_int_case(M, 528, 1040, 128, layout, seed=M + 3, b_block=128)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("cluster", ["1", "0"])
def test_block_scaled_split_k_exact(cluster, knobs):
    knobs(cluster_split=cluster)
    plan = dg.dgemm_plan(1, 256, 512, 4096, "nk", "f32", k_group=384, num_sms=0)
    assert plan["tail_split"] > 1 and plan["cluster_split"] == int(cluster)
    got, ref = grouped_int_case(256, 512, 4096, 384, "nk", seed=31, b_block=128)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("shape,layout", [((300, 528, 1024), "nk"), ((257, 512, 1024), "kn"),
                                          ((16, 4224, 1024), "nk")])
def test_block_scaled_recipe(shape, layout):
    w = wl.fp8_grouped(*shape, k_group=128, b_layout=layout, seed=sum(shape) + 1, b_block=128)
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


def test_block_scaled_needs_k_group():
    A = torch.zeros(16, 128, dtype=torch.float8_e4m3fn, device=dev())
    B = torch.zeros(128, 128, dtype=torch.float8_e4m3fn, device=dev())
    s = torch.ones(1, device=dev())
    D = torch.empty(16, 128, device=dev())
    with pytest.raises(dg.DgemmError):
        dg.dgemm_fp8_scaled(A, B, s, s, D, b_layout="nk", k_group=0, b_block=128)


def test_grouped_bf16_output_rounds_once():
    got, ref = grouped_int_case(257, 384, 528, 128, "nk", seed=9, d_dtype=torch.bfloat16)
    assert np.array_equal(got, oracle.round_bf16(ref))


@pytest.mark.parametrize("shape,g,layout", [((300, 528, 1024), 128, "nk"), ((1000, 1008, 2048), 128, "nk"),
                                            ((257, 512, 1024), 256, "kn"), ((16, 4224, 1024), 128, "nk"),
                                            ((1, 4224, 1024), 128, "kn"), ((600, 1024, 3072), 512, "nk")])
def test_grouped_recipe(shape, g, layout):
    w = wl.fp8_grouped(*shape, k_group=g, b_layout=layout, seed=sum(shape))
    D, _ = run_workload(w)
    ok, msg = bf16_ulp_ok(to_f64(D), ref_of(w))
    assert ok, msg


def test_grouped_with_c_bias_activation_f32_output():
    w = wl.fp8_grouped(200, 400, 512, k_group=128, seed=11, d_dtype="f32")
    rng = np.random.default_rng(12)
    w.C = torch.from_numpy(rng.standard_normal((200, 400)).astype(np.float32))
    w.alpha, w.beta = 1.25, 0.5
    w.bias = torch.from_numpy(rng.standard_normal(400).astype(np.float32))
    w.act = "silu"
    D, _ = run_workload(w)
    ok, msg = c1_ok(to_f64(D), ref_of(w), w.K)
    assert ok, msg


def test_grouped_k_zero_gives_beta_c():
    M, N = 130, 256
    C = torch.randn(M, N, device=dev())
    D = torch.empty(M, N, device=dev())
    z8 = torch.empty(M, 0, dtype=torch.float8_e4m3fn, device=dev())
    zb = torch.empty(N, 0, dtype=torch.float8_e4m3fn, device=dev())
    sa, sb = torch.ones(M, device=dev()), torch.ones(N, device=dev())   # no K groups: never read
    dg.dgemm_fp8_scaled(z8, zb, sa, sb, D, b_layout="nk", k_group=128, C=C, beta=2.0)
    assert status_ok()
    assert torch.equal(D, 2.0 * C)
