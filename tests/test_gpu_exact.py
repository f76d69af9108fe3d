"""Bit-exact GPU == oracle on small-integer inputs.

With integer operands of magnitude <= 8 every product is exact and every FP32
partial sum stays below 2^24, so the GPU result must equal the oracle exactly
whatever the accumulation order. A wrong shared-memory descriptor, swizzle,
operand layout, TMEM lane mapping or pipeline phase shows up here as a
mismatch instead of hiding inside a tolerance. Shapes are ragged in M, N and K
(tails of every tile dimension) and span several tiles.
"""
import numpy as np
import pytest
import torch

import dense_gemm_persistent_gb300 as dg
import oracle
import workloads as wl
from gpu_util import dev, status_ok

pytestmark = pytest.mark.gpu


def int_bf16(rng, shape, lo=-4, hi=4):
    return torch.from_numpy(rng.integers(lo, hi + 1, size=shape).astype(np.float32)).to(torch.bfloat16)


def int_e4m3(rng, shape, lo=-8, hi=8):
    return torch.from_numpy(rng.integers(lo, hi + 1, size=shape).astype(np.float32)).to(torch.float8_e4m3fn)


def workspace(fp8, M, N, K, layout):
    n = dg.dgemm_workspace_size(fp8, M, N, K, layout)
    return torch.empty(n, dtype=torch.uint8, device=dev()) if n else None


def bf16_case(M, N, K, layout, seed, d_dtype=torch.float32, ws=False):
    rng = np.random.default_rng(seed)
    A = int_bf16(rng, (M, K))
    B = int_bf16(rng, (K, N) if layout == "kn" else (N, K))
    D = torch.empty(M, N, dtype=d_dtype, device=dev())
    wsb = workspace(0, M, N, K, layout) if ws else None
    dg.dgemm_bf16(A.to(dev()), B.to(dev()), D, b_layout=layout, ws=wsb)
    assert status_ok(wsb)
    ref = oracle.bf16_gemm_ref(wl.bits_u16(A), wl.bits_u16(B), layout)
    return D.cpu().to(torch.float64).numpy(), ref


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("bn", [64, 128, 256])
def test_bf16_tile_exact(layout, bn, knobs):
    knobs(tile_n=str(bn))
    got, ref = bf16_case(300, 520, 200, layout, seed=bn)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M", [1, 5, 16, 17, 33, 64])
def test_bf16_swap_exact(layout, M):
    plan = dg.dgemm_plan(0, M, 304, 200, layout, "f32")
    assert plan["swap_ab"] == 1
    got, ref = bf16_case(M, 304, 200, layout, seed=M)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_bf16_exact_bf16_output(layout):
    # the FP32 sums are exact integers, so one rounding to BF16 must give exactly
    # the correctly rounded oracle value
    got, ref = bf16_case(257, 384, 72, layout, seed=3, d_dtype=torch.bfloat16)
    assert np.array_equal(got, oracle.round_bf16(ref))


def fp8_case(M, N, K, layout, seed, scales="pow2", ws=False):
    rng = np.random.default_rng(seed)
    Aq = int_e4m3(rng, (M, K))
    Bq = int_e4m3(rng, (K, N) if layout == "kn" else (N, K))
    if scales == "pow2":   # powers of two keep everything exact
        sa = torch.from_numpy(np.exp2(rng.integers(-3, 4, size=M)).astype(np.float32))
        sb = torch.from_numpy(np.exp2(rng.integers(-3, 4, size=N)).astype(np.float32))
    else:
        sa, sb = torch.ones(M), torch.ones(N)
    D = torch.empty(M, N, dtype=torch.float32, device=dev())
    wsb = workspace(1, M, N, K, layout) if ws else None
    dg.dgemm_fp8_scaled(Aq.to(dev()), Bq.to(dev()), sa.to(dev()), sb.to(dev()), D, b_layout=layout, ws=wsb)
    assert status_ok(wsb)
    ref = oracle.fp8_gemm_ref(wl.codes_u8(Aq), wl.codes_u8(Bq), layout, sa.numpy(), sb.numpy())
    return D.cpu().to(torch.float64).numpy(), ref


@pytest.mark.parametrize("layout,bn", [("nk", 64), ("nk", 128), ("nk", 256), ("kn", 128), ("kn", 256)])
def test_fp8_tile_exact(layout, bn, knobs):
    knobs(tile_n=str(bn))
    got, ref = fp8_case(300, 528, 272, layout, seed=100 + bn)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M", [1, 16, 40, 64])
def test_fp8_swap_exact(layout, M):
    got, ref = fp8_case(M, 400, 272, layout, seed=200 + M)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("kslices", ["2", "1"])
@pytest.mark.parametrize("layout,bn", [("nk", 64), ("nk", 128), ("kn", 64), ("kn", 128)])
@pytest.mark.parametrize("kblocks", [1, 3, 6])
def test_single_cta_two_slice_stages_exact(layout, bn, kblocks, kslices, knobs):
    """Single-CTA 128x64 and 128x128 tiles with one or two 128-byte K slices per
    stage (two: each operand of a stage one 3-D TMA copy; with an odd slice count
    the last stage's second slice is zero-filled), ragged M and N, several tiles
    per CTA; integer inputs, so the result is exact."""
    knobs(tile_n=str(bn), cta_pair="0", kslices=kslices)
    M, N, K = 1320, 1984, 64 * kblocks
    plan = dg.dgemm_plan(0, M, N, K, layout, "f32")
    assert (plan["cta_group"], plan["tile_n"], plan["k_slices"]) == (1, bn, int(kslices))
    got, ref = bf16_case(M, N, K, layout, seed=900 + 10 * bn + kblocks)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("kslices", ["2", "1"])
@pytest.mark.parametrize("layout,bn", [("nk", 64), ("nk", 128), ("kn", 128)])
@pytest.mark.parametrize("kblocks", [1, 3, 6])
def test_fp8_single_cta_two_slice_stages_exact(layout, bn, kblocks, kslices, knobs):
    """The same for E4M3 (128-element K slices) with power-of-two scales."""
    knobs(tile_n=str(bn), cta_pair="0", kslices=kslices)
    M, N, K = 1320, 1920, 128 * kblocks
    plan = dg.dgemm_plan(1, M, N, K, layout, "f32")
    assert (plan["cta_group"], plan["tile_n"], plan["k_slices"]) == (1, bn, int(kslices))
    got, ref = fp8_case(M, N, K, layout, seed=950 + 10 * bn + kblocks)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("kblocks", [1, 2, 3, 4, 5, 9, 13])
def test_odd_k_block_counts_exact(kblocks, knobs):
    """Odd numbers of K slices expose pipeline-phase bugs (DeepGEMM write-up,
    czchanglian.com/news/51329, §4.3); 640 tiles of 128x64 over at most 152 CTAs
    also carry the stage and accumulator phases across several tiles per CTA."""
    knobs(tile_n="64")
    got, ref = bf16_case(2560, 2048, 64 * kblocks, "nk", seed=kblocks)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("kblocks", [1, 3, 4, 5, 7])
def test_odd_k_block_counts_wide_tile_exact(kblocks, knobs):
    knobs(tile_n="256")
    got, ref = bf16_case(2560, 4096, 64 * kblocks, "kn", seed=50 + kblocks)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("M,kblocks", [(16, 37), (16, 5), (40, 23), (64, 9)])
def test_k_group_promotion_exact(M, kblocks):
    """The small-M kernel splits K into several tensor-core accumulators summed in
    FP32 (uneven splits here); integer inputs keep the result exact."""
    K = 64 * kblocks
    plan = dg.dgemm_plan(0, M, 304, K, "nk", "f32")
    tmem = 256 if plan["smem_bytes"] <= 115712 else 512   # compact footprint: half the Tensor Memory
    assert plan["swap_ab"] == 1 and plan["k_groups"] == min(kblocks, tmem // plan["tile_n"])
    got, ref = bf16_case(M, 304, K, "nk", seed=300 + kblocks)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("pair,halves", [("0", "1"), ("1", "0"), ("1", "1")])
def test_bf16_wide_tile_single_and_pair_exact(layout, pair, halves, knobs):
    """128 x 256 tiles on one CTA and 256 x 256 tiles on a CTA pair (cta_group::2),
    with M, N and K tails; the pair's 12 tiles run whole, or (all of them
    being the last wave's) as 24 halves of 128 columns."""
    knobs(cta_pair=pair)
    knobs(tile_n="256")
    knobs(tail_halves=halves)
    plan = dg.dgemm_plan(0, 700, 776, 328, layout, "f32")
    assert plan["cta_group"] == (2 if pair == "1" else 1) and plan["tile_n"] == 256
    assert plan["tail_halves"] == (1 if pair + halves == "11" else 0)
    got, ref = bf16_case(700, 776, 328, layout, seed=400 + int(pair))
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("pair,halves", [("0", "1"), ("1", "0"), ("1", "1")])
def test_fp8_wide_tile_single_and_pair_exact(layout, pair, halves, knobs):
    """As above for E4M3; an MN-major E4M3 B (128-column atoms) has no half
    tiles."""
    knobs(cta_pair=pair)
    knobs(tile_n="256")
    knobs(tail_halves=halves)
    plan = dg.dgemm_plan(1, 700, 784, 400, layout, "f32")
    assert plan["cta_group"] == (2 if pair == "1" else 1) and plan["tile_n"] == 256
    assert plan["tail_halves"] == (1 if pair + halves == "11" and layout == "nk" else 0)
    got, ref = fp8_case(700, 784, 400, layout, seed=500 + int(pair))
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("kslices", ["2", "1"])
@pytest.mark.parametrize("kblocks", [1, 5, 6, 7, 13])
def test_pair_phases_across_many_tiles_exact(kblocks, kslices, knobs):
    """CTA pairs with several tiles each (4096 x 8192 -> 512 tiles over <= 76 pairs)
    and K-slice counts around the ring depth (6 stages of one slice, or 3 of
    two slices, an odd count leaving the last stage's second slice beyond K)."""
    knobs(kslices=kslices)
    plan = dg.dgemm_plan(0, 4096, 8192, 64 * kblocks, "nk", "f32")
    assert plan["cta_group"] == 2 and plan["k_slices"] == int(kslices)
    got, ref = bf16_case(4096, 8192, 64 * kblocks, "nk", seed=600 + kblocks)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("seg_first", ["1", "0"])
@pytest.mark.parametrize("shape,layout,pair", [((4096, 4096, 1024), "kn", "1"), ((4096, 4096, 1024), "nk", "0"),
                                               ((2304, 2816, 1024), "nk", "1"), ((2560, 2048, 1024), "kn", "0"),
                                               ((4000, 1288, 1024), "kn", "1")])
def test_tail_split_exact(shape, layout, pair, seg_first, knobs):
    """The last partial wave's tiles split along K (FP32 partials in the
    workspace, each segment finishing its share of the units): still
    bit-exact, with the segments run before the whole tiles (at the raster's
    start) and after them (at its end)."""
    knobs(seg_first=seg_first)
    knobs(cta_pair=pair)
    knobs(tail_split="force")   # split even these short tiles
    knobs(tail_halves="0")      # along K, not N
    M, N, K = shape
    plan = dg.dgemm_plan(0, M, N, K, layout, "f32")
    assert plan["tail_split"] >= 2
    got, ref = bf16_case(M, N, K, layout, seed=700 + K, ws=True)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("seg_first", ["1", "0"])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_tail_split_fp8_exact(layout, seg_first, knobs):
    knobs(seg_first=seg_first)
    knobs(tail_split="force")
    knobs(tail_halves="0")
    plan = dg.dgemm_plan(1, 4096, 11008, 2048, layout, "f32")
    assert plan["tail_split"] >= 2
    got, ref = fp8_case(4096, 11008, 2048, layout, seed=800, ws=True)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


def test_tail_split_repeated_calls_reuse_workspace(knobs):
    """Arrival counters are tagged with a per-launch epoch: the same workspace,
    even filled with garbage first, serves consecutive calls."""
    knobs(tail_split="force")
    knobs(tail_halves="0")
    M, N, K = 4096, 4096, 1024
    ws = workspace(0, M, N, K, "nk")
    ws.fill_(0xA5)
    rng = np.random.default_rng(5)
    for i in range(3):
        A = int_bf16(rng, (M, K)); B = int_bf16(rng, (N, K))
        D = torch.empty(M, N, dtype=torch.float32, device=dev())
        dg.dgemm_bf16(A.to(dev()), B.to(dev()), D, b_layout="nk", ws=ws)
        assert status_ok(ws)
        ref = oracle.bf16_gemm_ref(wl.bits_u16(A), wl.bits_u16(B), "nk")
        assert np.array_equal(D.cpu().double().numpy(), ref)


@pytest.mark.parametrize("kslices", ["2", "1"])
@pytest.mark.parametrize("shape,layout", [((4096, 4096, 1024), "kn"), ((4096, 4096, 1024), "nk"),
                                          ((4000, 1288, 1024), "kn"), ((2304, 2816, 2000), "nk")])
def test_tail_halves_exact(shape, layout, kslices, knobs):
    """The last partial wave's CTA-pair tiles, too short to split along K, run
    as two 256 x 128 halves each (N = 128 MMAs over the whole K range, half of
    B loaded): bit-exact, ragged edges included."""
    knobs(kslices=kslices)
    M, N, K = shape
    plan = dg.dgemm_plan(0, M, N, K, layout, "f32")
    assert plan["cta_group"] == 2 and plan["tail_halves"] == 1 and plan["tail_tiles"] > 0
    assert plan["workspace_bytes"] == 0
    got, ref = bf16_case(M, N, K, layout, seed=1000 + K)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("shape", [(4096, 11008, 1024), (4000, 10900, 640)])
def test_tail_halves_fp8_exact(shape):
    M, N, K = shape
    plan = dg.dgemm_plan(1, M, N, K, "nk", "f32")
    assert plan["cta_group"] == 2 and plan["tail_halves"] == 1 and plan["tail_tiles"] > 0
    got, ref = fp8_case(M, N, K, "nk", seed=1100 + K)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


def test_tail_split_default_rule_on_long_tiles(knobs):
    """Without forcing, a tail is split along K only for long tiles: 4096^3 BF16
    (64 K slices) splits its 28-tile tail, the same shape at K = 2048 does not."""
    knobs(tail_halves="0")
    assert dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16")["tail_split"] >= 2
    assert dg.dgemm_plan(0, 4096, 4096, 2048, "kn", "bf16")["tail_split"] == 1
    got, ref = bf16_case(2304, 2816, 3072, "nk", seed=900, ws=True)
    assert dg.dgemm_plan(0, 2304, 2816, 3072, "nk", "f32")["tail_split"] >= 2
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("cluster", ["1", "0"])
@pytest.mark.parametrize("shape,layout", [((1024, 1024, 4096), "nk"), ((1024, 1000, 2048), "kn"),
                                          ((520, 776, 1600), "nk")])
def test_split_k_underfilled_tile_exact(shape, layout, cluster, knobs):
    """Grids that do not fill the GPU split every tile along K (up to 4
    segments). Each segment finishes its share of the tile's 32-column units,
    adding the other segments' partials to its own accumulator from TMEM: read
    from the peers' shared memory when the segments form a cluster, else from
    the workspace."""
    knobs(cluster_split=cluster)
    M, N, K = shape
    plan = dg.dgemm_plan(0, M, N, K, layout, "f32")
    assert plan["tail_split"] >= 2 and plan["tail_tiles"] == plan["num_tiles"]
    assert plan["cluster_split"] == int(cluster)
    got, ref = bf16_case(M, N, K, layout, seed=1000 + K, ws=True)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("cluster", ["1", "0"])
@pytest.mark.parametrize("M,layout", [(1, "nk"), (16, "nk"), (5, "kn"), (40, "nk"), (64, "kn")])
def test_split_k_small_m_exact(M, layout, cluster, knobs):
    """Small-M (transposed) tiles split along K, with the K groups of each
    segment inside the segment's range."""
    knobs(cluster_split=cluster)
    N, K = 4096, 4096
    plan = dg.dgemm_plan(0, M, N, K, layout, "f32")
    assert plan["swap_ab"] == 1 and plan["tail_split"] >= 2 and plan["k_groups"] > 1
    assert plan["cluster_split"] == int(cluster)
    got, ref = bf16_case(M, N, K, layout, seed=1100 + M, ws=True)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("cluster", ["1", "0"])
@pytest.mark.parametrize("M", [1, 48, 256])
def test_split_k_fp8_exact(M, cluster, knobs):
    knobs(cluster_split=cluster)
    N, K = 2048 if M < 256 else 512, 8192
    plan = dg.dgemm_plan(1, M, N, K, "nk", "f32")
    assert plan["tail_split"] >= 2 and plan["cluster_split"] == int(cluster)
    got, ref = fp8_case(M, N, K, "nk", seed=1200 + M, ws=True)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


def sampled_rows(M, tile_m, seed):
    """A row in every tile row, plus the first and last rows."""
    rng = np.random.default_rng(seed)
    pick = {0, M - 1} | {int(rng.integers(t0, min(M, t0 + tile_m))) for t0 in range(0, M, tile_m)}
    return np.array(sorted(pick), dtype=np.int64)


@pytest.mark.parametrize("case", ["tail_split_plain", "underfill_split_cooperative"])
def test_split_tiles_while_another_stream_holds_the_sms(case, knobs):
    """A split-tile GEMM launched while a large GEMM on another stream still
    occupies every SM, so its CTAs become resident a few at a time as the
    other kernel's CTAs leave. The tail split's plain launch never lets a
    segment wait for one that has not started; the cooperative launch of the
    under-filled split-K waits until its whole grid fits. Both must finish,
    bit-exact, with a clean status."""
    rng = np.random.default_rng(1500)
    # the occupying GEMM: 8192^3 BF16 (every SM busy for ~0.6 ms), on a side stream
    Ab = torch.randn(8192, 8192, device=dev()).to(torch.bfloat16)
    Bb = torch.randn(8192, 8192, device=dev()).to(torch.bfloat16)
    Db = torch.empty(8192, 8192, dtype=torch.bfloat16, device=dev())
    wsb = workspace(0, 8192, 8192, 8192, "nk")
    side = torch.cuda.Stream()
    if case == "tail_split_plain":
        M, N, K, layout = 4096, 4096, 4096, "kn"
    else:
        knobs(cluster_split="0")
        M, N, K, layout = 1024, 1024, 4096, "nk"
    plan = dg.dgemm_plan(0, M, N, K, layout, "f32", num_sms=0)
    assert plan["tail_split"] >= 2 and plan["cluster_split"] == 0
    assert plan["cooperative"] == (0 if case == "tail_split_plain" else 1)
    A = int_bf16(rng, (M, K))
    B = int_bf16(rng, (K, N) if layout == "kn" else (N, K))
    Ad, Bd = A.to(dev()), B.to(dev())
    D = torch.empty(M, N, dtype=torch.float32, device=dev())
    ws = workspace(0, M, N, K, layout)
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(side):
            for _ in range(2):
                dg.dgemm_bf16(Ab, Bb, Db, b_layout="nk", ws=wsb, stream=side)
        dg.dgemm_bf16(Ad, Bd, D, b_layout=layout, ws=ws)
    torch.cuda.synchronize()
    assert status_ok(ws) and status_ok(wsb, stream=side)
    rows = sampled_rows(M, plan["tile_m"], 1500)
    ref = oracle.bf16_gemm_ref(wl.bits_u16(A), wl.bits_u16(B), layout, rows=rows)
    got = D.cpu().double().numpy()[rows]
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"
