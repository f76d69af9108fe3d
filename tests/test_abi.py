"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and the host-side logic (validation, planning, workspace
sizes, status strings) behaves as documented. No compute call is made."""
import ctypes
import os
import re

import pytest

import dense_gemm_persistent_gb300 as dg
from dense_gemm_persistent_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgemm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return dg.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dgemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(["dgemm_bf16", "dgemm_fp8_scaled", "dgemm_fp8_blockscaled", "dgemm_workspace_size",
                            "dgemm_plan",
                            "dgemm_status_string", "dgemm_query_device_status",
                            "dgemm_overrides_init", "dgemm_set_overrides", "dgemm_get_overrides",
                            "dgemm_fp8_rowquant_noalloc"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_status_strings(lib):
    for code in range(8):
        s = dg.dgemm_status_string(code)
        assert s and s != "unknown status"
    assert dg.dgemm_status_string(99) == "unknown status"


def call_bf16(lib, **over):
    args = dict(A=16, B=16, bl=1, C=None, c_dt=0, D=16, d_dt=1, M=128, N=128, K=128, alpha=1.0, beta=0.0,
                epi=None, ws=None, ws_bytes=0, stream=None)
    args.update(over)
    return lib.dgemm_bf16(args["A"], args["B"], args["bl"], args["C"], args["c_dt"], args["D"], args["d_dt"],
                          args["M"], args["N"], args["K"], args["alpha"], args["beta"], args["epi"], args["ws"],
                          args["ws_bytes"], args["stream"])


def test_argument_errors_return_before_any_device_call(lib):
    # These return synchronously from validation (no CUDA call is reached).
    assert call_bf16(lib, M=-1) == 1
    assert call_bf16(lib, bl=7) == 1
    assert call_bf16(lib, d_dt=9) == 1
    assert call_bf16(lib, K=100) == 3                 # 200-byte A rows: not a multiple of 16
    assert call_bf16(lib, bl=0, N=100) == 3           # K x N B with 200-byte rows
    assert call_bf16(lib, A=8) == 3                   # misaligned pointer
    assert call_bf16(lib, A=None) == 1                # NULL operand
    assert call_bf16(lib, beta=1.0) == 1              # beta != 0 needs C
    assert call_bf16(lib, d_dt=2) == 1                # E4M3 output needs the requant epilogue
    epi = _lib.Epilogue(None, 0, 1, None)             # requant without a row-scale pointer
    assert call_bf16(lib, d_dt=2, epi=ctypes.byref(epi)) == 1
    epi = _lib.Epilogue(None, 0, 1, 16)
    assert call_bf16(lib, d_dt=2, epi=ctypes.byref(epi)) == 4   # no workspace
    epi = _lib.Epilogue(None, 9, 0, None)
    assert call_bf16(lib, epi=ctypes.byref(epi)) == 1           # bad activation
    # empty problems are a no-op and need no device
    assert call_bf16(lib, M=0) == 0 and call_bf16(lib, N=0) == 0
    # fp8 per-K-group scales: groups of whole 128-element K slices, no requantisation
    def fp8(k_group, epi=None, d_dt=1):
        return lib.dgemm_fp8_scaled(16, 16, 1, 16, 16, k_group, None, 0, 16, d_dt, 128, 128, 256, 1.0, 0.0, epi,
                                    None, 0, None)
    assert fp8(-1) == 1
    assert fp8(64) == 2 and fp8(200) == 2
    epi = _lib.Epilogue(None, 0, 1, 16)
    assert fp8(128, ctypes.byref(epi), d_dt=2) == 2
    # block-scaled weights: a per-group form (k_group > 0), same group rules
    def blk(k_group):
        return lib.dgemm_fp8_blockscaled(16, 16, 1, 16, 16, k_group, None, 0, 16, 1, 128, 128, 256, 1.0, 0.0,
                                         None, None, 0, None)
    assert blk(0) == 1 and blk(-128) == 1
    assert blk(64) == 2


def test_workspace_sizes(lib, knobs):
    # requantisation: status header, barrier header, row maxima, BF16 stash;
    # 1024 tiles on 76 pairs leave 36 for the last wave, split in halves: plus
    # counters and one 256 x 256 FP32 partial per unit
    base = 256 + 256 + 8192 * 4 + 8192 * 8192 * 2
    ws = dg.dgemm_workspace_size(1, 8192, 8192, 8192, "nk", out_quant="e4m3_row_amax")
    assert ws == base + 256 * ((76 * 2 * 8 * 8 + 255) // 256) + 76 * 2 * 128 * 256 * 4
    # tail splitting: 256 tiles on 76 pairs leave 28 tiles for the last wave,
    # each split in two K halves on 56 pairs; the workspace bounds one 256 x 256
    # FP32 partial per unit plus the counters
    p = dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16", num_sms=152)
    assert (p["tail_tiles"], p["tail_units"], p["tail_split"]) == (28, 56, 2)
    assert p["workspace_bytes"] == 256 + 256 * ((76 * 2 * 8 * 8 + 255) // 256) + 76 * 2 * 128 * 256 * 4
    # FP8 4096 x 11008 x 4096 has 32 K slices per tile: too short to split along
    # K; its 4 leftover tiles run as 8 N halves instead, with no workspace
    p = dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", num_sms=152)
    assert (p["tail_tiles"], p["tail_split"], p["tail_halves"], p["workspace_bytes"]) == (4, 1, 1, 0)
    knobs(tail_halves="0")
    assert dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", num_sms=152)["tail_halves"] == 0
    knobs(tail_split="0")
    assert dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16", num_sms=152)["workspace_bytes"] == 0
    assert dg.dgemm_workspace_size(1, 8192, 8192, 8192, "nk", out_quant="e4m3_row_amax") == base


def test_plans_for_the_five_workloads(lib):
    p1 = dg.dgemm_plan(0, 512, 512, 512, "kn", "f32", num_sms=152)
    assert p1["swap_ab"] == 0 and p1["grid"] <= 152 and p1["tile_n"] == 64
    p2 = dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16", num_sms=152)
    assert (p2["cta_group"], p2["tile_m"], p2["tile_n"]) == (2, 256, 256)
    # two 128-byte K slices per stage: 3 stages of 2 x 32 KB per CTA
    assert p2["num_tiles"] == 256 and p2["grid"] == 152 and (p2["stages"], p2["k_slices"]) == (3, 2)
    assert (p2["tail_tiles"], p2["tail_split"], p2["tail_units"]) == (28, 2, 56)   # 3 full waves + 28 tiles in K halves
    p3 = dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", num_sms=152)
    assert p3["cta_group"] == 2 and p3["num_tiles"] == 16 * 43 and p3["grid"] == 152
    p4 = dg.dgemm_plan(0, 16, 18432, 7168, "nk", "bf16", num_sms=152)
    assert p4["swap_ab"] == 1 and p4["tile_n"] == 16 and p4["num_tiles"] == 144 and p4["grid"] == 144
    p5 = dg.dgemm_plan(1, 8192, 8192, 8192, "nk", "e4m3", out_quant="e4m3_row_amax", act="silu", num_sms=152)
    assert p5["cooperative"] == 1 and p5["tile_n"] == 256 and p5["cta_group"] == 2 and p5["num_tiles"] == 32 * 32
    for p in (p1, p2, p3, p4, p5):
        assert p["smem_bytes"] <= 232448 and p["stages"] >= 2


def test_plan_of_per_group_scales(lib):
    """The plan query takes k_group: K groups of 128 on workload 3's shape are
    32 scale groups on the single-CTA 128 x 256 kernel with 3 stages (groups of
    one or two K slices skip CTA pairs; the scale ring takes shared memory);
    groups of 512 go back to the pair's 5 stages; invalid groups fail as the
    call would."""
    p = dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", k_group=128, num_sms=152)
    assert (p["k_groups"], p["cta_group"], p["tile_n"], p["stages"]) == (32, 1, 256, 3)
    p = dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", k_group=256, num_sms=152)
    assert (p["k_groups"], p["cta_group"], p["tile_n"]) == (16, 1, 256)
    p = dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", k_group=512, num_sms=152)
    assert (p["k_groups"], p["cta_group"], p["tile_n"], p["stages"]) == (8, 2, 256, 5)
    p = dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", num_sms=152)
    assert (p["stages"], p["k_slices"]) == (3, 2)   # per-row scales: two K slices per stage
    assert p["k_slices"] * p["stages"] * 32 == 2 * 96   # the same bytes in flight as 6 single slices
    with pytest.raises(dg.DgemmError):
        dg.dgemm_plan(1, 4096, 11008, 4096, "nk", "bf16", k_group=64, num_sms=152)


def test_split_exchange_launch_modes(lib, knobs):
    """Split tiles that exchange partials through the workspace: the under-filled
    grid's split-K (the exchange ends the kernel) is launched cooperatively, so
    its segments may wait for each other; the tail split of 4096^3 (exchange
    overlapped by whole tiles) is a plain launch, where no segment waits for
    one that may not have started. Cluster splits need neither."""
    p = dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16", num_sms=152)
    assert p["tail_split"] >= 2 and p["cooperative"] == 0
    knobs(cluster_split="0")
    p = dg.dgemm_plan(0, 1024, 1024, 4096, "nk", "bf16", num_sms=152)
    assert p["tail_split"] >= 2 and p["cluster_split"] == 0 and p["cooperative"] == 1
    knobs(cluster_split="1")
    p = dg.dgemm_plan(0, 1024, 1024, 4096, "nk", "bf16", num_sms=152)
    assert p["cluster_split"] == 1 and p["cooperative"] == 0
    knobs(cooperative="1")
    assert dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16", num_sms=152)["cooperative"] == 1
    knobs(cooperative="0")
    p5 = dg.dgemm_plan(1, 8192, 8192, 8192, "nk", "e4m3", out_quant="e4m3_row_amax", num_sms=152)
    assert p5["cooperative"] == 0


def test_overrides_validation_and_defaults(lib):
    d = dg.get_overrides()
    assert d == {"tile_n": 0, "cta_pair": -1, "tail_split": -1, "tail_halves": -1, "cluster_split": -1,
                 "seg_first": -1, "raster_group": 0, "cooperative": -1, "kslices": -1, "wait_limit_ns": 0,
                 "stall_after_loads": -1}
    for bad in ({"cta_pair": 2}, {"tail_halves": 1}, {"cooperative": -2}, {"wait_limit_ns": -1},
                {"stall_after_loads": -5}, {"tile_n": -64}):
        with pytest.raises(dg.DgemmError):
            dg.set_overrides(**bad)
        assert dg.get_overrides() == d          # a refused set changes nothing
    with dg.overrides(tile_n=128, wait_limit_ns=5_000_000):
        assert dg.get_overrides()["tile_n"] == 128
    assert dg.get_overrides() == d


ENV_PROBE = r"""
import sys
sys.path.insert(0, {root!r})
import dense_gemm_persistent_gb300 as dg
p = dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16", num_sms=152)
print(p["tile_n"], p["cta_group"], dg.get_overrides()["tile_n"])
"""


@pytest.mark.parametrize("opt_in,expect", [(None, "256 2 0"), ("1", "128 1 128")])
def test_environment_knobs_need_the_opt_in(lib, opt_in, expect):
    """A stray DGEMM_TILE_N in the environment changes nothing; with
    DGEMM_ENV_OVERRIDES=1 it is read once, at the first call."""
    import subprocess
    import sys
    env = dict(os.environ, DGEMM_TILE_N="128")
    env.pop("DGEMM_ENV_OVERRIDES", None)
    if opt_in:
        env["DGEMM_ENV_OVERRIDES"] = opt_in
    r = subprocess.run([sys.executable, "-c", ENV_PROBE.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == expect


def test_tile_width_and_pair_overrides(lib, knobs):
    knobs(tile_n="128")
    assert dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16")["tile_n"] == 128
    knobs(tile_n="96")     # no such variant: ignored
    assert dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16")["tile_n"] == 256
    knobs(tile_n=None)
    knobs(cta_pair="0")
    p = dg.dgemm_plan(0, 4096, 4096, 4096, "kn", "bf16")
    assert (p["cta_group"], p["tile_m"], p["tile_n"], p["num_tiles"], p["stages"]) == (1, 128, 256, 512, 4)


C_CALLER = r"""
/* A plain C11 caller of the library: the header must compile as C, and the
 * host-only entry points must link and behave without Python or a GPU. */
#include <stdio.h>
#include <string.h>
#include "dgemm.h"

int main(void) {
    dgemm_plan_t plan;
    memset(&plan, 0, sizeof plan);
    /* BF16 4096^3, B stored K x N, BF16 out, on a 152-SM GPU */
    dgemm_status_t st = dgemm_plan(0, 4096, 4096, 4096, DGEMM_B_KN, DGEMM_BF16, NULL, 0, 152, &plan);
    printf("plan %d %d %d %d %d %d\n", (int)st, plan.tile_m, plan.tile_n, plan.cta_group, plan.num_tiles,
           plan.swap_ab);
    /* decode shape: small M runs transposed */
    st = dgemm_plan(0, 16, 18432, 7168, DGEMM_B_NK, DGEMM_BF16, NULL, 0, 152, &plan);
    printf("decode %d %d\n", (int)st, plan.swap_ab);
    dgemm_epilogue_t epi = {NULL, DGEMM_ACT_SILU, DGEMM_QUANT_E4M3_ROW_AMAX, NULL};
    printf("ws %zu\n", dgemm_workspace_size(1, 256, 512, 384, DGEMM_B_NK, &epi));
    /* an argument error returns before any device call */
    st = dgemm_bf16(NULL, NULL, DGEMM_B_KN, NULL, DGEMM_F32, NULL, DGEMM_BF16, 128, 128, 128, 1.0f, 0.0f,
                    NULL, NULL, 0, NULL);
    printf("null %d %s\n", (int)st, dgemm_status_string(st));
    /* planner overrides: 128-wide single-CTA tiles, then the defaults again */
    dgemm_overrides_t o;
    dgemm_overrides_init(&o);
    o.tile_n = 128;
    st = dgemm_set_overrides(&o);
    dgemm_status_t st2 = dgemm_plan(0, 4096, 4096, 4096, DGEMM_B_KN, DGEMM_BF16, NULL, 0, 152, &plan);
    printf("override %d %d %d %d\n", (int)st, (int)st2, plan.tile_n, plan.cta_group);
    dgemm_set_overrides(NULL);
    dgemm_plan(0, 4096, 4096, 4096, DGEMM_B_KN, DGEMM_BF16, NULL, 0, 152, &plan);
    printf("restored %d\n", plan.tile_n);
    /* the status of a workspace's calls (no GPU here: the stream sync fails) */
    st = dgemm_query_device_status((const void*)0, (dgemm_stream_t)0);
    printf("query %d\n", (int)st);
    return 0;
}
"""


def test_header_compiles_as_c_and_links(lib, tmp_path):
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(_lib.lib_path())
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-ldgemm", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = dict(line.split(" ", 1) for line in out.stdout.strip().splitlines())
    assert lines["plan"] == "0 256 256 2 256 0"          # CTA-pair 256 x 256 tiles, 256 of them
    assert lines["decode"] == "0 1"                        # transposed small-M form
    ws = dg.dgemm_workspace_size(1, 256, 512, 384, "nk", out_quant="e4m3_row_amax", act="silu")
    assert int(lines["ws"]) == ws > 2 * 256 * 512          # at least the BF16 stash
    code, text = lines["null"].split(" ", 1)
    assert int(code) == 1 and text == dg.dgemm_status_string(1)   # DGEMM_ERR_INVALID_VALUE
    assert lines["override"] == "0 0 128 1" and lines["restored"] == "256"
    assert int(lines["query"]) in (0, 5)        # DGEMM_OK on a GPU machine, DGEMM_ERR_CUDA without a device


def test_underfilled_plans_by_streamed_and_exchanged_bytes(lib, knobs):
    """Under one wave of single-CTA tiles the tile width follows each CTA's TMA
    copies (a fixed cost per copy plus the bytes) and the partial sums its K
    segments exchange in a cluster. With two-slice stages for 128- and 64-wide
    tiles, 1024^2 x 4096 takes 128-wide tiles in two segments in BF16 and FP8
    (with one slice per stage the fit makes that plan and 128 x 256 in four
    segments cost the same, as measured). Full-wave plans are unchanged."""
    def plan(fp8, M, N, K, layout):
        p = dg.dgemm_plan(fp8, M, N, K, layout, "bf16", num_sms=152)
        return (p["tile_n"], p["cta_group"], p["tail_split"], p["cluster_split"])
    assert plan(1, 1024, 1024, 4096, "nk") == (128, 1, 2, 1)
    assert plan(0, 1024, 1024, 4096, "nk") == (128, 1, 2, 1)
    assert plan(0, 512, 512, 4096, "nk")[::2] == (64, 4)
    assert plan(0, 4096, 4096, 4096, "kn")[:2] == (256, 2)
    knobs(kslices="1")
    p = dg.dgemm_plan(0, 1024, 1024, 4096, "nk", "bf16", num_sms=152)
    assert p["k_slices"] == 1 and (p["tile_n"], p["tail_split"]) in ((128, 2), (256, 4))


def test_two_slice_stages_only_where_the_operands_are_whole_slices(lib, knobs):
    """CTA-pair tile and requantising plans, and single-CTA tiles 128 or 64
    wide, take two 128-byte K slices per stage (each operand one 3-D TMA copy)
    when K, and N for B stored K x N, are whole multiples of 128 bytes;
    otherwise, and for 128 x 256 single-CTA tiles, the small-M form and
    per-K-group scales, one slice per stage."""
    def plan(fp8, M, N, K, layout, **kw):
        return dg.dgemm_plan(fp8, M, N, K, layout, "bf16", num_sms=152, **kw)
    assert plan(0, 4096, 4096, 4096, "kn")["k_slices"] == 2
    assert plan(0, 4096, 4096, 1000, "kn")["k_slices"] == 1          # K not whole 64-element slices
    assert plan(0, 4096, 4000, 4096, "kn")["k_slices"] == 1          # N not whole 64-column atoms
    assert plan(0, 4096, 4000, 4096, "nk")["k_slices"] == 2          # (N is free for B stored N x K)
    assert plan(1, 4096, 11008, 4096, "nk", k_group=128)["k_slices"] == 1
    assert plan(0, 16, 4096, 4096, "nk")["k_slices"] == 1            # small M
    knobs(cta_pair="0")
    p = plan(0, 4096, 4096, 4096, "nk")                                # single-CTA 128 x 256 tiles
    assert (p["cta_group"], p["tile_n"], p["k_slices"]) == (1, 256, 1)
    knobs(cta_pair=None)
    p = plan(0, 128, 4096, 4096, "nk")                                 # single-CTA 128 x 128 tiles
    assert (p["cta_group"], p["tile_n"], p["k_slices"], p["stages"]) == (1, 128, 2, 3)
    p = plan(1, 512, 512, 4096, "nk")                                  # FP8, 128 x 64 tiles
    assert (p["cta_group"], p["tile_n"], p["k_slices"]) == (1, 64, 2)
    assert dg.dgemm_plan(1, 8192, 8192, 8192, "nk", "e4m3", out_quant="e4m3_row_amax", num_sms=152)["k_slices"] == 2
    knobs(kslices="1")
    p = plan(0, 4096, 4096, 4096, "kn")
    assert (p["k_slices"], p["stages"]) == (1, 6)


def test_short_small_m_calls_take_half_an_sm(lib):
    """Small-M calls whose work items are at most 16 K slices long run in a
    compact footprint -- at most half of an SM's shared memory (228 KB less the
    1 KB reserved per CTA, halved) and 256 of its 512 Tensor Memory columns, so
    the K groups halve -- letting the next call's CTAs become resident early;
    longer streams keep the full ring and all 512 columns."""
    def plan(M, N, K):
        return dg.dgemm_plan(0, M, N, K, "nk", "bf16", num_sms=152)
    half_sm = (228 * 1024) // 2 - 1024
    for M in (1, 16):
        p = plan(M, 4096, 4096)   # 32 tiles x 4 K segments of 16 slices
        assert p["swap_ab"] == 1 and (p["tail_split"], p["cluster_split"]) == (4, 1)
        assert p["smem_bytes"] <= half_sm and p["stages"] == 6
        assert p["k_groups"] == 256 // p["tile_n"]
    p = plan(16, 18432, 7168)      # 144 tiles, 112 slices each: the full ring
    assert p["smem_bytes"] > half_sm and p["stages"] == 12 and p["k_groups"] == 512 // 16
    p = plan(64, 8192, 8192)       # 2 segments of 64 slices
    assert p["smem_bytes"] > half_sm and p["tail_split"] == 2
    p = plan(32, 4096, 4096)       # 32 wide, 4 segments of 16 slices: compact
    assert p["tile_n"] == 32 and p["smem_bytes"] <= half_sm
    p = dg.dgemm_plan(1, 64, 8192, 8192, "nk", "bf16", num_sms=152)   # FP8: 2 segments of 32 slices
    assert p["smem_bytes"] > half_sm
    p = plan(4096, 4096, 4096)     # tile kernels are never compact
    assert p["smem_bytes"] > half_sm
