"""The traffic / intensity helpers reproduce the numbers the pages print."""
import math
import os

from dense_gemm_persistent_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiling_page_h100.txt")


def load():
    rows = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        key = parts[0] if parts[0] != "reads_per_output" else f"{parts[0]} {parts[1]}"
        rows[key] = parts[2] if parts[0] == "reads_per_output" else parts[1]
    return rows


def close(value, printed: str):
    """Equal to the printed figure at the precision it is printed with."""
    p = float(printed)
    digits = len(printed.replace(".", "").replace("e11", "").lstrip("0"))
    return math.isclose(value, p, rel_tol=0.5 * 10 ** (1 - digits) + 1e-12)


def test_reads_per_output_table():
    g = load()
    K = 4096
    for T in (1, 4, 8, 32):
        coef, _, div = g[f"reads_per_output T={T}"].partition("/")
        want = float(coef.replace("K", "") or 1) * K / float(div or 1)
        assert roofline.reads_per_output(K, T) == want


def test_worked_example_4096():
    g = load()
    n = 4096
    reads = roofline.untiled_read_elements(n, n, n)
    assert close(reads, g["untiled_reads_4096"])
    gb = reads * 2 / 1e9
    assert close(gb, g["untiled_bytes_4096_fp16"])
    assert close(gb / 3.35e3 * 1e3, g["untiled_hbm_ms_at_3.35TBps"])
    assert close(roofline.gemm_flops(n, n, n) / 989e12 * 1e3, g["compute_ms_at_989TFLOPS"])
    # square tiles of edge T cut the reads by T: 2MNK/T
    assert roofline.tiled_read_elements(n, n, n, 128) == reads / 128


def test_intensity_and_ridge():
    g = load()
    assert close(roofline.ridge_point(989e12, 3.35e12), g["ridge_h100"])
    assert roofline.tile_intensity(128) == float(g["intensity_T128"])
    assert close(roofline.tile_intensity(128) * 3.35e12 / 1e12, g["bound_T128"])


def test_tile_grid_arithmetic():
    g = load()
    blocks = (4096 // 128) ** 2
    assert blocks == int(g["grid_blocks_4096_tile128"])
    assert close(blocks / 132, g["blocks_per_sm_132"])
    assert 128 * 32 * 2 == int(g["smem_tile_bytes_128x32_fp16"]) * 1024
