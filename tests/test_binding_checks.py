"""The Python binding's argument checks, on the CPU.

The C ABI receives raw device pointers and trusts that they address dense
row-major buffers of the stated sizes; the binding refuses tensors that are
not (CPU tensors, transposed or sliced views, wrong shapes or element types)
before calling it. These tests replace the library with a recorder and the
device test with one that accepts CPU tensors, so they need no GPU.
"""
import pytest
import torch

import dense_gemm_persistent_gb300 as dg


class Recorder:
    """Stands in for libdgemm.so: records each call's arguments, returns DGEMM_OK."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def entry(*args):
            self.calls.append((name, args))
            return 0
        return entry


@pytest.fixture
def lib(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(dg, "load", lambda *a, **k: rec)
    monkeypatch.setattr(dg, "_on_device", lambda t: True)
    return rec


def bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def e4m3(*shape):
    return torch.zeros(*shape, dtype=torch.float8_e4m3fn)


def f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


def test_valid_bf16_call_passes_sizes_and_pointers(lib):
    A, B, D = bf16(8, 16), bf16(16, 24), f32(8, 24)
    dg.dgemm_bf16(A, B, D, b_layout="kn", stream=0)
    name, args = lib.calls[-1]
    assert name == "dgemm_bf16"
    assert args[0] == A.data_ptr() and args[1] == B.data_ptr() and args[5] == D.data_ptr()
    assert args[7:10] == (8, 24, 16)


def test_in_place_c_equal_to_d(lib):
    A, B, D = bf16(8, 16), bf16(24, 16), bf16(8, 24)
    dg.dgemm_bf16(A, B, D, b_layout="nk", C=D, alpha=0.75, beta=-1.25, stream=0)
    assert lib.calls[-1][0] == "dgemm_bf16"


def test_k_zero_and_block_scales_left_to_the_library(lib):
    # K = 0 with per-K-group scales: no group exists, the 1-D tables are never read
    dg.dgemm_fp8_scaled(e4m3(8, 0), e4m3(24, 0), f32(8), f32(24), f32(8, 24), b_layout="nk", k_group=128,
                        C=f32(8, 24), beta=2.0, stream=0)
    # scale-table shapes depend on k_group and b_block: the library decides
    dg.dgemm_fp8_scaled(e4m3(16, 128), e4m3(128, 128), f32(1), f32(1), f32(16, 128), b_layout="nk",
                        k_group=0, b_block=128, stream=0)
    assert [c[0] for c in lib.calls] == ["dgemm_fp8_scaled", "dgemm_fp8_blockscaled"]


def test_uint8_codes_and_e4m3_output(lib):
    Aq = torch.zeros(8, 32, dtype=torch.uint8)
    Bq = torch.zeros(24, 32, dtype=torch.uint8)
    q = torch.zeros(8, 24, dtype=torch.uint8)
    dg.dgemm_fp8_scaled(Aq, Bq, f32(8), f32(24), q, b_layout="nk", bias=f32(24), act="silu",
                        out_quant="e4m3_row_amax", out_row_scale=f32(8), ws=torch.zeros(64, dtype=torch.uint8),
                        stream=0)
    dg.dgemm_fp8_rowquant_noalloc(Aq, Bq, f32(8), f32(24), q, f32(8), b_layout="nk", bias=f32(24), act="silu",
                                  stream=0)
    assert [c[0] for c in lib.calls] == ["dgemm_fp8_scaled", "dgemm_fp8_rowquant_noalloc"]


def test_c_is_not_checked_when_beta_is_zero(lib):
    dg.dgemm_bf16(bf16(8, 16), bf16(16, 24), f32(8, 24), C=f32(3, 3), beta=0.0, stream=0)
    assert len(lib.calls) == 1


@pytest.mark.parametrize("case", ["transposed_a", "sliced_b", "d_shape", "c_shape", "bias_len", "row_scale_len",
                                  "a_dtype", "scale_dtype", "ws_view"])
def test_refused_before_the_call(lib, case):
    A, B, D = bf16(8, 16), bf16(16, 24), f32(8, 24)
    kw = {}
    if case == "transposed_a":
        A = bf16(16, 8).t()                 # 8 x 16 but column-major
    elif case == "sliced_b":
        B = bf16(16, 48)[:, ::2]            # 16 x 24 with a stride of 2
    elif case == "d_shape":
        D = f32(24, 8)
    elif case == "c_shape":
        kw = dict(C=f32(8, 23), beta=1.0)
    elif case == "bias_len":
        kw = dict(bias=f32(23))
    elif case == "row_scale_len":
        kw = dict(out_quant="e4m3_row_amax", out_row_scale=f32(7))
        D = torch.zeros(8, 24, dtype=torch.uint8)
    elif case == "a_dtype":
        A = f32(8, 16)
    elif case == "ws_view":
        kw = dict(ws=torch.zeros(64, 2, dtype=torch.uint8).t())
    if case == "scale_dtype":
        with pytest.raises(ValueError):
            dg.dgemm_fp8_scaled(e4m3(8, 16), e4m3(24, 16), torch.zeros(8, dtype=torch.float64), f32(24),
                                D, b_layout="nk", stream=0)
    else:
        with pytest.raises(ValueError):
            dg.dgemm_bf16(A, B, D, b_layout="kn", stream=0, **kw)
    assert lib.calls == []


def test_cpu_tensors_are_refused(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(dg, "load", lambda *a, **k: rec)
    with pytest.raises(ValueError, match="CUDA"):
        dg.dgemm_bf16(bf16(8, 16), bf16(16, 24), f32(8, 24), stream=0)
    assert rec.calls == []
