"""The seeded generators give the recipe each workload states (small shapes)."""
import numpy as np
import torch

import oracle
import workloads as wl


def test_deterministic_and_seeded():
    a = wl.make(2, M=64, N=48, K=32)
    b = wl.make(2, M=64, N=48, K=32)
    c = wl.make(2, M=64, N=48, K=32, seed=7)
    assert torch.equal(a.A, b.A) and torch.equal(a.B, b.B)
    assert not torch.equal(a.A, c.A)


def test_shapes_dtypes_layouts():
    w1 = wl.make(1, M=40, N=24, K=16)
    assert w1.A.dtype == torch.bfloat16 and w1.A.shape == (40, 16)
    assert w1.B.shape == (16, 24) and w1.b_layout == "kn"
    assert w1.C.dtype == torch.float32 and w1.C.shape == (40, 24)
    assert (w1.alpha, w1.beta, w1.d_dtype) == (1.5, 0.5, "f32")
    w3 = wl.make(3, M=32, N=40, K=64)
    assert w3.A.dtype == torch.float8_e4m3fn and w3.B.shape == (40, 64) and w3.b_layout == "nk"
    assert w3.a_scale.shape == (32,) and w3.b_scale.shape == (40,)
    w4 = wl.make(4, M=16, N=256, K=128)
    assert w4.B.shape == (256, 128) and w4.b_layout == "nk" and w4.A.dtype == torch.bfloat16
    w5 = wl.make(5, M=32, N=64, K=64)
    assert w5.bias.shape == (64,) and w5.act == "silu" and w5.out_quant == "e4m3_row_amax"


def test_value_recipes():
    w2 = wl.make(2, M=256, N=256, K=1024)
    sd = w2.A.float().std().item()
    assert abs(sd - 1 / 32) < 0.002                       # N(0,1)/sqrt(K)
    w1 = wl.make(1, M=256, N=256, K=256)
    assert w1.A.float().abs().max() <= 1 and w1.C.abs().max() <= 1
    w4 = wl.make(4, M=16, N=512, K=512)
    assert abs(w4.B.float().std().item() - 0.02) < 0.001   # sigma = 0.02


def test_fp8_quantisation_recipe():
    w = wl.make(3, M=64, N=96, K=256)
    codes = wl.codes_u8(w.A)
    dq = oracle.decode_e4m3(codes)
    # every row uses its full range: the amax element quantises to +-448
    assert np.all(np.abs(dq).max(axis=1) == 448.0)
    # per-token magnitudes span the log-uniform [0.1, 10] range: the scales differ
    s = w.a_scale.numpy()
    assert s.max() / s.min() > 5
    # per-channel weight scales near 0.02 * (max |N(0,1)| over K) / 448
    sw = w.b_scale.numpy()
    assert np.all((sw > 0.02 * 2 / 448) & (sw < 0.02 * 6 / 448))


def test_grouped_quantisation_scales_per_group():
    w = wl.fp8_grouped(32, 24, 300, k_group=128, seed=3)
    assert tuple(w.a_scale.shape) == (3, 32) and tuple(w.b_scale.shape) == (3, 24)
    assert tuple(w.B.shape) == (24, 300) and w.k_group == 128
    a = w.A.to(torch.float32).numpy()
    # each (row, group) slice has its amax at the largest finite code, 448
    for j, ks in enumerate((slice(0, 128), slice(128, 256), slice(256, 300))):
        assert np.allclose(np.abs(a[:, ks]).max(axis=1), 448.0)
    # the scales differ from group to group (the recipe's per-group magnitudes)
    assert (w.a_scale[0] != w.a_scale[1]).any()
    kn = wl.fp8_grouped(32, 24, 300, k_group=128, seed=3, b_layout="kn")
    assert torch.equal(kn.B.view(torch.uint8), w.B.view(torch.uint8).t())


def test_block_quantisation_scales_per_weight_block():
    w = wl.fp8_grouped(16, 300, 300, k_group=128, seed=4, b_block=128)
    assert tuple(w.b_scale.shape) == (3, 3) and tuple(w.a_scale.shape) == (3, 16) and w.b_block == 128
    b = w.B.to(torch.float32).numpy()
    # every (channel block, K group) block has its amax at the largest finite code
    for j, ks in enumerate((slice(0, 128), slice(128, 256), slice(256, 300))):
        for i, ns in enumerate((slice(0, 128), slice(128, 256), slice(256, 300))):
            assert np.abs(b[ns, ks]).max() == 448.0
    # decoded codes times their block's scale approximate the generated weights
    # (E4M3 keeps 3 mantissa bits: relative error <= 2^-4 away from underflow)
    assert (w.b_scale[:, 0] != w.b_scale[:, 1]).any()
