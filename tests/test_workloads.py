"""Seeded input generators: shapes, determinism and the row-prefix property the
full-size sampled parity tests rely on (CPU only)."""
import numpy as np
import torch

from nvfp4_gemm_act_b300 import workloads as W


def test_shapes_and_determinism():
    w = W.TINY_BIAS
    x = W.make_x(w)
    assert x.shape == (128, 256) and x.dtype == torch.bfloat16
    assert torch.equal(x, W.make_x(w))
    assert W.make_w(w).shape == (256, 256)
    assert W.make_bias(w).shape == (256,) and W.make_gamma(w) is None
    q = W.QKV_RMSNORM
    assert W.make_gamma(q).shape == (6144,)
    assert W.GATED_UP.out_cols == 12288 and W.make_bias(W.GATED_UP) is None


def test_row_prefix_matches_full_draw():
    for base in (W.QKV_RMSNORM, W.DOWN_BIAS):
        w = base.with_m(64)
        full = W.make_x(w)
        part = W.make_x(w, rows=16)
        assert torch.equal(full[:16], part)


def test_outlier_channels_and_heavy_tail():
    x = W.make_x(W.QKV_RMSNORM.with_m(256)).float().numpy()
    col_rms = np.sqrt((x ** 2).mean(0))
    assert (col_rms > 10).sum() == 31            # 1% of 3072 channels scaled x20
    t = W.make_x(W.DOWN_BIAS.with_m(64)).float().numpy()
    assert np.abs(t).max() > 10                  # Student-t(3) tail


def test_sweep_covers_three_gemms_at_five_sizes():
    s = W.sweep_workloads()
    assert len(s) == 15
    assert sorted({w.M for w in s}) == list(W.SWEEP_M)
    assert {w.seed for w in s} == set(range(10, 15))


def test_dit_block_layers_chain():
    # each layer's K is the previous stage's output width; the narrow variant keeps head_dim 256
    for heads, mlp in ((12, 12288), (4, 4096)):
        qkv, o, up, down = W.dit_block(384, seed=5, heads=heads, mlp=mlp)
        h = heads * 256
        assert (qkv.K, qkv.N, qkv.norm_cols, qkv.head_dim) == (h, 3 * h, 2 * h, 256)
        assert (o.K, o.N) == (h, h)
        assert (up.K, up.N, up.out_cols) == (h, 2 * mlp, mlp)
        assert (down.K, down.N) == (mlp, h)
        assert all(w.M == 384 for w in (qkv, o, up, down))
    # the full-width block reuses the benchmark layers' weights (same seeds)
    full = W.dit_block(4608)
    assert torch.equal(W.make_w(full[2]), W.make_w(W.GATED_UP))


def test_attention_qkv_is_seeded_and_scales_only_q():
    a = W.attention_qkv(16, 2, seed=3)
    b = W.attention_qkv(16, 2, seed=3, q_scale=4.0)
    assert a.shape == (16, 3 * 512) and a.dtype == torch.bfloat16
    assert torch.equal(a, W.attention_qkv(16, 2, seed=3))
    assert torch.equal(a[:, 512:], b[:, 512:])
    assert not torch.equal(a[:, :512], b[:, :512])
