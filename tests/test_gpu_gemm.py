"""GPU parity of the fused NVFP4 GEMM (bias, per-head RMSNorm, gated-SiLU epilogues)
against the oracle, element by element, in fp32 and bf16 output modes (through the C ABI)."""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import Case, assert_bf16_close, assert_fp32_close, to_np_f32

pytestmark = pytest.mark.gpu


def check_case(w, rows=None):
    c = Case(w)
    y32 = c.run_gpu(torch.float32)
    y16 = c.run_gpu(torch.bfloat16)
    ref = c.oracle_y(rows)
    if rows is not None:
        y32, y16 = y32[rows], y16[rows]
    assert y32.shape == ref.shape
    assert_fp32_close(y32, ref, f"{w.name} fp32")
    assert_bf16_close(y16, ref, f"{w.name} bf16")
    return c


def test_tiny_bias():
    check_case(W.TINY_BIAS)


@pytest.mark.parametrize("base", [W.QKV_RMSNORM, W.GATED_UP, W.DOWN_BIAS], ids=lambda w: w.name)
def test_dit_shapes_ragged_m(base):
    # M = 200: two row tiles, the second one ragged (rows 200..255 masked)
    check_case(base.with_m(200))


SAMPLED_ROWS = np.unique(np.concatenate([[0, 1, 31, 32, 127, 128, 2047, 4095, 4096, 4607],
                                         np.random.default_rng(11).integers(0, 4608, 22)]))


@pytest.mark.parametrize("base", [W.QKV_RMSNORM, W.GATED_UP, W.DOWN_BIAS], ids=lambda w: w.name)
def test_dit_shapes_full_size_sampled_rows(base):
    # the launch configuration the benchmark times (M = 4608), sampled output rows
    check_case(base, rows=SAMPLED_ROWS)


@pytest.mark.parametrize("M,N,K", [(1, 32, 64), (64, 288, 320), (129, 544, 1024), (300, 256, 64)])
@pytest.mark.parametrize("epi", ["bias", "head_rmsnorm", "gated_silu"])
def test_edge_shapes(M, N, K, epi):
    # ragged M, N tiles with a missing second scale band (N % 256 in {32, 32}), K with a
    # partial pipeline stage (K % 256 = 64), single-row and single-stage problems
    hd = 32 if epi == "head_rmsnorm" else 256
    norm_cols = (N // 2) // hd * hd if epi == "head_rmsnorm" else 0
    w = W.Workload(f"edge_{epi}", M, K, N, epi, seed=M + N + K, norm_cols=norm_cols,
                   head_dim=hd, bias_std=0.01)
    check_case(w)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_rmsnorm_head_dims_and_unit_rms(hd):
    w = W.Workload("rms", 256, 512, 768, W.EPI_HEAD_RMSNORM, seed=5, norm_cols=512,
                   head_dim=hd, gamma_std=0.0)
    c = check_case(w)
    # gamma = 1: every normalised head has RMS sqrt(ms / (ms + eps)) ~ 1
    y = c.run_gpu(torch.float32)
    heads = y[:, :512].reshape(256, 512 // hd, hd)
    rms = np.sqrt((heads.astype(np.float64) ** 2).mean(-1))
    assert np.allclose(rms, 1.0, atol=1e-3)


def test_no_bias_and_explicit_out_stride():
    w = dict(M=128, K=256, N=256)
    x = W.make_x(W.TINY_BIAS).cuda()
    wt = W.make_w(W.TINY_BIAS).cuda()
    qa = nv.nvfp4_quantize(x)
    qb = nv.nvfp4_pack_weights(wt)
    big = torch.full((128, 320), 7.0, dtype=torch.float32, device="cuda")
    out = big[:, :256]
    nv.nvfp4_gemm(qa, qb, "bias", out_dtype=torch.float32, out=out)
    torch.cuda.synchronize()
    a = R.quantize_ref(to_np_f32(W.make_x(W.TINY_BIAS)))
    b = R.pack_weights_ref(to_np_f32(W.make_w(W.TINY_BIAS)))
    ref = R.gemm_ref(*a, *b, "bias")
    assert_fp32_close(to_np_f32(out), ref, "no bias, ldo 320")
    assert (big[:, 256:] == 7.0).all(), "columns past N must not be written"


def test_gated_output_pairs_match_unpermuted_formula():
    # the gated epilogue on interleaved weights equals the page's formula on the plain GEMM
    w = W.Workload("gpair", 128, 256, 512, W.EPI_GATED_SILU, seed=9, bias_std=0.05)
    c = Case(w)
    g = c.run_gpu(torch.float32)
    d = "cuda:0"
    qa = nv.nvfp4_quantize(c.x.to(d))
    qb = nv.nvfp4_pack_weights(c.wt.to(d), gated_interleave=False)
    plain = nv.nvfp4_gemm(qa, qb, "bias", bias=c.bias.to(d), out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = R.gated_silu_ref(to_np_f32(plain).astype(np.float64))
    assert_fp32_close(g, ref, "gated vs formula on plain GEMM")


MANY_TILE_ROWS = np.unique(np.concatenate([[0, 127, 128, 255, 256, 2047, 2048, 4095],
                                           np.random.default_rng(13).integers(0, 4096, 24)]))


@pytest.mark.parametrize("epi", ["bias", "head_rmsnorm", "gated_silu"])
def test_many_tiles_per_pair_partial_stage(epi):
    # 16 x 9 = 144 pair tiles on 74 CTA pairs (two tiles for most pairs) with K = 1344: six
    # 256-deep stages per tile, the last holding one 64-deep step, so the 5-slot ring's
    # position drifts against tile boundaries and the accumulator handshake alternates phase
    norm_cols = 1536 if epi == "head_rmsnorm" else 0
    w = W.Workload(f"many_{epi}", 4096, 1344, 2304, epi, seed=77, norm_cols=norm_cols, head_dim=64)
    check_case(w, rows=MANY_TILE_ROWS)
