"""GPU parity of the attention kernel (attention_fwd, through the C ABI) against the oracle's
fp64 softmax attention of the same bf16 Q, K, V.

Tolerance: the kernel rounds the probabilities to bf16 (relative 2^-9 each) before they
multiply V, and its output to bf16 (2^-9); with fp32 scores and sums elsewhere the output
error is about 2^-9 * rms(v) / sqrt(effective keys) plus the output rounding. Bounds: RMS of
the error <= 5e-3 of the output's RMS, largest error <= 5e-2 of it plus one bf16 ulp of the
element. Cases: ragged query and key tiles, one token, large logits (the O rescaling path), a
dominant key (exact answer), and the full DiT shape (4608 tokens, 12 heads) on sampled rows.
"""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import assert_attention_close, attention_oracle, to_np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HD = 256


def _ref(qkv: np.ndarray, heads: int, rows=None) -> np.ndarray:
    return attention_oracle(qkv, heads, HD, rows)


def _run(qkv: torch.Tensor, heads: int) -> np.ndarray:
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.attention(qkv.to(DEV), heads, device_error=err)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_error(err) == 0
    return to_np_f32(y).astype(np.float64)


def _check(got, ref, what):
    return assert_attention_close(got, ref, what)


@pytest.mark.parametrize("M,heads,q_scale", [(200, 2, 1.0), (1, 1, 1.0), (64, 1, 1.0), (65, 1, 1.0),
                                             (384, 4, 1.0), (300, 2, 4.0), (700, 1, 8.0), (1000, 3, 1.0)])
def test_attention_matches_oracle(M, heads, q_scale):
    qkv = W.attention_qkv(M, heads, seed=M + heads, q_scale=q_scale)
    got = _run(qkv, heads)
    _check(got, _ref(to_np_f32(qkv).astype(np.float64), heads), f"M={M} heads={heads} q x{q_scale}")


def test_attention_strided_input_and_output():
    # qkv and out as column windows of wider buffers (row pitches 3 H + 64 and H + 128)
    M, heads = 200, 2
    H = heads * HD
    qkv = W.attention_qkv(M, heads, seed=12)
    wide = torch.zeros((M, 3 * H + 64), dtype=torch.bfloat16)
    wide[:, 32:32 + 3 * H] = qkv
    src = wide.to(DEV)[:, 32:32 + 3 * H]
    big_out = torch.full((M, H + 128), 7.0, dtype=torch.bfloat16, device=DEV)
    out = big_out[:, 64:64 + H]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nv.attention(src, heads, out=out, device_error=err)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_error(err) == 0
    _check(to_np_f32(out).astype(np.float64), _ref(to_np_f32(qkv).astype(np.float64), heads), "strided")
    # nothing outside the output window was written
    assert bool((big_out[:, :64] == 7.0).all()) and bool((big_out[:, 64 + H:] == 7.0).all())


def test_attention_single_token_returns_v():
    qkv = W.attention_qkv(1, 3, seed=7)
    got = _run(qkv, 3)
    v = to_np_f32(qkv)[:, 2 * 3 * HD:]
    assert np.array_equal(got, v)


def test_attention_dominant_key_selects_its_value():
    # every query is key 5 scaled up: its score (40) exceeds every other (|.| < 12 for unit
    # vectors in 256 dimensions) by about 30, a weight ratio near e^-30, so the output is v_5 up
    # to the bf16 rounding of the output
    M, heads = 150, 1
    g = np.random.default_rng(8)
    k = g.standard_normal((M, HD))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = np.repeat(40.0 * np.sqrt(HD) * k[5:6], M, axis=0)
    v = g.standard_normal((M, HD))
    qkv = torch.from_numpy(np.concatenate([q, k, v], axis=1).astype(np.float32)).to(torch.bfloat16)
    got = _run(qkv, heads)
    vb = to_np_f32(qkv)[5, 2 * HD:].astype(np.float64)
    assert np.all(np.abs(got - vb[None, :]) <= R.bf16_ulp(vb)[None, :])


def test_attention_full_dit_shape_sampled_rows():
    M, heads = 4608, 12
    qkv = W.attention_qkv(M, heads, seed=9)
    got = _run(qkv, heads)
    rows = np.unique(np.concatenate([[0, 127, 128, 4095, 4607], np.random.default_rng(10).integers(0, M, 11)]))
    ref = _ref(to_np_f32(qkv).astype(np.float64), heads, rows=rows)
    _check(got[rows], ref, "4608 x 12 heads sampled")


def test_attention_matches_torch_in_the_dit_block():
    # the block's own QKV output (RMSNorm'd Q and K): the kernel against the oracle, and torch's
    # scaled_dot_product_attention held to the same bound, on the same input
    from nvfp4_gemm_act_b300.dit_block import seeded_dit_block
    blk, x = seeded_dit_block(512, DEV, seed=11, heads=4, mlp=4096)
    t = blk.qkv_rmsnorm(x)
    got = _run(t, 4)
    ref = _ref(to_np_f32(t).astype(np.float64), 4)
    _check(got, ref, "block qkv")
    _check(to_np_f32(blk.attention_torch(t)).astype(np.float64), ref, "torch on block qkv")
