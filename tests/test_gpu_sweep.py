"""Batch sweep: the three DiT GEMMs (QKV + head RMSNorm, gated-SiLU up-projection, down-
projection + bias) at M in {512, 1024, 4608, 9216, 18432} tokens, each layer keeping its
weights while the activations are redrawn (seeds 10..14). Parity against the oracle on
sampled output rows (all columns), fp32 and bf16 outputs, through the C ABI."""
import functools

import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import assert_bf16_close, assert_fp32_close, to_np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@functools.lru_cache(maxsize=None)
def oracle_weights(base_name: str):
    w = W.WORKLOADS[base_name]
    return R.pack_weights_ref(to_np_f32(W.make_w(w)), w.epilogue == W.EPI_GATED_SILU)


@functools.lru_cache(maxsize=None)
def device_weights(base_name: str):
    w = W.WORKLOADS[base_name]
    return nv.nvfp4_pack_weights(W.make_w(w).to(DEV), gated_interleave=w.epilogue == W.EPI_GATED_SILU)


CASES = [(w.name.rsplit("_m", 1)[0], w.M, w.seed) for w in W.sweep_workloads()]


@pytest.mark.parametrize("base_name,M,seed", CASES, ids=[f"{b}-M{m}" for b, m, _ in CASES])
def test_sweep_case(base_name, M, seed):
    base = W.WORKLOADS[base_name]
    w = base.with_m(M, seed=seed)
    x = W.make_x(w)
    bias, gamma = W.make_bias(w), W.make_gamma(w)
    qa = nv.nvfp4_quantize(x.to(DEV))
    qb = device_weights(base_name)
    kw = dict(bias=None if bias is None else bias.to(DEV), gamma=None if gamma is None else gamma.to(DEV),
              head_dim=w.head_dim, norm_cols=w.norm_cols, eps=w.eps)
    y32 = to_np_f32(nv.nvfp4_gemm(qa, qb, w.epilogue, out_dtype=torch.float32, **kw))
    y16 = to_np_f32(nv.nvfp4_gemm(qa, qb, w.epilogue, out_dtype=torch.bfloat16, **kw))
    rows = np.unique(np.concatenate([[0, 127, 128, M - 129, M - 1],
                                     np.random.default_rng(M).integers(0, M, 11)]))
    xn = to_np_f32(x)
    a = R.quantize_ref(xn[rows], R.tensor_scale_ref(xn))
    ref = R.gemm_ref(*a, *oracle_weights(base_name), w.epilogue,
                     bias=None if bias is None else bias.double().numpy(),
                     gamma=None if gamma is None else gamma.double().numpy(),
                     head_dim=w.head_dim, norm_cols=w.norm_cols, eps=w.eps)
    assert_fp32_close(y32[rows], ref, f"{w.name} fp32")
    assert_bf16_close(y16[rows], ref, f"{w.name} bf16")
