"""GPU parity of the GEMM with an NVFP4 output (nvfp4_gemm_nvfp4_out): the epilogue's values,
rounded to bf16, quantized with a static output tensor scale, written as codes + tiled scales
for the next layer (through the C ABI).

Expected values come from the oracle alone: its fp64 epilogue output, rounded to bf16, then
its block quantizer with the same static scale. The GPU's fp32 epilogue value can round to
the neighbouring bf16 value where the oracle's value lies within fp32 error of a bf16 rounding
midpoint. The same GEMM's fp32 output (held to the fp32 bar) shows which: a 16-block whose 16
values round to the same bf16 on both sides has identical quantizer inputs and must match bit
for bit; the other blocks (a few percent) are compared after dequantization.
"""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import Case, assert_nvfp4_out_close as _check_against_oracle, gpu_nvfp4_to_np, to_np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
def _run(w: W.Workload, ts_scale: float = 1.0, rows=None):
    c = Case(w)
    ref = c.oracle_y(rows)
    # a static output scale taken from the oracle's output (amax of the rows it computed,
    # / 2688), times ts_scale; any positive value is a valid static scale
    ts_out = np.float32(np.float32(np.abs(ref).max()) / np.float32(2688.0) * np.float32(ts_scale))
    d = DEV
    qa = nv.nvfp4_quantize(c.x.to(d))
    qb = nv.nvfp4_pack_weights(c.wt.to(d), gated_interleave=c.gated)
    tso = torch.tensor([ts_out], dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    kw = dict(bias=None if c.bias is None else c.bias.to(d), gamma=None if c.gamma is None else c.gamma.to(d),
              head_dim=w.head_dim, norm_cols=w.norm_cols, eps=w.eps)
    q = nv.nvfp4_gemm_nvfp4_out(qa, qb, w.epilogue, tso, device_error=err, **kw)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_error(err) == 0
    # the same GEMM to bf16, then the quantizer with the same static scale: identical bytes
    y16 = nv.nvfp4_gemm(qa, qb, w.epilogue, out_dtype=torch.bfloat16, **kw)
    q2 = nv.nvfp4_quantize(y16, tensor_scale_in=tso)
    torch.cuda.synchronize()
    got = gpu_nvfp4_to_np(q)
    two = gpu_nvfp4_to_np(q2)
    assert np.array_equal(got[1], two[1]) and np.array_equal(got[0], two[0]), \
        "fused NVFP4 output differs from bf16 output + nvfp4_quantize"
    assert np.array_equal(q.scales.cpu().numpy(), q2.scales.cpu().numpy()), "scale padding differs"
    # the fp32 values the NVFP4 output rounds to bf16 (the same kernel, fp32 output mode)
    y32 = to_np_f32(nv.nvfp4_gemm(qa, qb, w.epilogue, out_dtype=torch.float32, **kw)).astype(np.float64)
    if rows is not None:
        got = (got[0][rows], got[1][rows], got[2])
        y32 = y32[rows]
    return got, ref, ts_out, y32


# the last two: output width 320, so the last tile's second half lies past the width (a ragged
# final 64-column group boundary inside a 256-column tile)
@pytest.mark.parametrize("epi,M,N,K", [("bias", 256, 512, 512), ("gated_silu", 300, 512, 320),
                                       ("head_rmsnorm", 200, 768, 256), ("bias", 192, 320, 256),
                                       ("gated_silu", 130, 640, 192)])
def test_nvfp4_out_small(epi, M, N, K):
    norm_cols = 512 if epi == "head_rmsnorm" else 0
    w = W.Workload(f"q_{epi}", M, K, N, epi, seed=M + N, norm_cols=norm_cols, head_dim=128)
    got, ref, ts, y32 = _run(w)
    _check_against_oracle(got, ref, ts, f"{epi} M={M}", y_gpu32=y32)


@pytest.mark.parametrize("ts_scale", [0.05, 20.0])
def test_nvfp4_out_saturating_and_coarse_static_scales(ts_scale):
    # a static scale far too small (block scales saturate at 448, codes at 6) or too large
    w = W.Workload("q_sat", 128, 256, 256, "bias", seed=31)
    got, ref, ts, y32 = _run(w, ts_scale=ts_scale)
    _check_against_oracle(got, ref, ts, f"ts x{ts_scale}", y_gpu32=y32)


def test_nvfp4_out_up_projection_full_size_sampled_rows():
    rows = np.unique(np.concatenate([[0, 127, 128, 4095, 4607], np.random.default_rng(17).integers(0, 4608, 19)]))
    got, ref, ts, y32 = _run(W.GATED_UP, rows=rows)
    _check_against_oracle(got, ref, ts, "gated up-projection 4608x12288 sampled", y_gpu32=y32)


def test_up_down_chain_through_nvfp4():
    # up-projection (gated) writes NVFP4, the down GEMM reads it directly: against the oracle
    # chain (fp64 up output -> bf16 -> block quantize with the static scale -> down GEMM)
    up = W.Workload("chain_up", 256, 512, 1024, "gated_silu", seed=41, bias_std=0.02)
    down = W.Workload("chain_down", 256, 512, 384, "bias", seed=42)
    cu, cd = Case(up), Case(down)
    y_up = cu.oracle_y()
    ts_mid = np.float32(np.float32(np.abs(y_up).max()) / np.float32(2688.0))
    a_mid = R.quantize_ref(R.round_to_bf16(y_up), ts_mid)
    ref = R.gemm_ref(*a_mid, *cd.oracle_b(), "bias", bias=cd.bias.double().numpy())
    d = DEV
    qa = nv.nvfp4_quantize(cu.x.to(d))
    qb_up = nv.nvfp4_pack_weights(cu.wt.to(d), gated_interleave=True)
    qb_dn = nv.nvfp4_pack_weights(cd.wt.to(d))
    tso = torch.tensor([ts_mid], dtype=torch.float32, device=d)
    mid = nv.nvfp4_gemm_nvfp4_out(qa, qb_up, "gated_silu", tso, bias=cu.bias.to(d))
    y = nv.nvfp4_gemm(mid, qb_dn, "bias", bias=cd.bias.to(d), out_dtype=torch.float32)
    torch.cuda.synchronize()
    # a few intermediate blocks may hold a neighbouring code (see the module docstring), so
    # the bound is the fp32 one widened by the effect of one code step in a few blocks
    y = to_np_f32(y)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.isfinite(y))
    assert float(np.abs(y - ref).max()) <= 2e-2 * rms
    assert float(np.sqrt(np.mean((y - ref) ** 2))) <= 2e-3 * rms
