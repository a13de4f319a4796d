"""GPU parity of the FP8 (E4M3, one scale per tensor) variant through the C ABI: quantizer and
weight packer bit for bit against the oracle, the fused GEMM at the tolerances of the NVFP4
GEMM (products of two E4M3 values are exact in fp32, so the only GEMM error is the order of
the fp32 accumulation, plus the epilogue's fp32 arithmetic).
"""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import assert_bf16_close, assert_fp32_close, to_np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu_fp8(q: nv.Fp8Tensor):
    torch.cuda.synchronize()
    return q.codes.cpu().numpy(), np.float32(q.ts.cpu().item())


def _assert_codes_equal(got, ref, what):
    gc, gt = got
    rc, rt = ref
    assert np.float32(gt).view(np.uint32) == np.float32(rt).view(np.uint32), (what, gt, rt)
    bad = np.argwhere(gc != rc)
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first {bad[:5].tolist()}"


# ---- quantizer ------------------------------------------------------------------------------

@pytest.mark.parametrize("w", [W.TINY_BIAS, W.QKV_RMSNORM.with_m(300, seed=71), W.DOWN_BIAS.with_m(257, seed=72)],
                         ids=lambda w: w.name)
def test_fp8_quantize_matches_oracle(w):
    x = W.make_x(w)
    got = _gpu_fp8(nv.fp8_quantize(x.to(DEV)))
    _assert_codes_equal(got, R.fp8_quantize_ref(to_np_f32(x)), w.name)


def test_fp8_quantize_strided_static_and_edge_values():
    g = np.random.default_rng(5)
    M, K, ld = 70, 192, 256
    big = g.standard_normal((M, ld))
    big[0, :8] = [1e-7, -1e-7, 3e-9, -3e-9, 0.0, -0.0, 448.0, -1000.0]  # underflow, sign of zero, saturation
    xb = torch.from_numpy(big.astype(np.float32)).to(torch.bfloat16)
    view = xb.to(DEV)[:, :K]
    x = to_np_f32(xb)[:, :K]
    _assert_codes_equal(_gpu_fp8(nv.fp8_quantize(view)), R.fp8_quantize_ref(x), "dynamic strided")
    for ts in (1.0, 0.01, 2.0 ** -120, 1e-39):   # unit, saturating, near the smallest normal, below it
        tsd = torch.tensor([ts], dtype=torch.float32, device=DEV)
        got = _gpu_fp8(nv.fp8_quantize(view, tensor_scale_in=tsd))
        _assert_codes_equal(got, R.fp8_quantize_ref(x, np.float32(ts)), f"static ts {ts}")


def test_fp8_quantize_zero_tensor_and_workspace_reuse():
    ws = torch.zeros(nv.nvfp4_workspace_bytes(), dtype=torch.uint8, device=DEV)
    z = torch.zeros((128, 64), dtype=torch.bfloat16, device=DEV)
    codes, ts = _gpu_fp8(nv.fp8_quantize(z, workspace=ws))
    assert ts == 0 and not codes.any()
    # the workspace comes back zeroed: a second tensor through it sees only its own amax
    x = W.make_x(W.TINY_BIAS)
    got = _gpu_fp8(nv.fp8_quantize(x.to(DEV), workspace=ws))
    _assert_codes_equal(got, R.fp8_quantize_ref(to_np_f32(x)), "after reuse")
    assert not ws.any()


# ---- weight packer --------------------------------------------------------------------------

@pytest.mark.parametrize("gated", [False, True])
def test_fp8_pack_weights_matches_oracle(gated):
    w = W.Workload("fp8_pack", 64, 320, 512, "gated_silu" if gated else "bias", seed=73)
    wt = W.make_w(w)
    got = _gpu_fp8(nv.fp8_pack_weights(wt.to(DEV), gated_interleave=gated))
    _assert_codes_equal(got, R.fp8_pack_weights_ref(to_np_f32(wt), gated), f"pack gated={gated}")


# ---- fused GEMM -----------------------------------------------------------------------------

def _run(w: W.Workload, out_dtype=torch.float32, rows=None):
    x, wt, bias, gamma = W.make_x(w), W.make_w(w), W.make_bias(w), W.make_gamma(w)
    gated = w.epilogue == W.EPI_GATED_SILU
    qa = nv.fp8_quantize(x.to(DEV))
    qb = nv.fp8_pack_weights(wt.to(DEV), gated_interleave=gated)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.fp8_gemm(qa, qb, w.epilogue, bias=None if bias is None else bias.to(DEV),
                    gamma=None if gamma is None else gamma.to(DEV), head_dim=w.head_dim, norm_cols=w.norm_cols,
                    eps=w.eps, out_dtype=out_dtype, device_error=err)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_error(err) == 0
    xs = to_np_f32(x)
    ac, ats = R.fp8_quantize_ref(xs if rows is None else xs[rows], R.fp8_tensor_scale_ref(xs))
    bc, bts = R.fp8_pack_weights_ref(to_np_f32(wt), gated)
    ref = R.fp8_gemm_ref(ac, ats, bc, bts, w.epilogue, bias=None if bias is None else bias.double().numpy(),
                         gamma=None if gamma is None else gamma.double().numpy(), head_dim=w.head_dim,
                         norm_cols=w.norm_cols, eps=w.eps)
    got = to_np_f32(y)
    return (got if rows is None else got[rows]), ref


@pytest.mark.parametrize("epi,M,N,K", [("bias", 256, 512, 512), ("gated_silu", 300, 512, 320),
                                       ("head_rmsnorm", 200, 768, 256), ("bias", 1, 256, 64),
                                       ("bias", 520, 1280, 1344)])
def test_fp8_gemm_small(epi, M, N, K):
    norm_cols = 512 if epi == "head_rmsnorm" else 0
    w = W.Workload(f"fp8_{epi}", M, K, N, epi, seed=M + N + K, norm_cols=norm_cols, head_dim=128)
    got, ref = _run(w)
    assert_fp32_close(got, ref, f"fp8 {epi} {M}x{N}x{K}")
    got16, _ = _run(w, torch.bfloat16)
    assert_bf16_close(got16, ref, f"fp8 {epi} bf16")


@pytest.mark.parametrize("w", [W.QKV_RMSNORM, W.GATED_UP, W.DOWN_BIAS], ids=lambda w: w.name)
def test_fp8_gemm_full_size_sampled_rows(w):
    rows = np.unique(np.concatenate([[0, 255, 256, w.M - 1], np.random.default_rng(19).integers(0, w.M, 12)]))
    got, ref = _run(w, torch.bfloat16, rows=rows)
    assert_bf16_close(got, ref, f"fp8 {w.name} sampled")


def test_fp8_gemm_zero_activations_give_the_bias():
    w = W.Workload("fp8_zero", 128, 256, 256, "bias", seed=74)
    bias = W.make_bias(w).to(DEV)
    qa = nv.fp8_quantize(torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV))
    qb = nv.fp8_pack_weights(W.make_w(w).to(DEV))
    y = nv.fp8_gemm(qa, qb, "bias", bias=bias, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y, bias.expand(128, 256))
