"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and the CPU
oracle on the same seeded inputs, and compare them.

Tolerances (fixed here, used by every GEMM parity test):
  * quantized codes and scales: bit-exact;
  * fp32 outputs: max |gpu - oracle| <= 2e-3 * RMS(oracle output);
  * bf16 outputs: where |oracle| >= 2^-8 * RMS, the GPU value is RN_bf16(oracle) or one of its
    two bf16 neighbours (1 ulp); smaller elements (cancellation) are held to the fp32 bound.
"""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

FP32_RTOL_RMS = 2e-3
BF16_SMALL = 2.0 ** -8


def to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def gpu_nvfp4_to_np(q: nv.Nvfp4Tensor):
    """Device Nvfp4Tensor -> (codes [rows, K] nibbles, scales [rows, K/16], ts float32)."""
    torch.cuda.synchronize()
    codes = R.unpack_nibbles(q.codes.cpu().numpy())
    scales = R.untile_scales(q.scales.cpu().numpy(), q.rows, q.K)
    return codes, scales, np.float32(q.ts.cpu().item())


def assert_quant_equal(gpu, ref, what=""):
    gc, gs, gt = gpu
    rc, rs, rt = ref
    assert np.float32(gt).view(np.uint32) == np.float32(rt).view(np.uint32), (what, gt, rt)
    bad_s = np.argwhere(gs != rs)
    assert bad_s.size == 0, f"{what}: {len(bad_s)} scale mismatches, first {bad_s[:5].tolist()}"
    bad_c = np.argwhere(gc != rc)
    assert bad_c.size == 0, f"{what}: {len(bad_c)} code mismatches, first {bad_c[:5].tolist()}"


def assert_fp32_close(y_gpu: np.ndarray, y_ref: np.ndarray, what=""):
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    worst = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite outputs"
    assert worst <= FP32_RTOL_RMS * rms, f"{what}: max|err| {worst:.3e} > {FP32_RTOL_RMS} * rms {rms:.3e}"
    return worst / max(rms, 1e-300)


def assert_bf16_close(y_gpu: np.ndarray, y_ref: np.ndarray, what=""):
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    y_gpu = y_gpu.astype(np.float64)
    big = np.abs(y_ref) >= BF16_SMALL * rms
    rn = R.round_to_bf16(y_ref)
    ulp = R.bf16_ulp(rn)
    ok_big = np.abs(y_gpu - rn) <= ulp * (1 + 1e-12)
    ok_small = np.abs(y_gpu - y_ref) <= FP32_RTOL_RMS * rms
    bad = (big & ~ok_big) | (~big & ~ok_small)
    n_bad = int(bad.sum())
    assert n_bad == 0, (f"{what}: {n_bad} bf16 elements off by more than 1 ulp; first "
                        f"{np.argwhere(bad)[:5].tolist()}")
    # how many small elements would fail the literal "within 1 ulp" reading
    return int((~big & ~(np.abs(y_gpu - rn) <= ulp)).sum())


class Case:
    """One workload's inputs on host and device, the GPU result and the oracle's."""

    def __init__(self, w: W.Workload, dev="cuda:0"):
        self.w = w
        self.x = W.make_x(w)
        self.wt = W.make_w(w)
        self.bias = W.make_bias(w)
        self.gamma = W.make_gamma(w)
        self.dev = dev
        self.gated = w.epilogue == W.EPI_GATED_SILU

    def run_gpu(self, out_dtype=torch.float32):
        d = self.dev
        self.qa = nv.nvfp4_quantize(self.x.to(d))
        self.qb = nv.nvfp4_pack_weights(self.wt.to(d), gated_interleave=self.gated)
        self.err = torch.zeros(1, dtype=torch.int32, device=d)
        y = nv.nvfp4_gemm(self.qa, self.qb, self.w.epilogue,
                          bias=None if self.bias is None else self.bias.to(d),
                          gamma=None if self.gamma is None else self.gamma.to(d),
                          head_dim=self.w.head_dim, norm_cols=self.w.norm_cols, eps=self.w.eps,
                          out_dtype=out_dtype, device_error=self.err)
        torch.cuda.synchronize()
        assert nv.nvfp4_get_device_error(self.err) == 0
        return to_np_f32(y)

    def oracle_a(self, rows=None):
        x = to_np_f32(self.x)
        ts = R.tensor_scale_ref(x)
        xs = x if rows is None else x[rows]
        return R.quantize_ref(xs, ts)

    def oracle_b(self, packed_rows=None):
        w = to_np_f32(self.wt)
        ts = R.tensor_scale_ref(w)
        wt = w.T
        if self.gated:
            wt = wt[R.gated_permutation(w.shape[1])]
        if packed_rows is not None:
            wt = wt[packed_rows]
        return R.quantize_ref(np.ascontiguousarray(wt), ts)

    def oracle_y(self, rows=None):
        """Oracle output for all columns (rows optionally sampled)."""
        a = self.oracle_a(rows)
        b = self.oracle_b()
        return R.gemm_ref(*a, *b, self.w.epilogue,
                          bias=None if self.bias is None else self.bias.double().numpy(),
                          gamma=None if self.gamma is None else self.gamma.double().numpy(),
                          head_dim=self.w.head_dim, norm_cols=self.w.norm_cols, eps=self.w.eps)
