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
        """The oracle's packed weights (pack_weights_ref), optionally only some packed rows."""
        codes, scales, ts = R.pack_weights_ref(to_np_f32(self.wt), gated_interleave=self.gated)
        if packed_rows is not None:
            codes, scales = codes[packed_rows], scales[packed_rows]
        return codes, scales, ts

    def oracle_y(self, rows=None):
        """Oracle output for all columns (rows optionally sampled)."""
        a = self.oracle_a(rows)
        b = self.oracle_b()
        return R.gemm_ref(*a, *b, self.w.epilogue,
                          bias=None if self.bias is None else self.bias.double().numpy(),
                          gamma=None if self.gamma is None else self.gamma.double().numpy(),
                          head_dim=self.w.head_dim, norm_cols=self.w.norm_cols, eps=self.w.eps)


# ---------------------------------------------------------------------------------------
# Attention: the kernel rounds the probabilities to bf16 (relative 2^-9 each) before they
# multiply V, and its output to bf16; with fp32 scores and sums elsewhere the output error is
# about 2^-9 * rms(v) / sqrt(effective keys) plus the output rounding. Bounds: RMS of the
# error <= 5e-3 of the output's RMS, largest error <= 5e-2 of it plus one bf16 ulp.
# ---------------------------------------------------------------------------------------
ATT_RMS_REL = 5e-3
ATT_MAX_REL = 5e-2


def attention_oracle(qkv: np.ndarray, heads: int, head_dim: int = 256, rows=None) -> np.ndarray:
    """The oracle's attention of a QKV projection output [M, 3 H] (Q | K | V, heads side by
    side): [M or len(rows), H]; every token's K and V enter."""
    M = qkv.shape[0]
    t = np.asarray(qkv, np.float64).reshape(M, 3, heads, head_dim).transpose(1, 2, 0, 3)
    q = t[0] if rows is None else t[0][:, rows]
    return R.attention_ref(q, t[1], t[2]).transpose(1, 0, 2).reshape(-1, heads * head_dim)


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what=""):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.isfinite(got)), what
    rel = float(np.sqrt(np.mean((got - ref) ** 2))) / rms
    worst = float(np.max(np.abs(got - ref) - R.bf16_ulp(ref)))
    assert rel <= ATT_RMS_REL, f"{what}: rms error {rel:.2e} of rms"
    assert worst <= ATT_MAX_REL * rms, f"{what}: max error {worst / rms:.2e} of rms"
    return rel


# ---------------------------------------------------------------------------------------
# NVFP4 output of a GEMM (static output scale): the GPU rounds its fp32 epilogue value to bf16
# and quantizes that; where the oracle's fp64 value lies within fp32 error of a bf16 rounding
# midpoint the two bf16 inputs can differ by one ulp. The GPU's error has a relative part
# (alpha, the epilogue's exp and divide: a few fp32 ulp of |y|) and an absolute part: the fp32
# sums across the K/64 block products (each exact) err by about sqrt(K/64) * 2^-24 of the
# output's RMS (2.4e-7 of it at K = 1024, 8e-7 at K = 12288); SAFE_ABS allows several times
# that. A 16-block whose oracle values all lie farther than SAFE_REL * |y| + SAFE_ABS * RMS
# from every midpoint has identical bf16 inputs on both sides and must match bit for bit; the
# others (a few percent) are compared after dequantization.
# ---------------------------------------------------------------------------------------
SAFE_REL = 1e-5
SAFE_ABS = 2e-6


def midpoint_margin(y_ref: np.ndarray) -> np.ndarray:
    """Distance of each oracle value from the nearest bf16 rounding midpoint, over the margin
    the GPU's fp32 arithmetic may move it (> 1: both sides round to the same bf16 value)."""
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    rn = R.round_to_bf16(y_ref)
    dist = R.bf16_ulp(rn) / 2 - np.abs(y_ref - rn)
    return dist / (SAFE_REL * np.abs(y_ref) + SAFE_ABS * rms + 1e-300)


def safe_blocks(y_ref: np.ndarray) -> np.ndarray:
    """[rows, W/16] bool: every value of the block lies farther from a bf16 midpoint than the
    GPU's arithmetic can move it."""
    safe = midpoint_margin(y_ref) > 1.0
    return safe.reshape(y_ref.shape[0], -1, 16).all(axis=2)


def assert_nvfp4_out_close(got, y_ref, ts_out, what="", y_gpu32=None):
    """got = (codes, scales, ts) from the GPU; y_ref the oracle's fp64 epilogue output.
    ``y_gpu32``: the same GEMM's fp32 output on the GPU (the values the NVFP4 output rounds to
    bf16 before quantizing). Given, it is held to the fp32 bar and a block counts as exactly
    checkable when all 16 of its values round to the same bf16 on both sides (exact); without
    it, when they lie clear of every bf16 midpoint by the margin above (a bound)."""
    gc, gs, gt = got
    rc, rs, _ = R.quantize_ref(R.round_to_bf16(y_ref), np.float32(ts_out))
    assert np.float32(gt) == np.float32(ts_out)
    if y_gpu32 is not None:
        assert_fp32_close(y_gpu32, y_ref, f"{what} (fp32 epilogue values)")
        g16, r16 = R.round_to_bf16(np.asarray(y_gpu32, np.float64)), R.round_to_bf16(y_ref)
        # equal bf16 values with equal signs: the quantizer codes -0 and +0 differently
        same = (g16 == r16) & (np.signbit(g16) == np.signbit(r16))
        safe = same.reshape(y_ref.shape[0], -1, 16).all(axis=2)
    else:
        safe = safe_blocks(y_ref)
    assert safe.mean() > 0.9, f"{what}: only {safe.mean():.3f} of the blocks are exactly checkable"
    bad_s = np.argwhere((gs != rs) & safe)
    assert bad_s.size == 0, f"{what}: scale mismatch in exactly checkable blocks {bad_s[:5].tolist()}"
    code_safe = np.repeat(safe, 16, axis=1)
    bad_c = np.argwhere((gc != rc) & code_safe)
    if bad_c.size:
        rms = float(np.sqrt(np.mean(y_ref ** 2)))
        mm = midpoint_margin(y_ref)
        info = [(int(r), int(c), float(y_ref[r, c] / rms), float(mm[r, c])) for r, c in bad_c[:5]]
        raise AssertionError(f"{what}: {len(bad_c)} code mismatches in exactly checkable blocks; "
                             f"(row, col, y/rms, margin): {info}")
    # the rest: dequantized values within two steps of the coarser of the two grids
    dq_g = R.dequantize_ref(gc, gs, ts_out)
    dq_r = R.dequantize_ref(rc, rs, ts_out)
    step = 2.0 * np.maximum(np.repeat(R.e4m3_decode(gs), 16, axis=1), np.repeat(R.e4m3_decode(rs), 16, axis=1))
    assert np.all(np.abs(dq_g - dq_r) <= 2 * step * float(ts_out) + 1e-30), f"{what}: far-off block"
    return safe.mean()
