"""GPU parity of one DiT block's chained linears (DitBlockLinears, with this package's attention
kernel between the first two) against the oracle, on the same seeded inputs.

Element by element, stage by stage: each oracle stage is fed the GPU's output of the stage
before it (exactly the bf16 values, or the NVFP4 codes and scales, the GPU handed on), so every
stage is held to the bar of its own kernel:
  * QKV + per-head RMSNorm (from x): the bf16 bar (RN_bf16 of the oracle value or a neighbour);
  * attention (from the GPU's QKV output): the attention bound (error RMS <= 5e-3 of the output
    RMS, largest error <= 5e-2 of it plus one bf16 ulp);
  * output projection (from the GPU's attention output; dynamic tensor scale): the bf16 bar;
  * gated up-projection written as NVFP4 with the static scale (from the GPU's output
    projection; dynamic scale of that): codes and scales bit for bit in every block whose
    values lie clear of a bf16 rounding midpoint, the rest within two code steps;
  * down-projection (from the GPU's NVFP4 codes, scales and static scale): the bf16 bar.

The chained comparison is kept as an extra check: quantizing again at every layer lets a value
within rounding error of a code or block-scale boundary round either way, and such differences
grow through three quantizations, so the chains are compared through their error against the
exact fp64 block: rel(gpu, exact) within 2% of rel(oracle, exact), and the two chains closer to
each other than to the exact block (at most 0.15 of it for the output projection, 0.5 for the
up-projection and the block output; independent rounding would put them sqrt(2) of it apart).
"""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv  # noqa: F401
from nvfp4_gemm_act_b300 import workloads as W
from nvfp4_gemm_act_b300.dit_block import seeded_dit_block
from oracle import nvfp4_ref as R

from parity import (assert_attention_close, assert_bf16_close, assert_nvfp4_out_close, attention_oracle,
                    gpu_nvfp4_to_np, to_np_f32)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HD = 256

# (M, seed, heads, mlp): a narrow block (4 heads of 256, MLP 4096) and the full-width one
# (12 heads, MLP 12288) on 384 tokens (one and a half 256-row tiles)
CONFIGS = {"narrow": (384, 60, 4, 4096), "full_width": (384, 61, 12, 12288)}


def _rel(a, b):
    return float(np.sqrt(np.mean((a - b) ** 2) / np.mean(b ** 2)))


def _layers(ls):
    """The four layers as numpy (W [K, N] fp32, bias fp64 or None, gamma fp64 or None) and each
    weight packed once by the oracle (the up-projection's with the gated interleave)."""
    layers, packed = [], []
    for w in ls:
        b, g = W.make_bias(w), W.make_gamma(w)
        wn = W.make_w(w).float().numpy()
        layers.append((wn, None if b is None else b.double().numpy(), None if g is None else g.double().numpy()))
        packed.append(R.pack_weights_ref(wn, gated_interleave=w.epilogue == W.EPI_GATED_SILU))
    return layers, packed


def _stages_from_gpu(keep, layers, packed, heads, ts_mid, rows=None):
    """Each stage of the oracle fed the GPU's previous-stage output; ``rows``: the tokens to
    compute (every token's K, V and every dynamic tensor scale still come from all tokens)."""
    hidden = heads * HD
    (_, _, _), (_, b_o, _), (_, b_up, _), (_, b_dn, _) = layers
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    t = to_np_f32(keep["qkv_rmsnorm"])
    att = attention_oracle(t, heads, HD, rows)
    a_gpu = to_np_f32(keep["attention"])
    o = R.gemm_ref(*R.quantize_ref(sel(a_gpu), R.tensor_scale_ref(a_gpu)), *packed[1], R.EPI_BIAS, bias=b_o)
    o_gpu = to_np_f32(keep["out_proj"])
    up = R.gemm_ref(*R.quantize_ref(sel(o_gpu), R.tensor_scale_ref(o_gpu)), *packed[2], R.EPI_GATED_SILU,
                    bias=b_up)
    u_codes, u_scales, u_ts = gpu_nvfp4_to_np(keep["up_gated_silu"])
    assert np.float32(u_ts) == np.float32(ts_mid)
    down = R.gemm_ref(sel(u_codes), sel(u_scales), u_ts, *packed[3], R.EPI_BIAS, bias=b_dn)
    assert att.shape[1] == hidden
    return {"attention": att, "out_proj": o, "up": up, "down": down,
            "u_gpu": (sel(u_codes), sel(u_scales), u_ts)}


@pytest.fixture(scope="module", params=list(CONFIGS))
def block(request):
    M, seed, heads, mlp = CONFIGS[request.param]
    ls = W.dit_block(M, seed, heads=heads, mlp=mlp)
    x = W.make_x(ls[0])
    layers, packed = _layers(ls)
    xs = x.float().numpy()
    y_ref, ref = R.dit_block_ref(xs, layers, heads, HD, packed=packed)
    y_ex, ex = R.dit_block_ref(xs, layers, heads, HD, quantized=False)
    blk, xd = seeded_dit_block(M, DEV, seed=seed, heads=heads, mlp=mlp)
    blk.calibrate(xd, ts_mid=torch.tensor([ref["ts_mid"]], dtype=torch.float32, device=DEV))
    keep = {}
    y = blk(xd, keep=keep)
    torch.cuda.synchronize()
    st = _stages_from_gpu(keep, layers, packed, heads, ref["ts_mid"])
    ts_gpu = float(blk.calibrate(xd)[0])
    blk.calibrate(xd, ts_mid=torch.tensor([ref["ts_mid"]], dtype=torch.float32, device=DEV))
    return dict(name=request.param, y=to_np_f32(y).astype(np.float64), keep=keep, y_ref=y_ref, ref=ref,
                y_ex=y_ex, ex=ex, ts_gpu=ts_gpu, M=M, st=st, blk=blk)


# ---- element-wise, stage by stage -------------------------------------------------------

def test_qkv_stage_matches_bf16(block):
    got = to_np_f32(block["keep"]["qkv_rmsnorm"])
    assert_bf16_close(got, block["ref"]["qkv"], f"{block['name']} qkv")


def test_attention_stage_elementwise(block):
    got = to_np_f32(block["keep"]["attention"]).astype(np.float64)
    assert_attention_close(got, block["st"]["attention"], f"{block['name']} attention")


def test_out_proj_stage_elementwise(block):
    got = to_np_f32(block["keep"]["out_proj"])
    assert_bf16_close(got, block["st"]["out_proj"], f"{block['name']} out_proj")


def _up_fp32(blk, o, rows=None):
    """The block's up-projection on the GPU with an fp32 output: the values its NVFP4 output
    rounds to bf16 and quantizes."""
    y = nv.nvfp4_gemm(nv.nvfp4_quantize(o), blk.qb["up"], "gated_silu", bias=blk.bias["up"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    y = to_np_f32(y).astype(np.float64)
    return y if rows is None else y[rows]


def test_up_projection_nvfp4_stage_elementwise(block):
    y32 = _up_fp32(block["blk"], block["keep"]["out_proj"])
    assert_nvfp4_out_close(block["st"]["u_gpu"], block["st"]["up"], block["ref"]["ts_mid"],
                           f"{block['name']} up (NVFP4 out)", y_gpu32=y32)


def test_up_projection_fused_equals_bf16_then_quantize(block):
    # the block's fused NVFP4 output is, bit for bit, its up-projection written in bf16 then
    # quantized with the same static scale; that bf16 output meets the bf16 bar against the
    # oracle stage fed the GPU's output projection
    blk = block["blk"]
    o = block["keep"]["out_proj"]
    y16 = nv.nvfp4_gemm(nv.nvfp4_quantize(o), blk.qb["up"], "gated_silu", bias=blk.bias["up"])
    q = nv.nvfp4_quantize(y16, tensor_scale_in=blk.ts_mid)
    u = block["keep"]["up_gated_silu"]
    torch.cuda.synchronize()
    assert torch.equal(q.codes, u.codes) and torch.equal(q.scales, u.scales)
    assert_bf16_close(to_np_f32(y16), block["st"]["up"], f"{block['name']} up (bf16 out)")


def test_down_stage_elementwise(block):
    assert_bf16_close(block["y"], block["st"]["down"], f"{block['name']} down")


# ---- the chain as a whole (extra check) ---------------------------------------------------

def test_out_proj_chain_tracks_oracle(block):
    got = to_np_f32(block["keep"]["out_proj"]).astype(np.float64)
    ref, ex = block["ref"]["out_proj"], block["ex"]["out_proj"]
    q_err = _rel(ref, ex)
    assert _rel(got, ex) <= 1.02 * q_err
    assert _rel(got, ref) <= 0.15 * q_err, (_rel(got, ref), q_err)


def test_up_projection_chain_tracks_oracle(block):
    u = block["keep"]["up_gated_silu"]
    ts = np.float32(block["ref"]["ts_mid"])
    codes = R.unpack_nibbles(u.codes.cpu().numpy())
    scales = R.untile_scales(u.scales.cpu().numpy(), u.rows, u.K)
    got = R.dequantize_ref(codes, scales, ts)
    ref = R.dequantize_ref(*R.quantize_ref(block["ref"]["up"], ts))
    ex = block["ex"]["up"]
    q_err = _rel(ref, ex)
    assert _rel(got, ex) <= 1.02 * q_err
    assert _rel(got, ref) <= 0.5 * q_err, (_rel(got, ref), q_err)


def test_block_output_chain_tracks_oracle(block):
    y, ref, ex = block["y"], block["y_ref"], block["y_ex"]
    assert np.all(np.isfinite(y))
    q_err = _rel(ref, ex)
    assert _rel(y, ex) <= 1.02 * q_err, (_rel(y, ex), q_err)
    assert _rel(y, ref) <= 0.5 * q_err, (_rel(y, ref), q_err)


def test_calibrated_static_scale(block):
    # the GPU's own calibration (the library's tensor scale, amax / 2688, of its bf16
    # up-projection output) lands near the oracle's: one extreme value of a chain whose stages
    # differ by rounding
    ts_ref = float(block["ref"]["ts_mid"])
    assert abs(block["ts_gpu"] / ts_ref - 1.0) <= 0.05


def test_calibration_is_the_librarys_tensor_scale():
    # calibrate() takes the static scale from nvfp4_quantize's own tensor scale of the bf16
    # up-projection output (no amax arithmetic outside the library): equal to the oracle's
    # tensor_scale_ref of that same output, bit for bit
    blk, xd = seeded_dit_block(256, DEV, seed=73, heads=4, mlp=4096)
    ts = blk.calibrate(xd)
    o = blk.out_proj(blk.attention(blk.qkv_rmsnorm(xd)))
    u = nv.nvfp4_gemm(nv.nvfp4_quantize(o), blk.qb["up"], "gated_silu", bias=blk.bias["up"])
    torch.cuda.synchronize()
    want = R.tensor_scale_ref(to_np_f32(u))
    assert np.float32(ts.item()).view(np.uint32) == np.float32(want).view(np.uint32)


def test_full_size_block_sampled_rows():
    # the benchmarked shape: 4608 tokens through the full-width block, sampled output rows
    # (every token's K and V and every dynamic scale still come from all tokens); each stage
    # element-wise from the GPU's previous stage, and the chain as a whole
    M, seed = 4608, 70
    ls = W.dit_block(M, seed)
    x = W.make_x(ls[0])
    layers, packed = _layers(ls)
    rows = np.unique(np.concatenate([[0, 255, 256, M - 1], np.random.default_rng(71).integers(0, M, 12)]))
    xs = x.float().numpy()
    y_ref, ref = R.dit_block_ref(xs, layers, 12, HD, rows=rows, packed=packed)
    y_ex, ex = R.dit_block_ref(xs, layers, 12, HD, quantized=False, rows=rows)
    blk, xd = seeded_dit_block(M, DEV, seed=seed)
    blk.calibrate(xd, ts_mid=torch.tensor([ref["ts_mid"]], dtype=torch.float32, device=DEV))
    keep = {}
    y = to_np_f32(blk(xd, keep=keep)).astype(np.float64)[rows]
    torch.cuda.synchronize()
    st = _stages_from_gpu(keep, layers, packed, 12, ref["ts_mid"], rows=rows)
    assert_bf16_close(to_np_f32(keep["qkv_rmsnorm"])[rows], ref["qkv"][rows], "full block qkv rows")
    assert_attention_close(to_np_f32(keep["attention"]).astype(np.float64)[rows], st["attention"],
                           "full block attention rows")
    assert_bf16_close(to_np_f32(keep["out_proj"])[rows], st["out_proj"], "full block out_proj rows")
    assert_nvfp4_out_close(st["u_gpu"], st["up"], ref["ts_mid"], "full block up rows (NVFP4 out)",
                           y_gpu32=_up_fp32(blk, keep["out_proj"], rows))
    assert_bf16_close(y, st["down"], "full block down rows")
    # the chain as a whole
    o = to_np_f32(keep["out_proj"]).astype(np.float64)[rows]
    q_err_o = _rel(ref["out_proj"][rows], ex["out_proj"])
    assert _rel(o, ex["out_proj"]) <= 1.02 * q_err_o
    assert _rel(o, ref["out_proj"][rows]) <= 0.15 * q_err_o
    assert np.all(np.isfinite(y))
    q_err = _rel(y_ref, y_ex)
    assert _rel(y, y_ex) <= 1.02 * q_err, (_rel(y, y_ex), q_err)
    assert _rel(y, y_ref) <= 0.5 * q_err, (_rel(y, y_ref), q_err)


def test_cuda_graph_replay_matches_eager():
    # the whole block as one CUDA graph: the same kernels on the same inputs, so the same bytes
    blk, xd = seeded_dit_block(384, DEV, seed=72, heads=4, mlp=4096)
    blk.calibrate(xd)
    y_eager = blk(xd).clone()
    replay, y_graph = blk.graph(xd)
    replay()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y_eager)
    # a new input in the captured buffer gives that input's result
    x2 = torch.randn_like(xd.float()).to(torch.bfloat16)
    y2_eager = blk(x2).clone()
    xd.copy_(x2)
    replay()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y2_eager)
