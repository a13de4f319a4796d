"""One DiT block's linears chained on the GPU, attention between the first two:

  x -> quantize -> QKV GEMM + bias + per-head RMSNorm of Q and K (bf16)
    -> attention over all tokens (this package's attention kernel; torch's
       scaled_dot_product_attention with attention_impl="torch")
    -> quantize -> output-projection GEMM + bias (bf16)
    -> quantize -> gated up-projection GEMM, SiLU(gate) * up, written as NVFP4 (static scale)
    -> down-projection GEMM + bias (bf16)

Page "How fal made Ideogram V4 6x faster" (news.ditty.ir), epilogue-fusion paragraphs: the
transformer's linears run in NVFP4, and the small op after each large GEMM (RMSNorm,
gated-SiLU) is applied in the GEMM's epilogue so its output reaches HBM once; a pass costs
the sum of its layers. The up-projection hands the down-projection NVFP4 directly, so the
widest activation never round-trips through HBM in bf16. Residual connections and the
timestep modulation of a full DiT block are not part of that path and are left out.

Every GEMM, epilogue, quantizer and (by default) the attention runs in this package's kernels.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import torch
import torch.nn.functional as F

from . import attention as attention_fwd
from . import nvfp4_gemm, nvfp4_gemm_nvfp4_out, nvfp4_pack_weights, nvfp4_quantize
from . import workloads as W

STAGES = ("qkv_rmsnorm", "attention", "out_proj", "up_gated_silu", "down")


class DitBlockLinears:
    """The block's weights packed to NVFP4 on one device, and its forward pass.

    Weights are [K, N] (x @ W), bf16; biases fp32 [N] or None; gamma fp32 [2 * hidden]
    (the Q and K columns). w_up's columns are the gate half then the up half.
    """

    def __init__(self, w_qkv, b_qkv, gamma, w_o, b_o, w_up, b_up, w_down, b_down, heads: int,
                 head_dim: int = 256, eps: float = 1e-6, device="cuda:0", attention_impl: str = "kernel"):
        assert attention_impl in ("kernel", "torch")
        self.attention_impl = attention_impl
        self.heads, self.head_dim, self.eps = heads, head_dim, eps
        self.hidden = heads * head_dim
        self.mlp = w_up.shape[1] // 2
        h, m = self.hidden, self.mlp
        assert w_qkv.shape == (h, 3 * h) and w_o.shape == (h, h)
        assert w_up.shape == (h, 2 * m) and w_down.shape == (m, h)
        assert gamma is not None and gamma.numel() == 2 * h
        dev = torch.device(device)
        self.device = dev

        def put(t):
            return None if t is None else t.to(dev)

        self.qb = {"qkv": nvfp4_pack_weights(w_qkv.to(dev)), "o": nvfp4_pack_weights(w_o.to(dev)),
                   "up": nvfp4_pack_weights(w_up.to(dev), gated_interleave=True),
                   "down": nvfp4_pack_weights(w_down.to(dev))}
        self.bias = {"qkv": put(b_qkv), "o": put(b_o), "up": put(b_up), "down": put(b_down)}
        self.gamma = put(gamma)
        self.ts_mid: Optional[torch.Tensor] = None  # static NVFP4 scale of the up-projection output

    # the stages -------------------------------------------------------------------------
    def qkv_rmsnorm(self, x):
        return nvfp4_gemm(nvfp4_quantize(x), self.qb["qkv"], "head_rmsnorm", bias=self.bias["qkv"],
                          gamma=self.gamma, head_dim=self.head_dim, norm_cols=2 * self.hidden, eps=self.eps)

    def attention(self, t):
        """t [M, 3 hidden] (Q | K | V, heads side by side in each) -> [M, hidden]: this
        package's attention kernel, or torch's scaled_dot_product_attention."""
        if self.attention_impl == "kernel":
            return attention_fwd(t, self.heads, self.head_dim)
        return self.attention_torch(t)

    def attention_torch(self, t):
        M = t.shape[0]
        q, k, v = t.view(M, 3, self.heads, self.head_dim).permute(1, 2, 0, 3).unsqueeze(1).unbind(0)
        a = F.scaled_dot_product_attention(q, k, v)                  # [1, heads, M, head_dim]
        return a[0].transpose(0, 1).reshape(M, self.hidden)          # copies into [M, hidden]

    def out_proj(self, a):
        return nvfp4_gemm(nvfp4_quantize(a), self.qb["o"], "bias", bias=self.bias["o"])

    def up_gated_silu(self, o):
        if self.ts_mid is None:
            raise RuntimeError("DitBlockLinears: calibrate() sets the up-projection's output scale first")
        return nvfp4_gemm_nvfp4_out(nvfp4_quantize(o), self.qb["up"], "gated_silu", self.ts_mid,
                                    bias=self.bias["up"])

    def down(self, u):
        return nvfp4_gemm(u, self.qb["down"], "bias", bias=self.bias["down"])

    # ------------------------------------------------------------------------------------
    def calibrate(self, x: torch.Tensor, ts_mid: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Sets the static NVFP4 scale of the up-projection output: ``ts_mid`` (a one-element
        fp32 device tensor) if given, else the tensor scale amax / 2688 that nvfp4_quantize
        computes for that output on input ``x`` (one pass of the first layers with a bf16
        up-projection output, then the library's quantizer, whose tensor scale is kept)."""
        if ts_mid is None:
            o = self.out_proj(self.attention(self.qkv_rmsnorm(x)))
            u = nvfp4_gemm(nvfp4_quantize(o), self.qb["up"], "gated_silu", bias=self.bias["up"])
            ts_mid = nvfp4_quantize(u).ts
        self.ts_mid = ts_mid.to(self.device, torch.float32).reshape(1).contiguous()
        return self.ts_mid

    def forward(self, x: torch.Tensor, timings: Optional[Dict[str, List[float]]] = None,
                keep: Optional[Dict[str, torch.Tensor]] = None) -> torch.Tensor:
        """x: bf16 [M, hidden] on the device -> bf16 [M, hidden]. ``timings``: each stage's
        CUDA-event time in ms is appended under its name (events on the current stream, one
        synchronize at the end). ``keep``: each stage's output is stored under its name."""
        evs = []
        y = x
        for name in STAGES:
            fn = getattr(self, name)
            if timings is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                y = fn(y)
                e1.record()
                evs.append((name, e0, e1))
            else:
                y = fn(y)
            if keep is not None:
                keep[name] = y
        if timings is not None:
            torch.cuda.synchronize()
            for name, e0, e1 in evs:
                timings.setdefault(name, []).append(e0.elapsed_time(e1))
        return y

    __call__ = forward

    def graph(self, x: torch.Tensor):
        """The forward pass on the device buffer ``x`` captured once as a CUDA graph (after one
        eager pass, which also sets up every kernel's launch attributes). Returns (replay, y):
        ``replay()`` re-runs the whole block on the current contents of ``x`` with one graph
        launch and writes the result into ``y``."""
        if self.ts_mid is None:
            raise RuntimeError("DitBlockLinears: calibrate() sets the up-projection's output scale first")
        side = torch.cuda.Stream(device=x.device)
        side.wait_stream(torch.cuda.current_stream(x.device))
        with torch.cuda.stream(side):
            self.forward(x)
        torch.cuda.current_stream(x.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            y = self.forward(x)
        return g.replay, y

    def gemm_flops(self, M: int) -> int:
        h, m = self.hidden, self.mlp
        return 2 * M * h * (3 * h + h + 2 * m) + 2 * M * m * h


def seeded_dit_block(M: int = 4608, device="cuda:0", seed: Optional[int] = None,
                     heads: int = W.DIT_HEADS, mlp: int = 12288, attention_impl: str = "kernel"):
    """The seeded synthetic block (random-initialised weights of the four layers, drawn by
    ``workloads.dit_block``) on ``device``, and its bf16 input [M, heads * 256]."""
    qkv, o, up, down = W.dit_block(M, seed, heads=heads, mlp=mlp)
    blk = DitBlockLinears(W.make_w(qkv), W.make_bias(qkv), W.make_gamma(qkv), W.make_w(o), W.make_bias(o),
                          W.make_w(up), W.make_bias(up), W.make_w(down), W.make_bias(down),
                          heads=heads, head_dim=qkv.head_dim, eps=qkv.eps, device=device,
                          attention_impl=attention_impl)
    return blk, W.make_x(qkv).to(device)
