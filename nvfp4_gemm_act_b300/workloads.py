"""Seeded synthetic inputs shaped like the DiT linears of the fused NVFP4 GEMM path.

Random draws only: this module holds none of the method's arithmetic (no quantization, no
GEMM, no epilogue). Tests, the oracle checks and ``bench.py`` all draw their inputs here,
so the CUDA path and the CPU oracle see identical bf16 / fp32 values.

Shapes follow a FLUX-class DiT block (hidden 3072, MLP 12288, 12 heads x head_dim 256,
4608 tokens = 4096 image + 512 text):

  tiny_bias       X [128, 256] ~ N(0,1) seed 0; W [256, 256] ~ N(0, 0.02) seed 1; bias N(0, 0.01)
  qkv_rmsnorm     X [4608, 3072] ~ N(0,1), 1% of channels x20; W [3072, 9216] ~ N(0, 0.02);
                  bias N(0, 0.01) on all 9216 columns; RMSNorm over the Q and K heads
                  (norm_cols 6144, head_dim 256, eps 1e-6), gamma ~ 1 + N(0, 0.1)
  gated_up        X [4608, 3072] ~ N(0,1); W [3072, 24576] ~ N(0, 0.02) (gate | up halves),
                  no bias; output SiLU(C[:, :12288]) * C[:, 12288:]
  down_bias       X [4608, 12288] ~ 0.5 * Student-t(df=3); W [12288, 3072] ~ N(0, 0.02);
                  bias N(0, 0.01)

One DiT block chains four linears (attention between the first two): qkv_rmsnorm ->
attention -> out_proj (W [3072, 3072] ~ N(0, 0.02), bias N(0, 0.01), seed 5) -> gated_up ->
down_bias. The block's input is qkv_rmsnorm's X; every later layer takes the previous
stage's output, so only the weights, biases and gain of those layers are drawn.

Every array is drawn in fp64 from ``numpy.random.default_rng((seed, stream))`` (stream 0:
X, 1: W, 2: bias, 3: gamma, 4: outlier channels; all but X use the layer's seed,
which ``with_m`` keeps when it reseeds the activations) and rounded to bf16 (X, W) or fp32
(bias, gamma) by torch's round-to-nearest-even conversion.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

EPI_BIAS, EPI_HEAD_RMSNORM, EPI_GATED_SILU = "bias", "head_rmsnorm", "gated_silu"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int                      # GEMM N (packed width; the gated output is N/2 wide)
    epilogue: str
    seed: int
    x_dist: str = "normal"      # normal | normal_outliers | student_t
    w_std: float = 0.02
    bias_std: Optional[float] = 0.01
    head_dim: int = 256
    norm_cols: int = 0
    eps: float = 1e-6
    gamma_std: float = 0.1
    w_seed: Optional[int] = None  # weights / bias / gamma seed; None = `seed`

    @property
    def out_cols(self) -> int:
        return self.N // 2 if self.epilogue == EPI_GATED_SILU else self.N

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def layer_seed(self) -> int:
        return self.seed if self.w_seed is None else self.w_seed

    def with_m(self, M: int, seed: Optional[int] = None) -> "Workload":
        """The same layer (weights, bias, gamma) on M tokens; `seed` reseeds the activations."""
        return dataclasses.replace(self, M=M, seed=self.seed if seed is None else seed,
                                   w_seed=self.layer_seed, name=f"{self.name}_m{M}")


TINY_BIAS = Workload("tiny_bias", 128, 256, 256, EPI_BIAS, seed=0)
QKV_RMSNORM = Workload("qkv_rmsnorm", 4608, 3072, 9216, EPI_HEAD_RMSNORM, seed=2,
                       x_dist="normal_outliers", norm_cols=6144)
GATED_UP = Workload("gated_up", 4608, 3072, 24576, EPI_GATED_SILU, seed=3, bias_std=None)
DOWN_BIAS = Workload("down_bias", 4608, 12288, 3072, EPI_BIAS, seed=4, x_dist="student_t")

OUT_PROJ = Workload("out_proj", 4608, 3072, 3072, EPI_BIAS, seed=5)

WORKLOADS = {w.name: w for w in (TINY_BIAS, QKV_RMSNORM, GATED_UP, DOWN_BIAS)}

# One DiT block's linears in order; the 12 attention heads of 256 sit between the first two.
DIT_BLOCK = (QKV_RMSNORM, OUT_PROJ, GATED_UP, DOWN_BIAS)
DIT_HEADS = 12


def dit_block(M: int = 4608, seed: Optional[int] = None, heads: int = DIT_HEADS, mlp: int = 12288):
    """The block's four layers on M tokens (`seed` reseeds the block input). Fewer heads or a
    narrower MLP give a smaller block of the same structure (head_dim 256 throughout), its
    weights drawn from the same seeds at the smaller shapes."""
    h = heads * QKV_RMSNORM.head_dim
    shapes = ((h, 3 * h, 2 * h), (h, h, 0), (h, 2 * mlp, 0), (mlp, h, 0))
    out = []
    for i, (w, (K, N, norm_cols)) in enumerate(zip(DIT_BLOCK, shapes)):
        w = w.with_m(M, seed if i == 0 else None)
        if (K, N) != (w.K, w.N):
            w = dataclasses.replace(w, K=K, N=N, norm_cols=norm_cols, name=f"{w.name}_h{h}")
        out.append(w)
    return tuple(out)

# Batch sweep: the three DiT GEMMs at M in {512, 1024, 4608, 9216, 18432}; activations of
# the i-th size drawn with seed 10 + i, each layer keeping its weights.
SWEEP_M = (512, 1024, 4608, 9216, 18432)


def sweep_workloads():
    out = []
    for i, m in enumerate(SWEEP_M):
        for base in (QKV_RMSNORM, GATED_UP, DOWN_BIAS):
            out.append(base.with_m(m, seed=10 + i))
    return out


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng((seed, stream))


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def make_x(w: Workload, rows: Optional[int] = None) -> torch.Tensor:
    """Activations X [M, K] as a CPU bf16 tensor (``rows`` < M draws only the first rows'
    worth of the same stream, identical to the leading rows of the full draw)."""
    M = w.M if rows is None else rows
    g = _rng(w.seed, 0)
    if w.x_dist in ("normal", "normal_outliers"):
        x = g.standard_normal((M, w.K))
    elif w.x_dist == "student_t":
        x = 0.5 * g.standard_t(3.0, size=(M, w.K))
    else:
        raise ValueError(w.x_dist)
    if w.x_dist == "normal_outliers":
        n_out = int(round(0.01 * w.K))
        ch = _rng(w.layer_seed, 4).choice(w.K, n_out, replace=False)  # a property of the layer input
        x[:, ch] *= 20.0
    return _bf16(x)


def make_w(w: Workload) -> torch.Tensor:
    """Weights W [K, N] (row-major, as a linear layer's x @ W) as a CPU bf16 tensor."""
    return _bf16(w.w_std * _rng(w.layer_seed, 1).standard_normal((w.K, w.N)))


def make_bias(w: Workload) -> Optional[torch.Tensor]:
    """fp32 bias indexed by original output column ([N]), or None."""
    if w.bias_std is None:
        return None
    return torch.from_numpy((w.bias_std * _rng(w.layer_seed, 2).standard_normal(w.N)).astype(np.float32))


def make_gamma(w: Workload) -> Optional[torch.Tensor]:
    """fp32 RMSNorm gain, one value per normalised column ([norm_cols]), or None."""
    if w.epilogue != EPI_HEAD_RMSNORM:
        return None
    g = 1.0 + w.gamma_std * _rng(w.layer_seed, 3).standard_normal(w.norm_cols)
    return torch.from_numpy(g.astype(np.float32))


def attention_qkv(M: int, heads: int, seed: int, q_scale: float = 1.0, head_dim: int = 256) -> torch.Tensor:
    """A QKV projection output [M, 3 * heads * head_dim] as a CPU bf16 tensor: Q, K, V ~ N(0, 1),
    Q times ``q_scale`` (larger logits), drawn from ``default_rng((seed, 5))``."""
    x = _rng(seed, 5).standard_normal((M, 3 * heads * head_dim))
    x[:, : heads * head_dim] *= q_scale
    return _bf16(x)

