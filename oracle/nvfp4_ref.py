"""CPU oracle for the NVFP4 linear layer with a fused epilogue.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module: only the test
suite, the smoke check in ``__graft_entry__`` and the CPU-baseline / reference legs of
``bench.py`` may call it. It shares no code, table or constant generator with the CUDA
path in ``nvfp4_gemm_act_b300/csrc``.

What it computes
----------------
The method is the one described on the page "How fal made Ideogram V4 6x faster"
(news.ditty.ir summary of fal's sub-second Ideogram V4 post):

* NVFP4 execution of the transformer's linears (paragraph "first step: run the transformer
  in NVFP4, a 4-bit float format native on Blackwell").
* Epilogue fusion: the small op that follows each GEMM is applied before the result is
  stored, so the output reaches HBM once (paragraph on epilogue fusion).
* Per-head RMSNorm with head_dim = 256 (same paragraph).
* Gated-SiLU: ``C = A @ B; output = SiLU(C[:, :N//2]) * C[:, N//2:]`` (the printed
  snippet), with B's columns rearranged in pairs at weight-packing time (the sentence after
  the snippet).

The NVFP4 tensor format used here: 4-bit E2M1 element codes, one unsigned E4M3 scale per
16 contiguous K-elements, one fp32 tensor scale ``ts = amax / (6 * 448)``.

Precision: steps that decide an integer (tensor scale, block scale code, element code) are
done in fp32, exactly as written below, because codes and scales are compared bit for bit.
Everything from dequantization on is fp64.

Readings taken where the pages are silent (each one is listed in the design notes):
  * per element, the value is multiplied by the fp32 reciprocal of the fp32 product
    dec(scale) * ts, then rounded to E2M1 (round to nearest, ties to even, saturating);
  * a block whose fp32 product dec(scale) * ts is below 2**-126 (this covers an all-zero
    block, a scale that underflows E4M3 and an all-zero tensor) stores scale code 0 and
    element codes +0;
  * a negative element that rounds to zero keeps its sign (code 0x8);
  * nibble order: element 2j in the low nibble of byte j, element 2j+1 in the high nibble;
  * bias is added before the norm / activation; HEAD_RMSNORM normalises columns
    [0, norm_cols) in heads of head_dim, other columns get the bias only;
  * gated weights interleave in pairs: packed column 2j = gate column j, 2j+1 = up column
    N/2 + j.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# ----------------------------------------------------------------------------------------
# Element formats, decoded from their bit fields (sign | exponent | mantissa).
# ----------------------------------------------------------------------------------------

E2M1_MAX = 6.0
E4M3_MAX = 448.0
TENSOR_SCALE_DIVISOR = 6.0 * 448.0  # = 2688: E2M1 max times E4M3 max
BLOCK = 16                          # K-elements per E4M3 block scale


def e2m1_decode(codes) -> np.ndarray:
    """Value of 4-bit E2M1 codes: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.

    exponent 0 is subnormal: m * 0.5; otherwise 2**(e-1) * (1 + m/2).
    """
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.power(2.0, e - 1))
    return np.where(sign == 1, -mag, mag)


def e4m3_decode(codes) -> np.ndarray:
    """Value of 8-bit E4M3 codes ("fn" variant: no infinities, S.1111.111 is NaN).

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
    m/8 * 2**-6, otherwise 2**(e-7) * (1 + m/8).
    """
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(sign == 1, -mag, mag)


# Non-negative grids, in code order (both are increasing in the code).
_E2M1_GRID = e2m1_decode(np.arange(8))             # codes 0..7
_E4M3_GRID = e4m3_decode(np.arange(0x7F))          # codes 0x00..0x7E (0x7F is NaN)


def _nearest_code(mag: np.ndarray, grid: np.ndarray, chunk: int = 1 << 16) -> np.ndarray:
    """Brute-force round-to-nearest onto ``grid`` (non-negative, increasing in the code).

    Every candidate code is measured; the closest wins and an exact tie goes to the even
    code (the one whose mantissa LSB is 0). Magnitudes above the largest grid point
    saturate to it (its distance is the smallest). ``mag`` must be finite and >= 0.
    """
    flat = np.asarray(mag, np.float64).reshape(-1)
    out = np.empty(flat.shape, np.uint8)
    parity_penalty = (np.arange(grid.size) & 1).astype(np.float64)  # 1 for odd codes
    for s in range(0, flat.size, chunk):
        v = flat[s:s + chunk, None]
        d = np.abs(v - grid[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # among the candidates (one, or two adjacent codes at a tie) take the even one
        score = np.where(cand, parity_penalty[None, :], np.inf)
        out[s:s + chunk] = np.argmin(score, axis=1).astype(np.uint8)
    return out.reshape(np.shape(mag))


def e2m1_encode(v) -> np.ndarray:
    """fp32 -> E2M1 code, round to nearest even, saturating at 6; sign kept (so -0.1 -> 0x8)."""
    v = np.asarray(v, F32)
    assert np.all(np.isfinite(v)), "non-finite input to the E2M1 encoder"
    code = _nearest_code(np.abs(v), _E2M1_GRID)
    return (code | (np.signbit(v).astype(np.uint8) << 3)).astype(np.uint8)


def e4m3_encode_nonneg(v) -> np.ndarray:
    """fp32 >= 0 -> E4M3 code, round to nearest even, saturating at 448 (satfinite)."""
    v = np.asarray(v, F32)
    assert np.all(np.isfinite(v)) and np.all(v >= 0)
    return _nearest_code(v, _E4M3_GRID)


# ----------------------------------------------------------------------------------------
# Quantizer: bf16 [M, K] -> E2M1 codes, E4M3 block scales, fp32 tensor scale.
# ----------------------------------------------------------------------------------------

FLT_MIN = F32(2.0 ** -126)


def tensor_scale_ref(x: np.ndarray) -> np.float32:
    """ts = amax(|x|) / (6 * 448), one fp32 IEEE division (amax of bf16 values is exact)."""
    x = np.asarray(x, F32)
    amax = F32(np.max(np.abs(x))) if x.size else F32(0.0)
    return F32(amax / F32(TENSOR_SCALE_DIVISOR))


def quantize_ref(x: np.ndarray, tensor_scale=None):
    """Quantize rows of ``x`` (fp32 array holding bf16 values) to NVFP4.

    Steps, per row and per block b of 16 contiguous K-elements:
      1. ts = amax / 2688 (fp32), unless ``tensor_scale`` is given (a static scale);
      2. s_f32 = bamax_b / fp32(6 * ts)                       (fp32 multiply, fp32 divide)
      3. s = E4M3(s_f32), nearest even, saturating at 448
      4. d = fp32(dec(s) * ts); if d < 2**-126 the block is zero: s = 0, codes = +0
      5. inv = fp32(1 / d); code = E2M1(fp32(x * inv)), nearest even, saturating at 6.

    Returns (codes [M, K] uint8 nibble values, scales [M, K/16] uint8 E4M3 codes, ts fp32).
    """
    x = np.asarray(x, F32)
    assert x.ndim == 2 and x.shape[1] % BLOCK == 0
    assert np.all(np.isfinite(x)), "non-finite inputs are outside the format"
    M, K = x.shape
    ts = tensor_scale_ref(x) if tensor_scale is None else F32(tensor_scale)
    nb = K // BLOCK
    codes = np.zeros((M, K), np.uint8)
    scales = np.zeros((M, nb), np.uint8)
    if M == 0 or K == 0 or not (ts > 0):
        return codes, scales, ts
    blocks = x.reshape(M, nb, BLOCK)
    bamax = np.abs(blocks).max(axis=2).astype(F32)
    six_ts = F32(F32(6.0) * ts)
    with np.errstate(over="ignore", under="ignore"):
        s_f32 = (bamax / six_ts).astype(F32)
    s_code = e4m3_encode_nonneg(np.minimum(s_f32, F32(E4M3_MAX * 2)))  # clamp keeps inf out
    dec_s = e4m3_decode(s_code).astype(F32)
    with np.errstate(over="ignore", under="ignore"):
        d = (dec_s * ts).astype(F32)
    live = d >= FLT_MIN
    d_safe = np.where(live, d, F32(1.0)).astype(F32)
    inv = (F32(1.0) / d_safe).astype(F32)
    v = (blocks * inv[:, :, None]).astype(F32)
    q = e2m1_encode(v)
    q = np.where(live[:, :, None], q, np.uint8(0))
    s_code = np.where(live, s_code, np.uint8(0)).astype(np.uint8)
    return q.reshape(M, K).astype(np.uint8), s_code, ts


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[M, K] nibble codes -> [M, K/2] bytes; element 2j in the low nibble."""
    c = np.asarray(codes, np.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[M, K/2] bytes -> [M, K] nibble codes."""
    p = np.asarray(packed, np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


# ----------------------------------------------------------------------------------------
# Block-scale storage layout (the layout the tensor cores read for 1-D block scaling).
# ----------------------------------------------------------------------------------------

def scale_tile_rows(rows: int) -> int:
    return -(-rows // 128) * 128


def scales_bytes(rows: int, K: int) -> int:
    """Bytes of the tiled scale buffer: rows padded to 128, 512-byte tiles of 128 x 4 blocks."""
    return scale_tile_rows(rows) // 128 * (K // 64) * 512


def scale_offset(r, kb, K: int):
    """Byte offset of the scale of row r, 16-element block kb in the tiled buffer.

    Tiles of 128 rows x 4 blocks (512 B), K-tiles fastest; inside a tile, row r sits in
    16-byte line r % 32 at 4-byte slot (r // 32) % 4, block kb % 4 is the byte in the slot.
    """
    r = np.asarray(r, np.int64)
    kb = np.asarray(kb, np.int64)
    tile = (r // 128) * (K // 64) + kb // 4
    return tile * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (kb % 4)


def tile_scales(scales: np.ndarray, K: int) -> np.ndarray:
    """[rows, K/16] scale codes -> tiled byte buffer (padding zero)."""
    rows = scales.shape[0]
    buf = np.zeros(scales_bytes(rows, K), np.uint8)
    r, kb = np.meshgrid(np.arange(rows), np.arange(K // 16), indexing="ij")
    buf[scale_offset(r, kb, K)] = scales
    return buf


def untile_scales(buf: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Tiled byte buffer -> [rows, K/16] scale codes."""
    r, kb = np.meshgrid(np.arange(rows), np.arange(K // 16), indexing="ij")
    return np.asarray(buf, np.uint8)[scale_offset(r, kb, K)]


# ----------------------------------------------------------------------------------------
# Weight packing: W [K, N] -> K-major W^T [N, K], optional pair interleave, quantize.
# ----------------------------------------------------------------------------------------

def gated_permutation(N: int) -> np.ndarray:
    """perm[p] = original column stored at packed position p (pairs: gate j, up N/2 + j)."""
    assert N % 2 == 0
    h = N // 2
    perm = np.empty(N, np.int64)
    perm[0::2] = np.arange(h)
    perm[1::2] = h + np.arange(h)
    return perm


def interleave_columns(w: np.ndarray) -> np.ndarray:
    """Reorder the columns of w [.., N] into packed (gate, up) pairs."""
    return np.asarray(w)[..., gated_permutation(w.shape[-1])]


def deinterleave_columns(wp: np.ndarray) -> np.ndarray:
    """Inverse of interleave_columns."""
    perm = gated_permutation(wp.shape[-1])
    out = np.empty_like(np.asarray(wp))
    out[..., perm] = wp
    return out


def pack_weights_ref(w: np.ndarray, gated_interleave: bool = False, tensor_scale=None):
    """W [K, N] -> quantize_ref(W^T) with rows in packed order. Returns (codes, scales, ts)."""
    w = np.asarray(w, F32)
    wt = w.T
    if gated_interleave:
        wt = wt[gated_permutation(w.shape[1])]
    return quantize_ref(np.ascontiguousarray(wt), tensor_scale)


# ----------------------------------------------------------------------------------------
# GEMM + epilogue, fp64 from dequantization on.
# ----------------------------------------------------------------------------------------

def dequantize_ref(codes: np.ndarray, scales: np.ndarray, ts) -> np.ndarray:
    """x_hat = dec(code) * dec(scale of its block) * ts, in fp64."""
    M, K = codes.shape
    s = np.repeat(e4m3_decode(scales), BLOCK, axis=1)
    return e2m1_decode(codes) * s * float(ts)


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def gated_silu_ref(c: np.ndarray) -> np.ndarray:
    """The page's gated-SiLU on an unpermuted GEMM result: SiLU(C[:, :N//2]) * C[:, N//2:]."""
    n = c.shape[1]
    return silu(c[:, : n // 2]) * c[:, n // 2:]


def head_rmsnorm_ref(z: np.ndarray, gamma: np.ndarray, head_dim: int, norm_cols: int,
                     eps: float) -> np.ndarray:
    """Columns [0, norm_cols): per head of head_dim columns, z / sqrt(mean(z^2) + eps) * gamma."""
    y = np.array(z, np.float64, copy=True)
    M = z.shape[0]
    heads = z[:, :norm_cols].reshape(M, norm_cols // head_dim, head_dim)
    ms = np.mean(heads * heads, axis=2, keepdims=True)
    y[:, :norm_cols] = (heads / np.sqrt(ms + eps)).reshape(M, norm_cols) * np.asarray(
        gamma, np.float64)[None, :norm_cols]
    return y


EPI_BIAS, EPI_HEAD_RMSNORM, EPI_GATED_SILU = "bias", "head_rmsnorm", "gated_silu"


def gemm_ref(a_codes, a_scales, a_ts, b_codes, b_scales, b_ts, epilogue=EPI_BIAS,
             bias=None, gamma=None, head_dim=256, norm_cols=0, eps=1e-6):
    """y = epilogue(A_hat @ B_hat^T + bias) in fp64.

    A: [M, K] codes with [M, K/16] scales; B: [N, K] codes (K-major, packed column order
    for the gated epilogue) with [N, K/16] scales. ``bias`` is indexed by ORIGINAL column.
    For GATED_SILU the packed B is returned to original column order first and the page's
    formula SiLU(C[:, :N//2]) * C[:, N//2:] is applied to C = A_hat @ B^T + bias.
    """
    A = dequantize_ref(a_codes, a_scales, a_ts)
    B = dequantize_ref(b_codes, b_scales, b_ts)
    return _gemm_epilogue_ref(A, B, epilogue, bias, gamma, head_dim, norm_cols, eps)


def _gemm_epilogue_ref(A, B, epilogue, bias, gamma, head_dim, norm_cols, eps):
    """epilogue(A @ B^T + bias) in fp64 for dequantized A [M, K] and B [N, K] (B's rows in
    packed order for the gated epilogue, returned to original column order here)."""
    N = B.shape[0]
    if epilogue == EPI_GATED_SILU:
        B = B[np.argsort(gated_permutation(N))]  # packed rows back to original column order
    C = A @ B.T
    if bias is not None:
        C = C + np.asarray(bias, np.float64)[None, :]
    if epilogue == EPI_BIAS:
        return C
    if epilogue == EPI_HEAD_RMSNORM:
        return head_rmsnorm_ref(C, gamma, head_dim, norm_cols, eps)
    if epilogue == EPI_GATED_SILU:
        return gated_silu_ref(C)
    raise ValueError(epilogue)


def gemm_block_form_ref(a_codes, a_scales, a_ts, b_codes, b_scales, b_ts):
    """acc[m, n] = sum_kb sA[m,kb] sB[n,kb] sum_{k in kb} qA[m,k] qB[n,k]; returns ts_A ts_B acc.

    The block-scaled form a tensor core evaluates; fp64, loops over blocks (small inputs).
    """
    qa = e2m1_decode(a_codes)
    qb = e2m1_decode(b_codes)
    sa = e4m3_decode(a_scales)
    sb = e4m3_decode(b_scales)
    M, K = qa.shape
    N = qb.shape[0]
    acc = np.zeros((M, N))
    for kb in range(K // BLOCK):
        blk = slice(kb * BLOCK, (kb + 1) * BLOCK)
        acc += sa[:, kb, None] * sb[None, :, kb] * (qa[:, blk] @ qb[:, blk].T)
    return float(a_ts) * float(b_ts) * acc


# ----------------------------------------------------------------------------------------
# Output rounding.
# ----------------------------------------------------------------------------------------

def round_to_bf16(y: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (8 significant bits, ties to even), returned as fp64. A zero
    keeps its sign (IEEE rounding: -0 rounds to -0, as a tiny negative value does)."""
    y = np.asarray(y, np.float64)
    out = np.where(y == 0, y, 0.0)
    nz = (y != 0) & np.isfinite(y)
    _, e = np.frexp(y[nz])                      # |y| = m * 2**e, m in [0.5, 1)
    quantum = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
    out[nz] = np.rint(y[nz] / quantum) * quantum
    out[~np.isfinite(y)] = y[~np.isfinite(y)]
    return out


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |y| (for |y| a bf16 value or between two)."""
    y = np.asarray(y, np.float64)
    _, e = np.frexp(np.where(y == 0, 1.0, y))
    return np.ldexp(1.0, np.maximum(e - 1, -126) - 7)


# ----------------------------------------------------------------------------------------
# FP8 (E4M3) variant: per-tensor scaled operands, the same fused epilogues.
#
# Page "WaveSpeedAI x DataCrunch: FLUX real-time image inference on B200" (wavespeed.ai) lists
# BF16/FP8 mixed precision through Blackwell's Transformer Engine among its optimizations;
# page "FLUX.1-dev inference optimization with LoRAs" (aitime.ge) calls FP8 quantization lossy
# but the best speed/memory trade-off. Neither fixes the scheme; read here as one fp32 scale
# per tensor, ts = amax / 448 (E4M3's largest value), and per element
# code = E4M3(fp32(x * fp32(1 / ts))), round to nearest even, saturating at 448, sign kept
# (a negative value that rounds to zero is 0x80). A tensor with ts < 2**-126 (all zeros, or
# so small that 1 / ts overflows) stores codes +0.
# ----------------------------------------------------------------------------------------

FP8_TENSOR_SCALE_DIVISOR = 448.0


def e4m3_encode(v) -> np.ndarray:
    """fp32 -> signed E4M3 code: sign bit | E4M3 code of |v| (nearest even, saturating). An
    fp32 product that overflowed to +-inf lies beyond 448 too and saturates the same way."""
    v = np.asarray(v, F32)
    assert not np.any(np.isnan(v))
    mag = np.minimum(np.abs(v), F32(2 * E4M3_MAX))  # anything above 448 saturates to 448
    return (e4m3_encode_nonneg(mag) | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)


def fp8_tensor_scale_ref(x: np.ndarray) -> np.float32:
    """ts = amax(|x|) / 448, one fp32 IEEE division."""
    x = np.asarray(x, F32)
    amax = F32(np.max(np.abs(x))) if x.size else F32(0.0)
    return F32(amax / F32(FP8_TENSOR_SCALE_DIVISOR))


def fp8_quantize_ref(x: np.ndarray, tensor_scale=None):
    """x (fp32 array holding bf16 values) [M, K] -> (E4M3 codes [M, K] uint8, ts fp32).

    ts = amax / 448 unless ``tensor_scale`` (a static scale) is given; inv = fp32(1 / ts);
    code = E4M3(fp32(x * inv)).
    """
    x = np.asarray(x, F32)
    assert np.all(np.isfinite(x)), "non-finite inputs are outside the format"
    ts = fp8_tensor_scale_ref(x) if tensor_scale is None else F32(tensor_scale)
    if not (ts >= FLT_MIN):
        return np.zeros(x.shape, np.uint8), ts
    inv = F32(F32(1.0) / ts)
    with np.errstate(over="ignore"):
        v = (x * inv).astype(F32)
    return e4m3_encode(v), ts


def fp8_pack_weights_ref(w: np.ndarray, gated_interleave: bool = False, tensor_scale=None):
    """W [K, N] -> fp8_quantize_ref(W^T) with rows in packed order: (codes [N, K], ts)."""
    wt = np.asarray(w, F32).T
    if gated_interleave:
        wt = wt[gated_permutation(wt.shape[0])]
    return fp8_quantize_ref(np.ascontiguousarray(wt), tensor_scale)


def fp8_dequantize_ref(codes: np.ndarray, ts) -> np.ndarray:
    """x_hat = dec(code) * ts in fp64."""
    return e4m3_decode(codes) * float(ts)


def fp8_gemm_ref(a_codes, a_ts, b_codes, b_ts, epilogue=EPI_BIAS, bias=None, gamma=None,
                 head_dim=256, norm_cols=0, eps=1e-6):
    """y = epilogue(A_hat @ B_hat^T + bias) in fp64 for E4M3 A [M, K] and B [N, K] (K-major,
    packed column order for the gated epilogue); the epilogues are those of gemm_ref."""
    A = fp8_dequantize_ref(a_codes, a_ts)
    B = fp8_dequantize_ref(b_codes, b_ts)
    return _gemm_epilogue_ref(A, B, epilogue, bias, gamma, head_dim, norm_cols, eps)


# ----------------------------------------------------------------------------------------
# One DiT block's linears chained, attention between the first two.
# ----------------------------------------------------------------------------------------

def attention_ref(q, k, v) -> np.ndarray:
    """Scaled dot-product attention per head, every query over every key, fp64.

    q, k, v: [heads, M, d]. out[h, i] = sum_j p[h, i, j] v[h, j] with
    p[h, i, :] = softmax_j(q[h, i] . k[h, j] / sqrt(d)). The pages name attention as the other
    large op of the transformer's pass without defining it; this is the textbook form with no
    mask (all tokens of a DiT block see each other). Subtracting a row's largest score before
    exp leaves p unchanged and keeps exp finite.
    """
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    out = np.empty((q.shape[0], q.shape[1], v.shape[2]))
    for h in range(q.shape[0]):
        s = (q[h] @ k[h].T) / np.sqrt(q.shape[2])
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[h] = (p / p.sum(axis=1, keepdims=True)) @ v[h]
    return out


def _linear_ref(x, w, bias, epilogue, quantized, gamma=None, head_dim=256, norm_cols=0, eps=1e-6,
                tensor_scale=None, packed=None):
    """One linear layer of the block: quantized, the layer as the NVFP4 path defines it (x and
    W quantized with their own amax scales unless ``tensor_scale`` fixes x's; fp64 GEMM and
    epilogue); not quantized, the exact fp64 layer epilogue(x @ W + bias). ``packed``: W
    already passed through pack_weights_ref (with the layer's interleave), to skip repacking."""
    kw = dict(bias=bias, gamma=gamma, head_dim=head_dim, norm_cols=norm_cols, eps=eps)
    if quantized:
        a = quantize_ref(x, tensor_scale)
        b = packed if packed is not None else pack_weights_ref(w, gated_interleave=(epilogue == EPI_GATED_SILU))
        return gemm_ref(*a, *b, epilogue, **kw)
    c = np.asarray(x, np.float64) @ np.asarray(w, np.float64)
    if bias is not None:
        c = c + np.asarray(bias, np.float64)[None, :]
    if epilogue == EPI_BIAS:
        return c
    if epilogue == EPI_HEAD_RMSNORM:
        return head_rmsnorm_ref(c, gamma, head_dim, norm_cols, eps)
    return gated_silu_ref(c)


def dit_block_ref(x, layers, heads: int, head_dim: int, eps: float = 1e-6, ts_mid=None,
                  quantized: bool = True, rows=None, packed=None):
    """One DiT block's linears with attention between the first two, in the order of the page
    "How fal made Ideogram V4 6x faster" (each large GEMM followed by its small op, fused).

    ``layers``: four (W [K, N], bias [N] or None, gamma or None) for the QKV projection (gamma
    over the Q and K columns), the output projection, the gated up-projection (W's columns are
    gate | up halves) and the down-projection. hidden = heads * head_dim.

    Steps; "bf16" is the rounding of a layer's output as it is stored between layers:
      1. t = bf16(head_rmsnorm(x W_qkv + b_qkv)) over columns [0, 2 hidden) in heads of head_dim
      2. q, k, v = t's three column blocks of width hidden; head h of each is its columns
         [h head_dim, (h+1) head_dim)
      3. a = bf16(attention(q, k, v)), heads side by side again
      4. o = bf16(a W_o + b_o)
      5. u = bf16(SiLU(o W_g + b_g) * (o W_u + b_u)); the NVFP4 scale handed to the next layer is
         ``ts_mid`` if given, else amax(u) / 2688 (the static scale a calibration pass sets)
      6. y = bf16(quant(u; ts_mid) W_down + b_down)
    ``quantized`` False: every quantization and bf16 rounding dropped, the exact fp64 function
    the quantized block approximates. ``rows`` (token indices): the output of those tokens
    only; every token's K and V still enter the attention, and the dynamic scales of the
    quantized block's activations are still those of all tokens, so the stages that feed a
    dynamic scale run over all tokens and the last two layers over ``rows`` (the default
    ts_mid is then amax / 2688 over those rows). ``packed``: the four weights already passed
    through pack_weights_ref (the up-projection's with the gated interleave), to skip
    repacking them. Returns (y, dict of the intermediates, for all tokens or for ``rows``
    where a stage ran only there, and ts_mid).
    """
    pk = packed if packed is not None else (None, None, None, None)
    hidden = heads * head_dim
    rnd = round_to_bf16 if quantized else (lambda z: np.asarray(z, np.float64))
    (w1, b1, g1), (w2, b2, _), (w3, b3, _), (w4, b4, _) = layers
    M = x.shape[0]
    t = rnd(_linear_ref(x, w1, b1, EPI_HEAD_RMSNORM, quantized, gamma=g1, head_dim=head_dim,
                        norm_cols=2 * hidden, eps=eps, packed=pk[0]))
    qkv = t.reshape(M, 3, heads, head_dim).transpose(1, 2, 0, 3)    # [3, heads, M, head_dim]
    q_rows = qkv[0] if (rows is None or quantized) else qkv[0][:, rows]
    a = rnd(attention_ref(q_rows, qkv[1], qkv[2]).transpose(1, 0, 2).reshape(-1, hidden))
    o = rnd(_linear_ref(a, w2, b2, EPI_BIAS, quantized, packed=pk[1]))
    o_ts = tensor_scale_ref(o) if quantized else None
    if rows is not None and quantized:
        o_in = o[rows]
    else:
        o_in = o
    u = rnd(_linear_ref(o_in, w3, b3, EPI_GATED_SILU, quantized, tensor_scale=o_ts, packed=pk[2]))
    if quantized and ts_mid is None:
        ts_mid = tensor_scale_ref(u)
    y = rnd(_linear_ref(u, w4, b4, EPI_BIAS, quantized, tensor_scale=ts_mid, packed=pk[3]))
    return y, {"qkv": t, "attention": a, "out_proj": o, "up": u, "ts_mid": ts_mid}
