"""Pins for the oracle's FP8 (E4M3, per-tensor scale) variant (CPU only).

The E4M3 encoder is pinned by its format (every finite code round-trips; hand-worked
roundings at midpoints, subnormals and saturation), the quantizer by exact cases (values on
the grid times a power-of-two scale, the amax element at +-448, a zero tensor), the GEMM by
brute force on integer-valued operands with power-of-two scales (every product and sum exact)
and by agreement with the NVFP4 GEMM oracle on operands that both formats hold exactly.
"""
import numpy as np
import pytest

from oracle import nvfp4_ref as R

F32 = np.float32


def test_e4m3_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = R.e4m3_decode(codes).astype(F32)
    assert np.array_equal(R.e4m3_encode(vals), codes)


@pytest.mark.parametrize("v,code", [
    (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (449.0, 0x7E), (464.0, 0x7E),          # midpoint of 448 and (absent) 480: saturates
    (1e30, 0x7E), (-1e30, 0xFE), (np.inf, 0x7E), (-np.inf, 0xFE),   # fp32 overflow saturates too
    (2.0 ** -9, 0x01),                     # smallest subnormal
    (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80),   # half of it: tie to the even code 0, sign kept
    (3 * 2.0 ** -11, 0x01),                # 0.75 of the smallest subnormal rounds up
    (1.0625, 0x38), (1.1875, 0x3A),        # midpoints 1|1.125 and 1.125|1.25: even codes
    (0.0, 0x00), (-0.0, 0x80),
    (2.0 ** -6, 0x08),                     # smallest normal
    (240.0, 0x77), (232.0, 0x76),          # 232 = midpoint of 224 (0x76) and 240 (0x77): even
])
def test_e4m3_encode_hand(v, code):
    assert int(R.e4m3_encode(np.array([v], F32))[0]) == code


def test_fp8_quantize_exact_on_grid_values():
    g = np.random.default_rng(0)
    codes = g.integers(0, 256, (5, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    ts = F32(2.0 ** -3)
    x = (R.e4m3_decode(codes) * float(ts)).astype(F32)
    got, t = R.fp8_quantize_ref(x, ts)
    # -0 and +0 decode to zeros of their sign and come back as the same code
    assert t == ts and np.array_equal(got, codes)


def test_fp8_quantize_dynamic_scale_maps_amax_to_448():
    g = np.random.default_rng(1)
    x = R.round_to_bf16(g.standard_normal((7, 96))).astype(F32)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    codes, ts = R.fp8_quantize_ref(x)
    assert ts == F32(F32(np.abs(x).max()) / F32(448.0))
    assert int(codes[i]) == (0xFE if x[i] < 0 else 0x7E)
    dq = R.fp8_dequantize_ref(codes, ts)
    # relative error of E4M3 rounding: at most half a mantissa step (2^-4) on normal values
    normal = np.abs(x) >= 2.0 ** -6 * float(ts)
    assert np.all(np.abs(dq - x)[normal] <= 2.0 ** -4 * np.abs(x)[normal] * (1 + 1e-6))


def test_fp8_quantize_degenerate_scales():
    x = np.zeros((3, 32), F32)
    codes, ts = R.fp8_quantize_ref(x)
    assert ts == 0 and not codes.any()
    codes, ts = R.fp8_quantize_ref(np.full((2, 16), 1e-30, F32), tensor_scale=F32(1e-39))
    assert not codes.any()  # ts below 2^-126: the tensor is stored as zeros


def test_fp8_pack_weights_layout_and_gated_order():
    g = np.random.default_rng(2)
    w = R.round_to_bf16(g.standard_normal((32, 8))).astype(F32)
    plain, ts = R.fp8_pack_weights_ref(w)
    gated, ts2 = R.fp8_pack_weights_ref(w, gated_interleave=True)
    assert ts == ts2 and plain.shape == (8, 32)
    col, _ = R.fp8_quantize_ref(np.ascontiguousarray(w.T), ts)
    assert np.array_equal(plain, col)
    for j in range(4):
        assert np.array_equal(gated[2 * j], col[j]) and np.array_equal(gated[2 * j + 1], col[4 + j])


def test_fp8_gemm_brute_force_integers():
    # operands with small integer values, power-of-two scales: every step is exact
    g = np.random.default_rng(3)
    M, N, K = 3, 5, 32
    ia = g.integers(-8, 9, (M, K))
    ib = g.integers(-8, 9, (N, K))
    a = R.e4m3_encode(ia.astype(F32))
    b = R.e4m3_encode(ib.astype(F32))
    bias = g.integers(-4, 5, N).astype(np.float64)
    y = R.fp8_gemm_ref(a, F32(0.5), b, F32(0.25), "bias", bias=bias)
    for m in range(M):
        for n in range(N):
            acc = 0
            for k in range(K):
                acc += int(ia[m, k]) * int(ib[n, k])
            assert y[m, n] == acc * 0.125 + bias[n]


@pytest.mark.parametrize("epi", ["bias", "head_rmsnorm", "gated_silu"])
def test_fp8_gemm_agrees_with_nvfp4_gemm_on_common_values(epi):
    # E2M1 values with block scale 1.0 and tensor scale 1 are E4M3 values too: both oracles
    # must give the same result on the same dequantized operands
    g = np.random.default_rng(4)
    M, N, K = 4, 16, 64
    qa = g.integers(0, 16, (M, K)).astype(np.uint8)
    qb = g.integers(0, 16, (N, K)).astype(np.uint8)
    one = np.uint8(0x38)
    sa = np.full((M, K // 16), one)
    sb = np.full((N, K // 16), one)
    kw = dict(bias=g.standard_normal(N), gamma=1 + 0.1 * g.standard_normal(N), head_dim=4,
              norm_cols=8 if epi == "head_rmsnorm" else 0, eps=1e-6)
    y4 = R.gemm_ref(qa, sa, F32(1), qb, sb, F32(1), epi, **kw)
    a8 = R.e4m3_encode(R.e2m1_decode(qa).astype(F32))
    b8 = R.e4m3_encode(R.e2m1_decode(qb).astype(F32))
    y8 = R.fp8_gemm_ref(a8, F32(1), b8, F32(1), epi, **kw)
    assert np.array_equal(y4, y8)
