"""Pins for the oracle's GEMM and epilogues (CPU only)."""
import math
import os

import numpy as np
import pytest

from oracle import nvfp4_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_codes(rng, rows, K):
    codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    scales = rng.integers(0x20, 0x50, (rows, K // 16)).astype(np.uint8)
    return codes, scales


def test_dense_matmul_equals_block_form():
    rng = np.random.default_rng(0)
    for (M, N, K) in [(1, 1, 16), (3, 5, 48), (7, 4, 64), (16, 9, 96)]:
        a, sa = _rand_codes(rng, M, K)
        b, sb = _rand_codes(rng, N, K)
        dense = R.gemm_ref(a, sa, 0.37, b, sb, 1.9, R.EPI_BIAS)
        block = R.gemm_block_form_ref(a, sa, 0.37, b, sb, 1.9)
        np.testing.assert_allclose(dense, block, rtol=1e-12, atol=1e-12)


def test_triple_loop_brute_force():
    # element by element from the format definition, no vectorisation
    rng = np.random.default_rng(1)
    M, N, K = 2, 3, 32
    a, sa = _rand_codes(rng, M, K)
    b, sb = _rand_codes(rng, N, K)
    bias = rng.standard_normal(N)
    got = R.gemm_ref(a, sa, 0.5, b, sb, 0.25, R.EPI_BIAS, bias=bias)
    grid = [0, .5, 1, 1.5, 2, 3, 4, 6]

    def e2m1(c):
        c = int(c)
        return (-1 if c & 8 else 1) * grid[c & 7]

    def e4m3(c):
        c = int(c)
        e, m = (c >> 3) & 15, c & 7
        return (m / 8) * 2 ** -6 if e == 0 else (1 + m / 8) * 2 ** (e - 7)

    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += (e2m1(a[m, k]) * e4m3(sa[m, k // 16]) * 0.5) * \
                       (e2m1(b[n, k]) * e4m3(sb[n, k // 16]) * 0.25)
            assert math.isclose(got[m, n], acc + bias[n], rel_tol=1e-12, abs_tol=1e-12)


def test_transposed_operand_would_fail():
    # guards the test above: swapping A and B roles changes the answer
    rng = np.random.default_rng(2)
    a, sa = _rand_codes(rng, 4, 32)
    b, sb = _rand_codes(rng, 3, 32)
    y = R.gemm_ref(a, sa, 1.0, b, sb, 1.0)
    y_t = R.gemm_ref(b, sb, 1.0, a, sa, 1.0)
    assert y.shape == (4, 3) and np.allclose(y, y_t.T)


def _load_gated_golden():
    cs, ys = [], []
    for line in open(os.path.join(GOLDEN, "gated_silu_2x4.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tag, rest = line.split(" ", 1)
        mat = np.array([[float(v) for v in row.split()] for row in rest.split(";")])
        (cs if tag == "C" else ys).append(mat)
    return list(zip(cs, ys))


def test_gated_silu_worked_examples():
    for c, y in _load_gated_golden():
        np.testing.assert_allclose(R.gated_silu_ref(c), y, rtol=2e-16, atol=1e-300)


def test_gated_gemm_on_interleaved_weights_equals_formula_on_unpermuted():
    import torch
    rng = np.random.default_rng(3)
    K, N, M = 64, 32, 5
    w = torch.from_numpy(rng.standard_normal((K, N)).astype(np.float32) * 0.1).to(torch.bfloat16).float().numpy()
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    bias = rng.standard_normal(N) * 0.1
    qa, sa, ta = R.quantize_ref(x)
    cu, su, tu = R.pack_weights_ref(w, gated_interleave=False)
    cp, sp, tp = R.pack_weights_ref(w, gated_interleave=True)
    plain = R.gemm_ref(qa, sa, ta, cu, su, tu, R.EPI_BIAS, bias=bias)
    fused = R.gemm_ref(qa, sa, ta, cp, sp, tp, R.EPI_GATED_SILU, bias=bias)
    assert fused.shape == (M, N // 2)
    assert np.array_equal(fused, R.gated_silu_ref(plain))
    # a wrong pairing (no de-interleave) gives a different answer
    wrong = R.gated_silu_ref(R.gemm_ref(qa, sa, ta, cp, sp, tp, R.EPI_BIAS, bias=bias[R.gated_permutation(N)]))
    assert not np.allclose(wrong, fused)


def test_head_rmsnorm_unit_rms_with_unit_gamma():
    rng = np.random.default_rng(4)
    z = rng.standard_normal((6, 768)) * 3
    eps = 1e-6
    y = R.head_rmsnorm_ref(z, np.ones(512), 256, 512, eps)
    heads = y[:, :512].reshape(6, 2, 256)
    ms = np.mean(z[:, :512].reshape(6, 2, 256) ** 2, axis=2)
    rms = np.sqrt(np.mean(heads ** 2, axis=2))
    np.testing.assert_allclose(rms, 1 / np.sqrt(1 + eps / ms), rtol=1e-12)
    assert np.array_equal(y[:, 512:], z[:, 512:])     # columns past norm_cols untouched
    # gamma scales linearly
    g = rng.uniform(0.5, 1.5, 512)
    y2 = R.head_rmsnorm_ref(z, g, 256, 512, eps)
    np.testing.assert_allclose(y2[:, :512], y[:, :512] * g[None, :], rtol=1e-12)


def test_head_rmsnorm_hand_head():
    z = np.array([[1.0, 2.0, 3.0, 4.0, 10.0]])
    y = R.head_rmsnorm_ref(z, np.array([1.0, 1.0, 2.0, 1.0]), 4, 4, 0.0)
    r = 1 / math.sqrt(7.5)  # mean of 1, 4, 9, 16
    np.testing.assert_allclose(y, [[1 * r, 2 * r, 6 * r, 4 * r, 10.0]], rtol=1e-15)


def test_epilogue_order_bias_before_norm():
    # bias enters before the RMSNorm: a constant bias on a zero GEMM normalises to +-1
    a = np.zeros((1, 16), np.uint8)
    sa = np.zeros((1, 1), np.uint8)
    b = np.zeros((4, 16), np.uint8)
    sb = np.zeros((4, 1), np.uint8)
    y = R.gemm_ref(a, sa, 1.0, b, sb, 1.0, R.EPI_HEAD_RMSNORM, bias=np.array([2.0, -2, 2, -2]),
                   gamma=np.ones(4), head_dim=4, norm_cols=4, eps=0.0)
    np.testing.assert_allclose(y, [[1, -1, 1, -1]])
