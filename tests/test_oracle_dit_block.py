"""Pins for the oracle's attention and its chained DiT block (CPU only).

Attention is pinned by cases whose answer is fixed by the definition alone: one key, a zero
query, one key far ahead of the rest, two keys (a logistic in the score difference, which
fixes the 1/sqrt(d) scale and the axis of the softmax), permutations and head independence.
The chain is pinned by weights that make a stage's output known in closed form (a zero V or
Q projection), which fixes the Q | K | V column order and the head layout, and by its
equivariance under a permutation of the tokens.
"""
import numpy as np
import pytest

from oracle import nvfp4_ref as R

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _qkv(heads, m_q, m_k, d, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((heads, m_q, d)), g.standard_normal((heads, m_k, d)),
            g.standard_normal((heads, m_k, d)))


def test_attention_single_key_returns_its_value():
    q, k, v = _qkv(2, 5, 1, 8, 0)
    out = R.attention_ref(q, k, v)
    assert np.array_equal(out, np.broadcast_to(v, out.shape))


def test_attention_zero_query_averages_values():
    q, k, v = _qkv(3, 4, 7, 16, 1)
    out = R.attention_ref(np.zeros_like(q), k, v)
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape), rtol=0, atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    # keys c * e_j (one-hot), query 1000 * e_j * sqrt(d) / c: score of key j = 1000, others 0
    heads, d, m = 1, 16, 6
    c = 3.0
    k = c * np.eye(d)[None, :m]
    v = np.random.default_rng(2).standard_normal((heads, m, 5))
    for j in range(m):
        q = (1000.0 * np.sqrt(d) / c) * np.eye(d)[None, j:j + 1]
        out = R.attention_ref(q, k, v)
        assert np.array_equal(out[0, 0], v[0, j])


def test_attention_two_keys_logistic_and_scale():
    # scores s1, s2 -> weight of key 1 = 1 / (1 + exp(s2 - s1)); scores carry 1/sqrt(d)
    d = 64
    q = np.zeros((1, 2, d))
    q[0, 0, 0] = 2.0
    q[0, 1, 1] = -1.0       # a second query with different scores: softmax runs over keys
    k = np.zeros((1, 2, d))
    k[0, 0, 0] = 4.0        # q0.k1 = 8 -> score 1;   q1.k1 = 0
    k[0, 1, 1] = 12.0       # q0.k2 = 0;              q1.k2 = -12 -> score -1.5
    v = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    out = R.attention_ref(q, k, v)
    w0 = 1.0 / (1.0 + np.exp(0.0 - 1.0))
    w1 = 1.0 / (1.0 + np.exp(-1.5 - 0.0))
    np.testing.assert_allclose(out[0], [[w0, 1 - w0], [w1, 1 - w1]], rtol=1e-15, atol=1e-16)


def test_attention_permutations_and_head_independence():
    q, k, v = _qkv(3, 6, 9, 8, 3)
    out = R.attention_ref(q, k, v)
    pk = np.random.default_rng(4).permutation(9)
    np.testing.assert_allclose(R.attention_ref(q, k[:, pk], v[:, pk]), out, rtol=1e-13, atol=1e-14)
    pq = np.random.default_rng(5).permutation(6)
    np.testing.assert_allclose(R.attention_ref(q[:, pq], k, v), out[:, pq], rtol=1e-13, atol=1e-14)
    v2 = v.copy()
    v2[1] += 5.0
    out2 = R.attention_ref(q, k, v2)
    assert np.array_equal(out2[[0, 2]], out[[0, 2]])
    np.testing.assert_allclose(out2[1], out[1] + 5.0, rtol=0, atol=1e-12)


# ---- the chained block, on a tiny one: 2 heads of 16, hidden 32, MLP 48, 12 tokens ----------

HEADS, HD, MLP, M = 2, 16, 48, 12
H = HEADS * HD


def _bf16(a):
    return R.round_to_bf16(a).astype(np.float32)


def _block(seed=7):
    g = np.random.default_rng(seed)
    x = _bf16(g.standard_normal((M, H)))
    layers = [(_bf16(0.2 * g.standard_normal((H, 3 * H))), 0.05 * g.standard_normal(3 * H),
               1.0 + 0.1 * g.standard_normal(2 * H)),
              (_bf16(0.2 * g.standard_normal((H, H))), 0.05 * g.standard_normal(H), None),
              (_bf16(0.2 * g.standard_normal((H, 2 * MLP))), 0.05 * g.standard_normal(2 * MLP), None),
              (_bf16(0.2 * g.standard_normal((MLP, H))), 0.05 * g.standard_normal(H), None)]
    return x, layers


def _zero_cols(layers, lo, hi):
    (w, b, gm), *rest = layers
    w, b = w.copy(), b.copy()
    w[:, lo:hi] = 0
    b[lo:hi] = 0
    return [(w, b, gm)] + rest


def test_block_zero_value_projection_leaves_the_output_bias():
    # V = 0 (its weights and bias): attention output 0, so the output projection gives its bias
    x, layers = _block()
    _, inter = R.dit_block_ref(x, _zero_cols(layers, 2 * H, 3 * H), HEADS, HD)
    assert np.all(inter["attention"] == 0)
    assert np.array_equal(inter["out_proj"], np.broadcast_to(R.round_to_bf16(layers[1][1]), (M, H)))


def test_block_zero_query_projection_averages_the_values():
    # Q = 0: every score 0, every token's attention output = mean over tokens of V, per column
    x, layers = _block(8)
    y, inter = R.dit_block_ref(x, _zero_cols(layers, 0, H), HEADS, HD)
    v = inter["qkv"][:, 2 * H:]
    np.testing.assert_array_equal(inter["attention"], np.broadcast_to(R.round_to_bf16(v.mean(axis=0)), (M, H)))
    assert np.all(y == y[0])


def test_block_token_permutation_equivariance():
    x, layers = _block(9)
    p = np.random.default_rng(10).permutation(M)
    y, inter = R.dit_block_ref(x, layers, HEADS, HD)
    yp, _ = R.dit_block_ref(x[p], layers, HEADS, HD, ts_mid=inter["ts_mid"])
    assert np.array_equal(yp, y[p])
    ye, _ = R.dit_block_ref(x, layers, HEADS, HD, quantized=False)
    yep, _ = R.dit_block_ref(x[p], layers, HEADS, HD, quantized=False)
    np.testing.assert_allclose(yep, ye[p], rtol=1e-12, atol=1e-13)


def test_block_static_scale_and_exact_limit():
    x, layers = _block(11)
    y, inter = R.dit_block_ref(x, layers, HEADS, HD)
    u = inter["up"]
    assert inter["ts_mid"] == R.tensor_scale_ref(u)
    # the down-projection reads quant(u; ts_mid): a power-of-two change of the static scale
    # moves every block scale by the same power of two (exact in E4M3 while the scales stay
    # normal) and leaves the output unchanged; a factor of 3 re-rounds the scales
    y2, _ = R.dit_block_ref(x, layers, HEADS, HD, ts_mid=np.float32(inter["ts_mid"] * 2))
    assert np.array_equal(y2, y)
    y3, _ = R.dit_block_ref(x, layers, HEADS, HD, ts_mid=np.float32(inter["ts_mid"] * 3))
    assert not np.array_equal(y3, y)
    # the quantized block approximates the exact one (4 bits per value: a few tens of percent)
    ye, ei = R.dit_block_ref(x, layers, HEADS, HD, quantized=False)
    rel = np.sqrt(np.mean((y - ye) ** 2) / np.mean(ye ** 2))
    assert 1e-3 < rel < 0.5
    # the exact QKV stage is the plain fp64 layer: RMSNorm'd Q, K heads of unit mean square / gamma
    t = ei["qkv"]
    qk = (t[:, :2 * H] / layers[0][2][None, :]).reshape(M, 2 * HEADS, HD)
    np.testing.assert_allclose(np.mean(qk ** 2, axis=2), 1.0, rtol=1e-4)


def test_block_sampled_rows_equal_the_full_block_rows():
    # the sampled-rows form computes the same numbers for those tokens as the full block
    x, layers = _block(12)
    rows = np.array([0, 3, 7, 11])
    y, inter = R.dit_block_ref(x, layers, HEADS, HD)
    ys, _ = R.dit_block_ref(x, layers, HEADS, HD, ts_mid=inter["ts_mid"], rows=rows)
    assert np.array_equal(ys, y[rows])
    ye, _ = R.dit_block_ref(x, layers, HEADS, HD, quantized=False)
    yes, _ = R.dit_block_ref(x, layers, HEADS, HD, quantized=False, rows=rows)
    np.testing.assert_allclose(yes, ye[rows], rtol=1e-12, atol=1e-13)
