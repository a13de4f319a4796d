"""Pins for the oracle's quantizer, scale layout and weight packing (CPU only)."""
import os

import numpy as np
import pytest

from oracle import nvfp4_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_quant_golden():
    rows = {}
    ts = None
    for line in open(os.path.join(GOLDEN, "quantize_2x128.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tag, *rest = line.split()
        if tag == "ts":
            ts = float(rest[0])
            continue
        r = int(rest[0])
        d = rows.setdefault(r, {})
        if tag == "x":
            d["x"] = np.array([float(v) for v in rest[1:]], np.float32)
        elif tag == "s":
            d["s"] = np.array([int(v, 16) for v in rest[1:]], np.uint8)
        elif tag == "q":
            d["q"] = np.array([int(c, 16) for c in "".join(rest[1:])], np.uint8)
    x = np.stack([rows[r]["x"] for r in sorted(rows)])
    s = np.stack([rows[r]["s"] for r in sorted(rows)])
    q = np.stack([rows[r]["q"] for r in sorted(rows)])
    assert x.shape == (2, 128) and q.shape == (2, 128) and s.shape == (2, 8)
    return x, s, q, ts


def test_quantize_hand_worked_fixture():
    x, s, q, ts = _load_quant_golden()
    codes, scales, ts_got = R.quantize_ref(x)
    assert ts_got == np.float32(ts)
    assert np.array_equal(scales, s)
    assert np.array_equal(codes, q)


def _rand_x(M, K, seed=0, scale=1.0):
    import torch
    v = np.random.default_rng(seed).standard_normal((M, K)) * scale
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).float().numpy()


def test_quantize_error_bound_and_amax_code():
    x = _rand_x(64, 256, seed=1)
    x[3, 17] = 9.5  # a clear tensor amax
    codes, scales, ts = R.quantize_ref(x)
    assert ts == np.float32(np.float32(9.5) / np.float32(2688))
    dec_s = np.repeat(R.e4m3_decode(scales), 16, axis=1)
    v = x / (dec_s * float(ts))                    # the exact scaled value
    qd = R.e2m1_decode(codes)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    # half the local grid spacing at |v|; beyond 6 the error is the saturation |v| - 6
    idx = np.clip(np.searchsorted(grid, np.abs(v)), 1, 7)
    half_step = (grid[idx] - grid[idx - 1]) / 2
    bound = np.where(np.abs(v) > 6, np.abs(v) - 6, half_step) + 1e-5
    assert (np.abs(v - qd) <= bound).all()
    # E4M3 rounding of the block scale is at most 2^-4 relative, so |v| <= 6 * (1 + 2^-4)
    assert np.abs(v).max() <= 6 * (1 + 2 ** -4) + 1e-6
    # the tensor's amax element lands on the largest code with scale 448
    assert scales[3, 1] == 0x7E and codes[3, 17] == 0x7


def test_quantize_on_grid_round_trip_is_exact():
    # values that already sit on the grid of a block with scale 1 and ts 1 come back unchanged
    rng = np.random.default_rng(2)
    q = rng.integers(0, 16, size=(8, 64)).astype(np.uint8)
    q[:, ::16] = 7                                       # each block's amax is 6 -> scale 1
    q[q == 8] = 0                                        # no negative zeros in the source
    x = R.e2m1_decode(q).astype(np.float32)
    x[0, 0] = 6.0
    ts = np.float32(1.0)
    codes, scales, _ = R.quantize_ref(x, tensor_scale=ts)
    assert (scales == 0x38).all()
    assert np.array_equal(codes, q)


def test_quantize_zero_tensor_and_zero_blocks():
    x = np.zeros((3, 64), np.float32)
    codes, scales, ts = R.quantize_ref(x)
    assert ts == 0 and not codes.any() and not scales.any()
    x[1, 20] = -3.0
    codes, scales, ts = R.quantize_ref(x)
    assert scales[1, 1] != 0 and codes[1, 20] == 0xF
    assert not np.delete(scales.reshape(-1), 1 * 4 + 1).any()


def test_static_tensor_scale_saturates():
    # a static scale far below amax/2688 saturates the block scale at 448 and codes at 6
    x = np.full((1, 16), 100.0, np.float32)
    codes, scales, ts = R.quantize_ref(x, tensor_scale=np.float32(1e-3))
    assert ts == np.float32(1e-3) and scales[0, 0] == 0x7E and (codes == 7).all()


def test_scale_layout_is_a_bijection_and_hand_offsets():
    K = 256
    assert R.scale_offset(0, 0, K) == 0
    assert R.scale_offset(1, 0, K) == 16
    assert R.scale_offset(32, 0, K) == 4
    assert R.scale_offset(0, 1, K) == 1
    assert R.scale_offset(0, 4, K) == 512          # next K tile of the same 128 rows
    assert R.scale_offset(128, 0, K) == 4 * 512    # next 128-row band after K/64 = 4 tiles
    rows = 256
    r, kb = np.meshgrid(np.arange(rows), np.arange(K // 16), indexing="ij")
    off = R.scale_offset(r, kb, K).reshape(-1)
    assert np.array_equal(np.sort(off), np.arange(R.scales_bytes(rows, K)))
    s = np.random.default_rng(4).integers(0, 127, (200, K // 16)).astype(np.uint8)
    buf = R.tile_scales(s, K)
    assert buf.size == R.scales_bytes(200, K) == 2 * 4 * 512
    assert np.array_equal(R.untile_scales(buf, 200, K), s)
    # padding rows 200..255 are zero
    pad = np.ones(buf.size, bool)
    r, kb = np.meshgrid(np.arange(200), np.arange(K // 16), indexing="ij")
    pad[R.scale_offset(r, kb, K).reshape(-1)] = False
    assert not buf[pad].any()


def test_nibble_packing_low_nibble_first():
    c = np.array([[1, 2, 3, 4, 15, 0]], np.uint8)
    p = R.pack_nibbles(c)
    assert p.tolist() == [[0x21, 0x43, 0x0F]]
    assert np.array_equal(R.unpack_nibbles(p), c)


def test_interleave_round_trip_and_packing_commutes():
    w = _rand_x(64, 48, seed=5, scale=0.02)              # W [K=64, N=48]
    assert np.array_equal(R.deinterleave_columns(R.interleave_columns(w)), w)
    perm = R.gated_permutation(48)
    assert perm[:6].tolist() == [0, 24, 1, 25, 2, 26]
    cu, su, tu = R.pack_weights_ref(w, gated_interleave=False)
    cp, sp, tp = R.pack_weights_ref(w, gated_interleave=True)
    # quantization is row-wise with a permutation-invariant tensor scale
    assert tu == tp
    assert np.array_equal(cp, cu[perm]) and np.array_equal(sp, su[perm])
    # packed rows are the K-major transpose
    assert cu.shape == (48, 64)
