"""Pins for the oracle's element formats and encoders (CPU only).

E2M1 and E4M3 are checked against their bit-field definitions, hand-listed values and
ties, and against an independent implementation (ml_dtypes) over dense sweeps.
"""
import numpy as np
import pytest

from oracle import nvfp4_ref as R


def test_e2m1_grid_is_the_eight_magnitudes():
    # positive codes 0..7 decode to {0, .5, 1, 1.5, 2, 3, 4, 6}; codes 8..15 are their negatives
    pos = R.e2m1_decode(np.arange(8))
    assert pos.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    neg = R.e2m1_decode(np.arange(8, 16))
    assert (neg == -pos).all()
    # both zeros decode to zero, the negative one with its sign bit
    assert R.e2m1_decode(0) == 0 and R.e2m1_decode(8) == 0
    assert not np.signbit(R.e2m1_decode(0)) and np.signbit(R.e2m1_decode(8))


def test_e4m3_hand_values():
    dec = lambda c: float(R.e4m3_decode(c))
    assert dec(0x38) == 1.0
    assert dec(0x40) == 2.0
    assert dec(0x7E) == 448.0          # largest finite
    assert dec(0x08) == 2.0 ** -6      # smallest normal
    assert dec(0x01) == 2.0 ** -9      # smallest subnormal
    assert dec(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert dec(0x35) == 0.8125
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0xB8) == -1.0


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),  # ties -> even
    (7.0, 7), (100.0, 7),                                                    # saturation
    (0.2, 0), (0.3, 1), (2.49, 4), (2.51, 5), (4.99, 6), (5.01, 7),
    (-0.1, 8), (-0.25, 8), (-0.0, 8), (0.0, 0), (-6.0, 15), (-5.0, 14),
])
def test_e2m1_encode_hand(v, code):
    assert int(R.e2m1_encode(np.float32(v))) == code


@pytest.mark.parametrize("v,code", [
    (1.0, 0x38), (448.0, 0x7E), (460.0, 0x7E), (1e6, 0x7E),   # saturate at 448
    (2.0 ** -10, 0x00),            # exact tie between 0 and 2^-9 -> even code 0
    (1.5 * 2.0 ** -10, 0x01), (3 * 2.0 ** -10, 0x02),          # 1.5 * 2^-9 tie -> code 2
    (5.0 / 6.0, 0x35), (0.0, 0x00),
    (1.0625, 0x38), (1.1875, 0x3A),  # 1 + 1/16 tie -> even (1.0); 1 + 3/16 tie -> 1.25
])
def test_e4m3_encode_hand(v, code):
    assert int(R.e4m3_encode_nonneg(np.float32(v))) == code


def test_e2m1_matches_ml_dtypes_dense_sweep():
    ml = pytest.importorskip("ml_dtypes")
    # every multiple of 1/64 in [-8, 8] (hits all ties), plus random fp32 values
    v = np.concatenate([np.arange(-512, 513) / 64.0,
                        np.random.default_rng(0).uniform(-7, 7, 20000)]).astype(np.float32)
    ours = R.e2m1_decode(R.e2m1_encode(v))
    theirs = v.astype(ml.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(ours, theirs)
    # sign of zero results agrees too
    assert np.array_equal(np.signbit(ours), np.signbit(theirs))


def test_e4m3_matches_ml_dtypes_in_range():
    ml = pytest.importorskip("ml_dtypes")
    # ml_dtypes turns values above 464 into NaN instead of saturating, so sweep [0, 464]
    grid = R.e4m3_decode(np.arange(0x7F))
    mids = (grid[1:] + grid[:-1]) / 2          # every tie point
    v = np.concatenate([grid, mids, np.random.default_rng(1).uniform(0, 464, 20000),
                        np.exp(np.random.default_rng(2).uniform(-14, 6, 20000))]).astype(np.float32)
    v = v[v <= 464]
    ours = R.e4m3_decode(R.e4m3_encode_nonneg(v))
    theirs = v.astype(ml.float8_e4m3fn).astype(np.float64)
    assert np.array_equal(ours, theirs)


def test_nearest_code_brute_force_agrees_with_pure_python():
    # a separate, loop-only statement of "nearest, ties to even code"
    grid = R.e2m1_decode(np.arange(8))

    def slow(m):
        best, bestd = None, None
        for c in range(8):
            d = abs(m - grid[c])
            if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
                best, bestd = c, d
        return best

    vals = np.arange(0, 7.5, 0.0625)
    assert [slow(m) for m in vals] == R.e2m1_encode(vals.astype(np.float32)).tolist()


def test_round_to_bf16_hand():
    one = 1.0
    cases = {
        one + 2 ** -8: 1.0,                       # tie -> even (1.0)
        one + 3 * 2 ** -8: one + 2 ** -6,         # tie between odd 1+2^-7 and even 1+2^-6
        one + 2 ** -8 + 2 ** -30: one + 2 ** -7,  # just above the tie
        -(one + 2 ** -8 + 2 ** -30): -(one + 2 ** -7),
        3.0: 3.0, 0.0: 0.0,
        2.0 ** -130: 2.0 ** -130,                 # subnormal bf16 (quantum 2^-133)
    }
    for x, y in cases.items():
        assert R.round_to_bf16(np.array([x]))[0] == y, x


def test_round_to_bf16_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    v = np.random.default_rng(3).standard_normal(50000).astype(np.float32) * 10
    # signed zeros and values that round to a signed zero or the smallest subnormals
    v = np.concatenate([v, np.array([0.0, -0.0, 1e-45, -1e-45, 2e-41, -2e-41, 1e-40, -1e-40], np.float32)])
    ours = R.round_to_bf16(v.astype(np.float64))
    theirs = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, theirs)
    assert np.array_equal(np.signbit(ours), np.signbit(theirs))  # the sign of zero too


def test_round_to_bf16_keeps_the_sign_of_zero():
    # IEEE round to nearest: -0 stays -0 (the quantizer codes it 0x8, +0 as 0x0)
    out = R.round_to_bf16(np.array([-0.0, 0.0]))
    assert list(np.signbit(out)) == [True, False] and np.all(out == 0.0)
