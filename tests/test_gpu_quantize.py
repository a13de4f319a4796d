"""GPU parity of the quantizer and the weight packer against the oracle: bit-exact codes,
scales and tensor scales (calls go through the C ABI)."""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import assert_quant_equal, gpu_nvfp4_to_np, to_np_f32
from test_oracle_quantize import _load_quant_golden

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def quant_both(x_bf16: torch.Tensor, ts_in=None, what=""):
    tsi = None if ts_in is None else torch.tensor([ts_in], dtype=torch.float32, device=DEV)
    q = nv.nvfp4_quantize(x_bf16.to(DEV), tensor_scale_in=tsi)
    gpu = gpu_nvfp4_to_np(q)
    ref = R.quantize_ref(to_np_f32(x_bf16), ts_in)
    assert_quant_equal(gpu, ref, what)
    return q


def test_hand_worked_fixture_on_gpu():
    x, s, qc, ts = _load_quant_golden()
    q = nv.nvfp4_quantize(_bf16(x).to(DEV))
    gc, gs, gt = gpu_nvfp4_to_np(q)
    assert gt == np.float32(ts)
    assert np.array_equal(gs, s)
    assert np.array_equal(gc, qc)


def test_tiny_activations():
    quant_both(W.make_x(W.TINY_BIAS), what="tiny")


@pytest.mark.parametrize("M", [1, 127, 129, 200])
def test_ragged_rows_and_zero_padding(M):
    x = W.make_x(W.QKV_RMSNORM.with_m(M))
    q = quant_both(x, what=f"M={M}")
    buf = q.scales.cpu().numpy()
    used = np.zeros(buf.size, bool)
    r, kb = np.meshgrid(np.arange(M), np.arange(x.shape[1] // 16), indexing="ij")
    used[R.scale_offset(r, kb, x.shape[1])] = True
    assert not buf[~used].any(), "padding rows of the scale tiles must be zero"


def test_qkv_activations_full_size():
    quant_both(W.make_x(W.QKV_RMSNORM), what="qkv X 4608x3072")


def test_down_activations_full_size_sampled_rows():
    w = W.DOWN_BIAS
    x = W.make_x(w)
    q = nv.nvfp4_quantize(x.to(DEV))
    gc, gs, gt = gpu_nvfp4_to_np(q)
    xn = to_np_f32(x)
    ts = R.tensor_scale_ref(xn)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 4607],
                                     np.random.default_rng(7).integers(0, w.M, 58)]))
    rc, rs, _ = R.quantize_ref(xn[rows], ts)
    assert_quant_equal((gc[rows], gs[rows], gt), (rc, rs, ts), "down X sampled")


def test_static_tensor_scale():
    x = W.make_x(W.TINY_BIAS)
    quant_both(x, ts_in=np.float32(1e-3), what="static small ts (saturating)")
    quant_both(x, ts_in=np.float32(0.05), what="static large ts")


def test_zero_tensor_and_degenerate_values():
    quant_both(torch.zeros(64, 128, dtype=torch.bfloat16), what="zeros")
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 256))
    x[:, :16] *= 1e-30                  # blocks far below the tensor amax: E4M3 underflow
    x[1] = -0.0                          # negative zeros
    x[2, ::3] = 0.0
    x[3] *= 1e-35                        # tiny row, still live blocks
    quant_both(_bf16(x), what="degenerate")
    t = np.full((8, 64), 1e-38)          # tiny tensor: fp32 subnormal products
    t[0, 0] = 3e-38
    quant_both(_bf16(t), what="tiny tensor")


def test_strided_rows():
    x = W.make_x(W.QKV_RMSNORM.with_m(96))
    big = torch.zeros(96, 3072 + 64, dtype=torch.bfloat16)
    big[:, :3072] = x
    view = big.to(DEV)[:, :3072]
    assert view.stride(0) == 3136
    q = nv.nvfp4_quantize(view)
    assert_quant_equal(gpu_nvfp4_to_np(q), R.quantize_ref(to_np_f32(x)), "strided")


def test_empty_input_is_a_no_op():
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device=DEV)
    q = nv.nvfp4_quantize(x)
    torch.cuda.synchronize()
    assert q.codes.numel() == 0


def pack_both(w_bf16, gated, what):
    q = nv.nvfp4_pack_weights(w_bf16.to(DEV), gated_interleave=gated)
    gpu = gpu_nvfp4_to_np(q)
    ref = R.pack_weights_ref(to_np_f32(w_bf16), gated)
    assert_quant_equal(gpu, ref, what)
    return q


@pytest.mark.parametrize("gated", [False, True])
def test_pack_small(gated):
    pack_both(W.make_w(W.TINY_BIAS), gated, f"tiny W gated={gated}")


@pytest.mark.parametrize("K,N", [(64, 8), (128, 72), (320, 200)])
def test_pack_ragged(K, N):
    rng = np.random.default_rng(K + N)
    w = _bf16(rng.standard_normal((K, N)) * 0.02)
    pack_both(w, False, f"W {K}x{N}")
    if N % 2 == 0:
        pack_both(w, True, f"W {K}x{N} gated")


def test_pack_gated_up_full_size_sampled_rows():
    w = W.GATED_UP
    wt = W.make_w(w)
    q = nv.nvfp4_pack_weights(wt.to(DEV), gated_interleave=True)
    gc, gs, gt = gpu_nvfp4_to_np(q)
    wn = to_np_f32(wt)
    ts = R.tensor_scale_ref(wn)
    perm = R.gated_permutation(w.N)
    rows = np.unique(np.concatenate([[0, 1, 2, 3, w.N - 2, w.N - 1, 12287, 12288],
                                     np.random.default_rng(8).integers(0, w.N, 56)]))
    rc, rs, _ = R.quantize_ref(np.ascontiguousarray(wn.T[perm[rows]]), ts)
    assert_quant_equal((gc[rows], gs[rows], gt), (rc, rs, ts), "gated W sampled")


def test_workspace_reused_across_calls():
    # one zeroed workspace, reused: amax going down, up, down again, with a static-scale call
    # and a weight pack on the same workspace in between; every call matches the oracle
    ws = torch.zeros(nv.nvfp4_workspace_bytes(), dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(21)
    scales = [50.0, 0.5, 7.0, 1e-3, 3.0]
    for i, s in enumerate(scales):
        x = _bf16(rng.standard_normal((130, 512)) * s)
        q = nv.nvfp4_quantize(x.to(DEV), workspace=ws)
        assert_quant_equal(gpu_nvfp4_to_np(q), R.quantize_ref(to_np_f32(x)), f"call {i}")
        if i == 1:
            tsi = torch.tensor([0.01], dtype=torch.float32, device=DEV)
            q = nv.nvfp4_quantize(x.to(DEV), tensor_scale_in=tsi, workspace=ws)
            assert_quant_equal(gpu_nvfp4_to_np(q), R.quantize_ref(to_np_f32(x), np.float32(0.01)), "static")
        if i == 2:
            w = _bf16(rng.standard_normal((128, 64)) * 100.0)
            nv.nvfp4_pack_weights(w.to(DEV), workspace=ws)


def test_rows_only_16_byte_aligned():
    # x starting 16 bytes into an allocation: the kernel must use 16-byte loads
    x = W.make_x(W.QKV_RMSNORM.with_m(64))
    big = torch.zeros(64, 3072 + 8, dtype=torch.bfloat16)
    big[:, 8:] = x
    view = big.to(DEV)[:, 8:]
    assert view.data_ptr() % 32 == 16
    q = nv.nvfp4_quantize(view)
    assert_quant_equal(gpu_nvfp4_to_np(q), R.quantize_ref(to_np_f32(x)), "16-byte aligned rows")


def _boundary_blocks(k: int, rng, with_neighbours=True):
    """Rows of 16-element blocks whose |max| is an E4M3 value or a midpoint between two, times
    2^k (exact in bf16), and its bf16 neighbours: with 6 ts = 2^k the block quotient lands on
    the E4M3 rounding boundaries, where the kernels' reciprocal route must defer to the exact
    division."""
    vals = R.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64)
    targets = np.concatenate([vals, (vals[:-1] + vals[1:]) / 2]) * 2.0 ** k
    t16 = torch.from_numpy(targets.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(t16.float().numpy().astype(np.float64), targets), "targets exact in bf16"
    bits = t16.view(torch.int16).numpy().astype(np.int32)
    if with_neighbours:
        bits = np.concatenate([bits, bits + 1, np.maximum(bits - 1, 0)])
    mags = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).float().numpy()
    n = mags.size
    x = rng.uniform(-1.0, 1.0, (n, 16)) * mags[:, None] * 0.9
    x[np.arange(n), rng.integers(0, 16, n)] = mags * rng.choice([-1.0, 1.0], n)
    rows = -(-n * 16 // 256)
    flat = np.zeros(rows * 256)
    flat[: n * 16] = x.ravel()
    return flat.reshape(rows, 256)


@pytest.mark.parametrize("k", [0, -3, 5, -9])
def test_scale_rounding_boundaries_static_scale(k):
    # two-launch path; 6 * fp32(2^k / 6) rounds to exactly 2^k
    ts = np.float32(2.0 ** k / 6.0)
    assert np.float32(6.0) * ts == np.float32(2.0 ** k)
    x = _bf16(_boundary_blocks(k, np.random.default_rng(40 + k)))
    quant_both(x, ts_in=ts, what=f"E4M3 boundaries, static ts, k={k}")


@pytest.mark.parametrize("k", [0, -4, 6])
def test_scale_rounding_boundaries_dynamic_scale(k):
    # single-launch path: one element of 448 * 2^k pins amax, so ts = fp32(2^k / 6)
    xb = _boundary_blocks(k, np.random.default_rng(60 + k))
    xb = np.clip(xb, -448.0 * 2.0 ** k, 448.0 * 2.0 ** k)
    xb[0, 0] = 448.0 * 2.0 ** k
    x = _bf16(xb)
    q = quant_both(x, what=f"E4M3 boundaries, dynamic ts, k={k}")
    assert np.float32(6.0) * gpu_nvfp4_to_np(q)[2] == np.float32(2.0 ** k)


def test_large_ragged_strided_dynamic_scale():
    # X of 1300 x 12288 (32 MB: too large for the SMs' shared memory, so the single-pass
    # launch keeps 8 of each CTA's 10 rows there and reads the other 2 again after the grid
    # barrier); ragged M (108 padding rows of scale tiles, which must come out zero from an
    # uninitialised buffer) and a row pitch of 12352 elements
    w = W.DOWN_BIAS.with_m(1300, seed=91)
    x = W.make_x(w)
    big = torch.zeros(1300, 12288 + 64, dtype=torch.bfloat16)
    big[:, :12288] = x
    view = big.to(DEV)[:, :12288]
    q = nv.nvfp4_quantize(view)
    gc, gs, gt = gpu_nvfp4_to_np(q)
    xn = to_np_f32(x)
    ts = R.tensor_scale_ref(xn)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 1279, 1280, 1299],
                                     np.random.default_rng(92).integers(0, 1300, 25)]))
    rc, rs, _ = R.quantize_ref(xn[rows], ts)
    assert_quant_equal((gc[rows], gs[rows], gt), (rc, rs, ts), "large ragged strided")
    buf = q.scales.cpu().numpy()
    used = np.zeros(buf.size, bool)
    r, kb = np.meshgrid(np.arange(1300), np.arange(12288 // 16), indexing="ij")
    used[R.scale_offset(r, kb, 12288)] = True
    assert not buf[~used].any(), "padding rows of the scale tiles must be zero"


def test_dynamic_scale_rows_larger_than_shared_memory():
    # a row of 106,496 elements (208 KB) does not fit the single-pass kernel's shared memory at
    # all: the amax pass and the quantize pass run as two launches; ragged M
    K = 106496
    x = _bf16(np.random.default_rng(94).standard_normal((70, K)) * 0.5)
    q = nv.nvfp4_quantize(x.to(DEV))
    assert_quant_equal(gpu_nvfp4_to_np(q), R.quantize_ref(to_np_f32(x)), "two-pass dynamic")


@pytest.mark.parametrize("M,K", [(4608, 6144), (2000, 12288), (150, 24576)])
def test_dynamic_scale_partly_resident_rows(M, K):
    # single-pass launches where only some of each CTA's rows stay in shared memory (X
    # [4608, 6144]: 16 of 32; [2000, 12288]: 8 of 14; [150, 24576]: both of 2): the resident
    # rows and the re-read rows quantize alike, bit for bit, on sampled rows
    x = _bf16(0.5 * np.random.default_rng(95 + M).standard_t(3, (M, K)))
    q = nv.nvfp4_quantize(x.to(DEV))
    gc, gs, gt = gpu_nvfp4_to_np(q)
    xn = to_np_f32(x)
    ts = R.tensor_scale_ref(xn)
    rows = np.unique(np.concatenate([[0, 1, 7, 8, 9, 13, 14, 15, 16, 31, 32, M - 1],
                                     np.random.default_rng(96).integers(0, M, 40)]))
    rows = rows[rows < M]
    rc, rs, _ = R.quantize_ref(xn[rows], ts)
    assert_quant_equal((gc[rows], gs[rows], gt), (rc, rs, ts), f"partly resident {M}x{K}")
