"""nvfp4_quantize_noalloc: the quantizer entry point for callers that cannot allocate device
memory (a plugin interface with no scratch buffer, a fixed memory pool, a loop that must not
call cudaMalloc/cudaFree). Its scratch is a fixed array inside the library.

The GPU test compares it, through the C ABI, with nvfp4_quantize on two calls in a row,
bit for bit (the tolerance every quantizer test here uses). The second input has a smaller
amax than the first, so a scratch word left over from the first call would show up as a
wrong tensor scale. This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv

from parity import gpu_nvfp4_to_np

ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DEVICE = 1, 2, 3, 4


def test_noalloc_host_checks():
    L = nv.lib()
    fake = 1 << 20
    assert L.nvfp4_quantize_noalloc(fake, 128, 96, 96, fake, fake, fake, None) == ERR_SHAPE
    assert L.nvfp4_quantize_noalloc(fake, -1, 64, 64, fake, fake, fake, None) == ERR_SHAPE
    assert L.nvfp4_quantize_noalloc(fake, 128, 64, 32, fake, fake, fake, None) == ERR_SHAPE  # ldx < K
    assert L.nvfp4_quantize_noalloc(None, 128, 64, 64, fake, fake, fake, None) == ERR_NULL
    assert L.nvfp4_quantize_noalloc(None, 0, 64, 64, None, None, None, None) == 0


def test_noalloc_checks_run_before_the_scratch_is_touched():
    # Every check of nvfp4_quantize runs before the scratch lookup and its zeroing: a refused
    # call reports its own status (on a machine without a GPU, the scratch lookup would fail
    # first and report a device or launch error instead).
    L = nv.lib()
    fake = 1 << 20
    assert L.nvfp4_quantize_noalloc(fake + 8, 128, 64, 64, fake, fake, fake, None) == ERR_ALIGN
    assert L.nvfp4_quantize_noalloc(fake, 128, 64, 68, fake, fake, fake, None) == ERR_ALIGN  # ldx % 8
    assert L.nvfp4_quantize_noalloc(fake, 128, 64, 64, fake + 4, fake, fake, None) == ERR_ALIGN
    assert L.nvfp4_quantize_noalloc(fake, 128, 64, 64, fake, fake, fake + 2, None) == ERR_ALIGN
    assert L.nvfp4_quantize_noalloc(fake, 1 << 22, 1 << 13, 1 << 13, fake, fake, fake, None) == ERR_SHAPE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_noalloc_without_a_gpu_reports_the_device():
    fake = 1 << 20
    assert nv.lib().nvfp4_quantize_noalloc(fake, 128, 64, 64, fake, fake, fake, None) == ERR_DEVICE


@pytest.mark.gpu
def test_noalloc_matches_workspace_quantizer_on_two_calls():
    rng = np.random.default_rng(1234)
    x1 = torch.from_numpy((rng.standard_normal((300, 3072)) * 10.0).astype(np.float32))
    x2 = torch.from_numpy(rng.standard_normal((300, 3072)).astype(np.float32))
    xs = [x1.to(torch.bfloat16).cuda(), x2.to(torch.bfloat16).cuda()]
    ts_seen = []
    for x in xs:
        got = gpu_nvfp4_to_np(nv.nvfp4_quantize_noalloc(x))
        want = gpu_nvfp4_to_np(nv.nvfp4_quantize(x))
        assert np.float32(got[2]).view(np.uint32) == np.float32(want[2]).view(np.uint32)
        assert np.array_equal(got[1], want[1]), "scales differ"
        assert np.array_equal(got[0], want[0]), "codes differ"
        ts_seen.append(got[2])
    assert ts_seen[1] < ts_seen[0]  # the second call did not reuse the first call's amax


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(4608, 12288), (300, 106496)])
def test_noalloc_large_inputs_match_on_two_calls(shape):
    # 4608 x 12288 is too large for the SMs' shared memory: the single cooperative launch keeps
    # a quarter of its rows there and reads the rest twice. A row of 106,496 elements (208 KB)
    # does not fit at all: the amax pass and the quantize pass run as two kernels. Both use the
    # library's scratch words.
    rng = np.random.default_rng(4321)
    x1 = torch.from_numpy((rng.standard_t(3, size=shape) * 4.0).astype(np.float32)).to(torch.bfloat16).cuda()
    x2 = torch.from_numpy((rng.standard_t(3, size=shape) * 0.5).astype(np.float32)).to(torch.bfloat16).cuda()
    ts_seen = []
    for x in (x1, x2):
        got = nv.nvfp4_quantize_noalloc(x)
        want = nv.nvfp4_quantize(x)
        torch.cuda.synchronize()
        assert torch.equal(got.ts.view(torch.int32), want.ts.view(torch.int32))
        assert torch.equal(got.scales, want.scales), "scales differ"
        assert torch.equal(got.codes, want.codes), "codes differ"
        ts_seen.append(float(got.ts.item()))
    assert ts_seen[1] < ts_seen[0]
