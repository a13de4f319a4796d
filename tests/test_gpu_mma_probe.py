"""The tensor-core instruction-rate probe (nvfp4_debug_mma_rate): host-side argument checks
(no GPU needed) and, on the GPU, every kind and CTA-group form returning a plausible rate."""
import ctypes
import os

import pytest
import torch

import nvfp4_gemm_act_b300 as nv

pytestmark_lib = pytest.mark.skipif(not os.path.exists(nv.LIB_PATH), reason="libnvfp4.so not built")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_ARG = 0, 1, 2, 3, 7
FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every call below fails a host check


def _rate(kind, cta_group, n, iters, ctas, out=FAKE):
    L = nv.lib()
    return L.nvfp4_debug_mma_rate(ctypes.c_int(kind), ctypes.c_int(cta_group), ctypes.c_int(n),
                                  ctypes.c_int64(iters), ctypes.c_int(ctas), ctypes.c_void_p(out),
                                  ctypes.c_void_p(None), ctypes.c_void_p(None))


@pytestmark_lib
def test_probe_rejects_bad_arguments_on_the_host():
    assert _rate(3, 2, 256, 100, 1) == ERR_ARG            # no such kind
    assert _rate(-1, 2, 256, 100, 1) == ERR_ARG
    assert _rate(0, 3, 256, 100, 1) == ERR_ARG            # cta_group 1 or 2 only
    assert _rate(0, 2, 96, 100, 1) == ERR_SHAPE           # N from {64, 128, 192, 256}
    assert _rate(0, 2, 512, 100, 1) == ERR_SHAPE
    assert _rate(0, 2, 256, 0, 1) == ERR_ARG              # at least one instruction
    assert _rate(0, 2, 256, 4000001, 1) == ERR_ARG        # bounded run length
    assert _rate(0, 2, 256, 100, 1, out=0) == ERR_NULL
    assert _rate(0, 2, 256, 100, 1, out=FAKE + 4) == ERR_ALIGN


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["nvfp4", "fp8", "bf16"])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_probe_reports_a_plausible_rate(kind, cta_group):
    iters, ctas = 2000, 4
    r = nv.nvfp4_debug_mma_rate(kind, cta_group, 256, iters, ctas)
    torch.cuda.synchronize()
    r = r.cpu()
    assert r.shape == (ctas, 2)
    assert bool((r > 0).all()), r  # every CTA (pair) finished within the time limit
    cycles = r[:, 0].double() / iters
    # one N=256 instruction takes on the order of a hundred SM cycles on this part; anything
    # far outside means the loop did not run back to back or the clock read is wrong
    assert bool(((cycles > 32) & (cycles < 1024)).all()), cycles
    ghz = r[:, 0].double() / r[:, 1].double()
    assert bool(((ghz > 0.3) & (ghz < 3.5)).all()), ghz
