"""Device-side error path: a bounded wait that runs out reports NVFP4_ERR_TIMEOUT and the
CUDA context stays usable (no fault, no trap, no hang)."""
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W
from oracle import nvfp4_ref as R

from parity import assert_fp32_close, to_np_f32

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    nv.nvfp4_debug_wait_timeout(err, 2_000_000)   # 2 ms on a barrier nothing completes
    assert nv.nvfp4_get_device_error(err) == 6    # NVFP4_ERR_TIMEOUT
    assert nv.nvfp4_get_device_error(err) == 0    # read clears it
    # the context still works: a small GEMM afterwards is correct
    x = W.make_x(W.TINY_BIAS)
    w = W.make_w(W.TINY_BIAS)
    qa = nv.nvfp4_quantize(x.cuda())
    qb = nv.nvfp4_pack_weights(w.cuda())
    y = nv.nvfp4_gemm(qa, qb, "bias", out_dtype=torch.float32, device_error=err)
    assert nv.nvfp4_get_device_error(err) == 0
    ref = R.gemm_ref(*R.quantize_ref(to_np_f32(x)), *R.pack_weights_ref(to_np_f32(w)), "bias")
    assert_fp32_close(to_np_f32(y), ref, "after timeout")


def test_host_checks_raise_before_launch():
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda:0")   # K % 64 != 0
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_quantize(x)
    assert e.value.status == 2


def test_host_memory_is_refused_before_launch():
    # Pinned host memory is reachable from the GPU through unified addressing, so a kernel
    # given its address would silently read host memory; the C ABI refuses any pointer that
    # is not memory of the current device (NVFP4_ERR_ARG) before launching anything. The
    # pointers chosen are ones that kernels only ever read with plain loads.
    dev = "cuda:0"
    L = nv.lib()
    x_host = torch.zeros((128, 256), dtype=torch.bfloat16).pin_memory()
    qa = nv._alloc_nvfp4(128, 256, dev)
    ts_in = torch.ones(1, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    st = L.nvfp4_quantize(x_host.data_ptr(), 128, 256, 256, qa.codes.data_ptr(), qa.scales.data_ptr(),
                          qa.ts.data_ptr(), ts_in.data_ptr(), None, s)
    assert st == 7  # NVFP4_ERR_ARG
    # the same call with device memory runs
    x_dev = x_host.to(dev)
    assert L.nvfp4_quantize(x_dev.data_ptr(), 128, 256, 256, qa.codes.data_ptr(), qa.scales.data_ptr(),
                            qa.ts.data_ptr(), ts_in.data_ptr(), None, s) == 0
    # a GEMM whose bias lives in pinned host memory is refused too
    qb = nv.nvfp4_pack_weights(torch.zeros((256, 256), dtype=torch.bfloat16, device=dev))
    bias_host = torch.zeros(256, dtype=torch.float32).pin_memory()
    out = torch.empty((128, 256), dtype=torch.bfloat16, device=dev)
    st = L.nvfp4_gemm(qa.codes.data_ptr(), qa.scales.data_ptr(), qa.ts.data_ptr(), qb.codes.data_ptr(),
                      qb.scales.data_ptr(), qb.ts.data_ptr(), 128, 256, 256, 0, bias_host.data_ptr(), None, 256, 0,
                      1e-6, 0, out.data_ptr(), 256, None, s)
    assert st == 7
    torch.cuda.synchronize()
