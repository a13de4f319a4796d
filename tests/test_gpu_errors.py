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
