"""The index-checking build of the library (libnvfp4_debug.so, compiled with -DNVFP4_DEBUG) on
ragged and strided shapes: every quantizer, packer and GEMM call (bf16, fp32 and NVFP4 outputs,
the three epilogues, the FP8 variant) gives the release library's bytes, and no index check
fails. The checks stand in for a memory checker, which this GPU pool does not offer."""
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from nvfp4_gemm_act_b300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).to(DEV)


def _run_all():
    """Every instrumented call on ragged shapes; returns the outputs, in a fixed order."""
    outs = []
    # activation quantizer: single pass with all rows in shared memory, single pass with part
    # of them there (dynamic), two passes (dynamic), static with a row stride
    x1 = _bf16((200, 320), 1)
    outs += list(nv.nvfp4_quantize(x1)[:3])
    x2 = _bf16((2000, 8192), 2, 3.0)  # 12 of each CTA's 14 rows kept in shared memory
    outs += list(nv.nvfp4_quantize(x2)[:3])
    x4 = _bf16((70, 106496), 5)  # a row larger than the shared-memory budget: two passes
    outs += list(nv.nvfp4_quantize(x4)[:3])
    x3 = _bf16((200, 328), 3)[:, :320]
    outs += list(nv.nvfp4_quantize(x3, tensor_scale_in=torch.tensor([0.01], device=DEV))[:3])
    # weight packer, plain and gated; GEMMs with every epilogue and output format
    w = _bf16((320, 224), 4, 0.02)
    qa = nv.nvfp4_quantize(x1)
    bias = _bf16((224,), 6, 0.01).float()
    gamma = 1.0 + _bf16((192,), 7, 0.1).float()
    for gated, epi, kw in ((False, "bias", dict(bias=bias)),
                           (False, "head_rmsnorm", dict(gamma=gamma, head_dim=32, norm_cols=192, bias=bias)),
                           (True, "gated_silu", {})):
        qb = nv.nvfp4_pack_weights(w, gated_interleave=gated)
        outs += list(qb[:3])
        for od in (torch.bfloat16, torch.float32):
            outs.append(nv.nvfp4_gemm(qa, qb, epi, out_dtype=od, **kw))
    w2 = _bf16((320, 256), 5, 0.02)
    # NVFP4 outputs for 200 rows (two 128-row blocks) and 300 rows (three: the last row pair's
    # second CTA lies wholly past the padded rows and must store nothing)
    qa3 = nv.nvfp4_quantize(_bf16((300, 320), 8))
    for gated, epi in ((False, "bias"), (True, "gated_silu")):
        qb = nv.nvfp4_pack_weights(w2, gated_interleave=gated)
        for a_op in (qa, qa3):
            q = nv.nvfp4_gemm_nvfp4_out(a_op, qb, epi, torch.tensor([0.002], device=DEV))
            outs += [q.codes, q.scales]
    # a bf16 GEMM over the same three row blocks
    outs.append(nv.nvfp4_gemm(qa3, nv.nvfp4_pack_weights(w, gated_interleave=False), "bias", bias=bias))
    # FP8 variant
    fa = nv.fp8_quantize(x1)
    fb = nv.fp8_pack_weights(w, gated_interleave=True)
    outs += [fa.codes, fa.ts, fb.codes, nv.fp8_gemm(fa, fb, "gated_silu")]
    torch.cuda.synchronize()
    return outs


def test_debug_build_matches_release_and_no_check_fails(monkeypatch):
    release = _run_all()
    dbg = nv.load_library(nv.DEBUG_LIB_PATH)
    assert dbg.nvfp4_debug_build() == 1 and nv.lib().nvfp4_debug_build() == 0
    monkeypatch.setattr(nv, "_lib", dbg)
    import ctypes
    n = ctypes.c_int64(-1)
    assert dbg.nvfp4_debug_index_failures(ctypes.addressof(n)) == 0  # clears anything earlier
    debug = _run_all()
    assert dbg.nvfp4_debug_index_failures(ctypes.addressof(n)) == 0
    assert n.value == 0, f"{n.value} index checks failed"
    assert len(release) == len(debug)
    for i, (a, b) in enumerate(zip(release, debug)):
        assert torch.equal(a, b), f"output {i} differs between the debug and release builds"
