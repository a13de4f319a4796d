"""C-ABI checks that need no GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import nvfp4_gemm_act_b300 as nv
from oracle import nvfp4_ref as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")

pytestmark = pytest.mark.skipif(not os.path.exists(nv.LIB_PATH), reason="libnvfp4.so not built")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DEVICE, ERR_ARG = 0, 1, 2, 3, 4, 7
FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every call below fails a host check


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def test_header_symbols_are_exported():
    names = header_functions()
    assert {"nvfp4_quantize", "nvfp4_pack_weights", "nvfp4_gemm"} <= set(names)
    L = ctypes.CDLL(nv.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    # and every exported entry point has a Python binding with the same name
    for n in names:
        assert n in nv._SIGS, n


def test_only_header_symbols_are_exported():
    out = os.popen(f"nm -D --defined-only {nv.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("nvfp4")}
    assert ours == set(header_functions())


def test_status_strings():
    for code, name in nv.STATUS.items():
        assert nv.lib().nvfp4_status_string(code).decode() == name
    assert nv.lib().nvfp4_status_string(99).decode() == "NVFP4_ERR_UNKNOWN"


def test_scale_helpers_match_the_oracle_layout():
    for rows, K in [(1, 64), (128, 256), (200, 3072), (4608, 12288)]:
        assert nv.nvfp4_scales_bytes(rows, K) == R.scales_bytes(rows, K)
    rng = np.random.default_rng(0)
    for _ in range(200):
        K = int(rng.integers(1, 200)) * 64
        r, kb = int(rng.integers(0, 5000)), int(rng.integers(0, K // 16))
        assert nv.nvfp4_scale_offset(r, kb, K) == int(R.scale_offset(r, kb, K))
    assert nv.nvfp4_scale_offset(0, 4, 64) == -1 and nv.nvfp4_scale_offset(-1, 0, 64) == -1
    assert nv.nvfp4_scales_bytes(0, 64) == 0 and nv.nvfp4_scales_bytes(4, 96) == 0
    assert nv.nvfp4_workspace_bytes() == 16


def q(x=FAKE, M=128, K=256, ldx=256, codes=FAKE, scales=FAKE, ts=FAKE, ts_in=None, ws=FAKE):
    return nv.lib().nvfp4_quantize(x, M, K, ldx, codes, scales, ts, ts_in, ws, None)


def test_quantize_host_checks():
    assert q(x=None) == ERR_NULL
    assert q(codes=None) == ERR_NULL
    assert q(ws=None) == ERR_NULL                  # dynamic scale needs the workspace
    assert q(K=96, ldx=96) == ERR_SHAPE            # K % 64
    assert q(K=0, ldx=0) == ERR_SHAPE
    assert q(M=-1) == ERR_SHAPE
    assert q(ldx=128) == ERR_SHAPE                 # ldx < K
    assert q(M=1 << 22, K=1 << 13, ldx=1 << 13) == ERR_SHAPE  # beyond 2^34 elements
    assert q(x=FAKE + 8) == ERR_ALIGN
    assert q(ldx=260) == ERR_ALIGN
    assert q(codes=FAKE + 4) == ERR_ALIGN
    assert q(M=0) == OK                            # empty: nothing launched
    assert q(M=0, x=None, codes=None) == OK        # empty tensors may have NULL storage


def g(**kw):
    a = dict(ac=FAKE, asc=FAKE, ats=FAKE, bc=FAKE, bsc=FAKE, bts=FAKE, M=128, N=256, K=256, epi=0,
             bias=None, gamma=None, hd=256, nc=0, eps=1e-6, od=0, out=FAKE, ldo=256, err=None)
    a.update(kw)
    return nv.lib().nvfp4_gemm(a["ac"], a["asc"], a["ats"], a["bc"], a["bsc"], a["bts"], a["M"], a["N"],
                               a["K"], a["epi"], a["bias"], a["gamma"], a["hd"], a["nc"], a["eps"],
                               a["od"], a["out"], a["ldo"], a["err"], None)


def test_gemm_host_checks():
    assert g(ac=None) == ERR_NULL
    assert g(out=None) == ERR_NULL
    assert g(epi=1, nc=256, gamma=None) == ERR_NULL
    assert g(epi=5) == ERR_ARG
    assert g(od=3) == ERR_ARG
    assert g(epi=1, hd=96, gamma=FAKE, nc=192) == ERR_ARG
    assert g(epi=1, gamma=FAKE, nc=256, eps=-1.0) == ERR_ARG
    assert g(K=96) == ERR_SHAPE
    assert g(N=48, ldo=48) == ERR_SHAPE            # N % 32
    assert g(epi=1, gamma=FAKE, nc=128) == ERR_SHAPE   # norm_cols % head_dim
    assert g(epi=1, gamma=FAKE, nc=512) == ERR_SHAPE   # norm_cols > N
    assert g(ldo=128) == ERR_SHAPE
    assert g(epi=2, ldo=128) != ERR_SHAPE          # gated output is N/2 wide
    assert g(ac=FAKE + 1) == ERR_ALIGN
    assert g(ldo=260) == ERR_ALIGN
    assert g(od=1, ldo=260) == ERR_SHAPE or g(od=1, ldo=260) != ERR_ALIGN
    assert g(M=0) == OK
    assert g(M=0, ac=None) == OK
    # operands larger than the quantizer / packer can produce, and more pair tiles than a
    # 32-bit index holds: refused before any device work
    assert g(M=2**31 - 1, N=256, K=64, ldo=256) == ERR_SHAPE     # M * K >= 2^34
    assert g(N=2**30, K=2**14, ldo=2**30) == ERR_SHAPE            # N * K >= 2^34
    assert g(M=2**25, N=2**25, K=64, ldo=2**25) == ERR_SHAPE      # 2^34 pair tiles
    assert g(M=2**20, N=2**20, K=64, ldo=2**20) != ERR_SHAPE      # within every bound


def gq(**kw):
    a = dict(ac=FAKE, asc=FAKE, ats=FAKE, bc=FAKE, bsc=FAKE, bts=FAKE, M=128, N=256, K=256, epi=0,
             bias=None, gamma=None, hd=256, nc=0, eps=1e-6, ots=FAKE, oc=FAKE, osc=FAKE, err=None)
    a.update(kw)
    return nv.lib().nvfp4_gemm_nvfp4_out(a["ac"], a["asc"], a["ats"], a["bc"], a["bsc"], a["bts"], a["M"],
                                         a["N"], a["K"], a["epi"], a["bias"], a["gamma"], a["hd"], a["nc"],
                                         a["eps"], a["ots"], a["oc"], a["osc"], a["err"], None)


def test_gemm_nvfp4_out_host_checks():
    assert gq(N=32) == ERR_SHAPE                   # output width % 64
    assert gq(epi=2, N=64) == ERR_SHAPE            # gated output width N/2 = 32
    assert gq(epi=2, N=128) != ERR_SHAPE
    assert gq(ots=None) == ERR_NULL
    assert gq(oc=None) == ERR_NULL
    assert gq(osc=None) == ERR_NULL
    assert gq(ac=None) == ERR_NULL
    assert gq(oc=FAKE + 8) == ERR_ALIGN
    assert gq(epi=5) == ERR_ARG
    assert gq(K=96) == ERR_SHAPE
    assert gq(M=0) == OK
    assert gq(M=0, oc=None, ots=None) == OK


def test_pack_host_checks():
    L = nv.lib()
    assert L.nvfp4_pack_weights(None, 256, 256, 0, FAKE, FAKE, FAKE, FAKE, None) == ERR_NULL
    assert L.nvfp4_pack_weights(FAKE, 256, 256, 2, FAKE, FAKE, FAKE, FAKE, None) == ERR_ARG
    assert L.nvfp4_pack_weights(FAKE, 100, 256, 0, FAKE, FAKE, FAKE, FAKE, None) == ERR_SHAPE
    assert L.nvfp4_pack_weights(FAKE, 256, 12, 0, FAKE, FAKE, FAKE, FAKE, None) == ERR_SHAPE
    assert L.nvfp4_pack_weights(FAKE + 2, 256, 256, 0, FAKE, FAKE, FAKE, FAKE, None) == ERR_ALIGN


def test_debug_timeout_host_checks():
    L = nv.lib()
    assert L.nvfp4_debug_wait_timeout(None, 1000, None) == ERR_NULL
    assert L.nvfp4_debug_wait_timeout(FAKE, 0, None) == ERR_ARG
    assert L.nvfp4_get_device_error(None, None, None) == ERR_NULL


def f8g(**kw):
    a = dict(ac=FAKE, ats=FAKE, bc=FAKE, bts=FAKE, M=128, N=256, K=256, epi=0, bias=None, gamma=None, hd=256,
             nc=0, eps=1e-6, od=0, out=FAKE, ldo=256, err=None)
    a.update(kw)
    return nv.lib().fp8_gemm(a["ac"], a["ats"], a["bc"], a["bts"], a["M"], a["N"], a["K"], a["epi"], a["bias"],
                             a["gamma"], a["hd"], a["nc"], a["eps"], a["od"], a["out"], a["ldo"], a["err"], None)


def test_fp8_gemm_host_checks():
    assert f8g(ac=None) == ERR_NULL
    assert f8g(bts=None) == ERR_NULL
    assert f8g(out=None) == ERR_NULL
    assert f8g(epi=1, nc=256, gamma=None) == ERR_NULL
    assert f8g(epi=5) == ERR_ARG
    assert f8g(od=3) == ERR_ARG
    assert f8g(K=96) == ERR_SHAPE
    assert f8g(N=48, ldo=48) == ERR_SHAPE
    assert f8g(ldo=128) == ERR_SHAPE
    assert f8g(epi=2, ldo=128) != ERR_SHAPE
    assert f8g(ac=FAKE + 1) == ERR_ALIGN
    assert f8g(bc=FAKE + 8) == ERR_ALIGN
    assert f8g(ldo=260) == ERR_ALIGN
    assert f8g(M=0) == OK
    assert f8g(M=0, ac=None, out=None) == OK


def test_fp8_quantize_and_pack_host_checks():
    L = nv.lib()
    assert L.fp8_quantize(FAKE, 128, 96, 96, FAKE, FAKE, None, FAKE, None) == ERR_SHAPE    # K % 64
    assert L.fp8_quantize(FAKE, 128, 128, 64, FAKE, FAKE, None, FAKE, None) == ERR_SHAPE   # ldx < K
    assert L.fp8_quantize(FAKE, -1, 128, 128, FAKE, FAKE, None, FAKE, None) == ERR_SHAPE
    assert L.fp8_quantize(FAKE, 0, 128, 128, None, None, None, None, None) == OK
    assert L.fp8_quantize(None, 128, 128, 128, FAKE, FAKE, None, FAKE, None) == ERR_NULL
    assert L.fp8_quantize(FAKE, 128, 128, 128, FAKE, FAKE, None, None, None) == ERR_NULL  # dynamic: workspace
    assert L.fp8_quantize(FAKE, 128, 128, 132, FAKE, FAKE, None, FAKE, None) == ERR_ALIGN  # ldx % 8
    assert L.fp8_quantize(FAKE, 128, 128, 128, FAKE + 8, FAKE, None, FAKE, None) == ERR_ALIGN
    assert L.fp8_quantize(FAKE, 128, 128, 128, FAKE, FAKE + 2, None, FAKE, None) == ERR_ALIGN
    assert L.fp8_pack_weights(None, 256, 256, 0, FAKE, FAKE, FAKE, None) == ERR_NULL
    assert L.fp8_pack_weights(FAKE, 256, 256, 2, FAKE, FAKE, FAKE, None) == ERR_ARG
    assert L.fp8_pack_weights(FAKE, 100, 256, 0, FAKE, FAKE, FAKE, None) == ERR_SHAPE
    assert L.fp8_pack_weights(FAKE, 256, 12, 0, FAKE, FAKE, FAKE, None) == ERR_SHAPE
    assert L.fp8_pack_weights(FAKE, 256, 256, 0, FAKE + 4, FAKE, FAKE, None) == ERR_ALIGN


def test_attention_host_checks():
    L = nv.lib()

    def a(**kw):
        d = dict(qkv=FAKE, M=256, ld=3 * 512, heads=2, hd=256, ws=FAKE, out=FAKE, ldo=512)
        d.update(kw)
        return L.attention_fwd(d["qkv"], d["M"], d["ld"], d["heads"], d["hd"], d["ws"], d["out"], d["ldo"], None,
                               None)
    assert a(hd=128) == ERR_ARG
    assert a(heads=0) == ERR_SHAPE
    assert a(ld=1000) == ERR_SHAPE          # < 3 * heads * 256
    assert a(ldo=256) == ERR_SHAPE
    assert a(M=-1) == ERR_SHAPE
    assert a(M=0, qkv=None, ws=None, out=None) == OK
    assert a(qkv=None) == ERR_NULL
    assert a(ws=None) == ERR_NULL
    assert a(out=None) == ERR_NULL
    assert a(qkv=FAKE + 2) == ERR_ALIGN
    assert a(ld=1540) == ERR_ALIGN
    assert L.attention_workspace_bytes(100, 2) == 2 * 256 * 104 * 2
    assert L.attention_workspace_bytes(0, 2) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_valid_arguments_without_a_gpu_report_the_device():
    assert q() == ERR_DEVICE
    assert g() == ERR_DEVICE
    assert f8g() == ERR_DEVICE
    assert nv.lib().attention_fwd(FAKE, 256, 1536, 2, 256, FAKE, FAKE, 512, None, None) == ERR_DEVICE
    assert nv.lib().fp8_quantize(FAKE, 128, 128, 128, FAKE, FAKE, None, FAKE, None) == ERR_DEVICE
    assert nv.lib().fp8_pack_weights(FAKE, 256, 256, 0, FAKE, FAKE, FAKE, None) == ERR_DEVICE
    assert nv.lib().nvfp4_debug_wait_timeout(FAKE, 1000, None) == ERR_DEVICE


def test_binding_refuses_host_tensors():
    # a host tensor's address must never reach a kernel: the binding refuses it before any call
    x = torch.zeros((128, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        nv.nvfp4_quantize(x)
    with pytest.raises(ValueError):
        nv.fp8_quantize(x)
    with pytest.raises(ValueError):
        nv.attention(torch.zeros((64, 3 * 256), dtype=torch.bfloat16), 1)


def test_debug_build_flag_and_exports():
    # the release library compiles the index checks out; the debug build has them and exports
    # the same entry points
    assert nv.lib().nvfp4_debug_build() == 0
    if os.path.exists(nv.DEBUG_LIB_PATH):
        assert nv.load_library(nv.DEBUG_LIB_PATH).nvfp4_debug_build() == 1
        out = os.popen(f"nm -D --defined-only {nv.DEBUG_LIB_PATH}").read()
        exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("nvfp4")}
        assert exported == set(header_functions())
    assert nv.lib().nvfp4_debug_index_failures(None) == ERR_NULL
