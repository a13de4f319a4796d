"""Python binding of libnvfp4.so, the fused NVFP4 linear layer for B300 (sm_103a).

Argument marshalling only: torch tensors supply device memory and the current CUDA stream,
and every step of the path runs in the library's CUDA kernels. There is no CPU fallback:
if the library is missing or the device is not a B300, calls raise.

    from nvfp4_gemm_act_b300 import nvfp4_quantize, nvfp4_pack_weights, nvfp4_gemm
    a = nvfp4_quantize(x)                                   # x: bf16 [M, K] on cuda
    b = nvfp4_pack_weights(w, gated_interleave=True)        # w: bf16 [K, N] on cuda
    y = nvfp4_gemm(a, b, "gated_silu")                      # bf16 [M, N/2]
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4.so")
# the same library built with the kernels' index checks (nvfp4_debug_build() == 1)
DEBUG_LIB_PATH = os.path.join(_HERE, "libnvfp4_debug.so")

EPILOGUES = {"bias": 0, "head_rmsnorm": 1, "gated_silu": 2}
OUT_DTYPES = {torch.bfloat16: 0, torch.float32: 1}
STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_NULL", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
          4: "NVFP4_ERR_DEVICE", 5: "NVFP4_ERR_LAUNCH", 6: "NVFP4_ERR_TIMEOUT", 7: "NVFP4_ERR_ARG"}

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGS = {
    "nvfp4_scales_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "nvfp4_scale_offset": (_I64, [_I64, _I64, _I64]),
    "nvfp4_workspace_bytes": (ctypes.c_size_t, []),
    "nvfp4_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P]),
    "nvfp4_pack_weights": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, _P]),
    "nvfp4_gemm": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P, _P,
                                  ctypes.c_int, _I64, ctypes.c_float, ctypes.c_int, _P, _I64, _P, _P]),
    "nvfp4_gemm_nvfp4_out": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P, _P,
                                            ctypes.c_int, _I64, ctypes.c_float, _P, _P, _P, _P, _P]),
    "nvfp4_get_device_error": (ctypes.c_int, [_P, _P, _P]),
    "nvfp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nvfp4_debug_wait_timeout": (ctypes.c_int, [_P, _I64, _P]),
    "nvfp4_quantize_noalloc": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
    "nvfp4_debug_build": (ctypes.c_int, []),
    "nvfp4_debug_index_failures": (ctypes.c_int, [_P]),
    "nvfp4_debug_mma_rate": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, ctypes.c_int, _P,
                                            _P, _P]),
    "fp8_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "fp8_pack_weights": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_int, _P, _P, _P, _P]),
    "fp8_gemm": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P, _P, ctypes.c_int, _I64,
                                ctypes.c_float, ctypes.c_int, _P, _I64, _P, _P]),
    "attention_workspace_bytes": (ctypes.c_size_t, [_I64, ctypes.c_int]),
    "attention_fwd": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_int, ctypes.c_int, _P, _P, _I64, _P, _P]),
}


class Nvfp4Error(RuntimeError):
    def __init__(self, func: str, status: int):
        super().__init__(f"{func} returned {STATUS.get(status, status)}")
        self.status = status


def load_library(path: str) -> ctypes.CDLL:
    """Loads a build of the C-ABI library and declares every entry point's signature."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing; build it with `python -m nvfp4_gemm_act_b300.build`")
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load_library(LIB_PATH)
    return _lib


def _check(func: str, status: int) -> None:
    if status != 0:
        raise Nvfp4Error(func, status)


def _ptr(t: Optional[torch.Tensor]):
    """Device address of a CUDA tensor (every tensor the library reads or writes is device
    memory: a host tensor's address would be dereferenced by a kernel)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("nvfp4_gemm_act_b300: expected a CUDA tensor, got one on " + str(t.device))
    return t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class Nvfp4Tensor(NamedTuple):
    """A row-major NVFP4 matrix: codes uint8 [rows, K/2], tiled E4M3 scales, fp32 ts [1]."""
    codes: torch.Tensor
    scales: torch.Tensor
    ts: torch.Tensor
    rows: int
    K: int


def nvfp4_scales_bytes(rows: int, K: int) -> int:
    return lib().nvfp4_scales_bytes(rows, K)


def nvfp4_scale_offset(row: int, kblock: int, K: int) -> int:
    return lib().nvfp4_scale_offset(row, kblock, K)


def nvfp4_workspace_bytes() -> int:
    return lib().nvfp4_workspace_bytes()


def _alloc_nvfp4(rows: int, K: int, device) -> Nvfp4Tensor:
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=device)
    scales = torch.empty(max(nvfp4_scales_bytes(rows, K), 16), dtype=torch.uint8, device=device)
    ts = torch.empty(1, dtype=torch.float32, device=device)
    return Nvfp4Tensor(codes, scales, ts, rows, K)


def nvfp4_quantize(x: torch.Tensor, tensor_scale_in: Optional[torch.Tensor] = None,
                   out: Optional[Nvfp4Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   stream=None) -> Nvfp4Tensor:
    """bf16 [M, K] (row stride x.stride(0)) -> Nvfp4Tensor, via nvfp4_quantize."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = _alloc_nvfp4(M, K, x.device)
    if workspace is None and tensor_scale_in is None:
        workspace = torch.zeros(nvfp4_workspace_bytes(), dtype=torch.uint8, device=x.device)
    _check("nvfp4_quantize", lib().nvfp4_quantize(
        _ptr(x), M, K, x.stride(0), _ptr(out.codes), _ptr(out.scales), _ptr(out.ts),
        _ptr(tensor_scale_in), _ptr(workspace), _stream(stream)))
    return out


def nvfp4_pack_weights(w: torch.Tensor, gated_interleave: bool = False,
                       out: Optional[Nvfp4Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> Nvfp4Tensor:
    """bf16 W [K, N] -> K-major Nvfp4Tensor [N, K] (gated pair interleave optional)."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.is_contiguous()
    K, N = w.shape
    if out is None:
        out = _alloc_nvfp4(N, K, w.device)
    if workspace is None:
        workspace = torch.zeros(nvfp4_workspace_bytes(), dtype=torch.uint8, device=w.device)
    _check("nvfp4_pack_weights", lib().nvfp4_pack_weights(
        _ptr(w), K, N, int(bool(gated_interleave)), _ptr(out.codes), _ptr(out.scales),
        _ptr(out.ts), _ptr(workspace), _stream(stream)))
    return out


def nvfp4_gemm(a: Nvfp4Tensor, b: Nvfp4Tensor, epilogue: str = "bias",
               bias: Optional[torch.Tensor] = None, gamma: Optional[torch.Tensor] = None,
               head_dim: int = 256, norm_cols: int = 0, eps: float = 1e-6,
               out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
               device_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Fused NVFP4 GEMM: epilogue(alpha * A B^T + bias) -> out [M, N] (gated: [M, N/2])."""
    assert a.K == b.K
    M, N, K = a.rows, b.rows, a.K
    width = N // 2 if epilogue == "gated_silu" else N
    if out is None:
        out = torch.empty((M, width), dtype=out_dtype, device=a.codes.device)
    assert out.dtype == out_dtype and out.stride(1) == 1
    _check("nvfp4_gemm", lib().nvfp4_gemm(
        _ptr(a.codes), _ptr(a.scales), _ptr(a.ts), _ptr(b.codes), _ptr(b.scales), _ptr(b.ts),
        M, N, K, EPILOGUES[epilogue], _ptr(bias), _ptr(gamma), head_dim, norm_cols, eps,
        OUT_DTYPES[out_dtype], _ptr(out), out.stride(0), _ptr(device_error), _stream(stream)))
    return out


def nvfp4_gemm_nvfp4_out(a: Nvfp4Tensor, b: Nvfp4Tensor, epilogue: str, out_tensor_scale: torch.Tensor,
                         bias: Optional[torch.Tensor] = None, gamma: Optional[torch.Tensor] = None,
                         head_dim: int = 256, norm_cols: int = 0, eps: float = 1e-6,
                         out: Optional[Nvfp4Tensor] = None, device_error: Optional[torch.Tensor] = None,
                         stream=None) -> Nvfp4Tensor:
    """The fused GEMM writing its output as NVFP4 with a static tensor scale (fp32 [1] on the
    device); the result is an A operand for the next nvfp4_gemm."""
    assert a.K == b.K
    assert out_tensor_scale.dtype == torch.float32 and out_tensor_scale.numel() == 1
    M, N, K = a.rows, b.rows, a.K
    width = N // 2 if epilogue == "gated_silu" else N
    if out is None:
        codes = torch.empty((M, width // 2), dtype=torch.uint8, device=a.codes.device)
        scales = torch.empty(max(nvfp4_scales_bytes(M, width), 16), dtype=torch.uint8, device=a.codes.device)
        out = Nvfp4Tensor(codes, scales, out_tensor_scale, M, width)
    _check("nvfp4_gemm_nvfp4_out", lib().nvfp4_gemm_nvfp4_out(
        _ptr(a.codes), _ptr(a.scales), _ptr(a.ts), _ptr(b.codes), _ptr(b.scales), _ptr(b.ts),
        M, N, K, EPILOGUES[epilogue], _ptr(bias), _ptr(gamma), head_dim, norm_cols, eps,
        _ptr(out_tensor_scale), _ptr(out.codes), _ptr(out.scales), _ptr(device_error), _stream(stream)))
    return out


class Fp8Tensor(NamedTuple):
    """A row-major FP8 (E4M3) matrix: codes uint8 [rows, K], fp32 tensor scale ts [1]."""
    codes: torch.Tensor
    ts: torch.Tensor
    rows: int
    K: int


def _alloc_fp8(rows: int, K: int, device) -> Fp8Tensor:
    return Fp8Tensor(torch.empty((rows, K), dtype=torch.uint8, device=device),
                     torch.empty(1, dtype=torch.float32, device=device), rows, K)


def fp8_quantize(x: torch.Tensor, tensor_scale_in: Optional[torch.Tensor] = None,
                 out: Optional[Fp8Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None) -> Fp8Tensor:
    """bf16 [M, K] (row stride x.stride(0)) -> Fp8Tensor (one scale per tensor), via fp8_quantize."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = _alloc_fp8(M, K, x.device)
    if workspace is None and tensor_scale_in is None:
        workspace = torch.zeros(nvfp4_workspace_bytes(), dtype=torch.uint8, device=x.device)
    _check("fp8_quantize", lib().fp8_quantize(
        _ptr(x), M, K, x.stride(0), _ptr(out.codes), _ptr(out.ts), _ptr(tensor_scale_in), _ptr(workspace),
        _stream(stream)))
    return out


def fp8_pack_weights(w: torch.Tensor, gated_interleave: bool = False, out: Optional[Fp8Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> Fp8Tensor:
    """bf16 W [K, N] -> K-major Fp8Tensor [N, K] (gated pair interleave optional)."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.is_contiguous()
    K, N = w.shape
    if out is None:
        out = _alloc_fp8(N, K, w.device)
    if workspace is None:
        workspace = torch.zeros(nvfp4_workspace_bytes(), dtype=torch.uint8, device=w.device)
    _check("fp8_pack_weights", lib().fp8_pack_weights(
        _ptr(w), K, N, int(bool(gated_interleave)), _ptr(out.codes), _ptr(out.ts), _ptr(workspace),
        _stream(stream)))
    return out


def fp8_gemm(a: Fp8Tensor, b: Fp8Tensor, epilogue: str = "bias", bias: Optional[torch.Tensor] = None,
             gamma: Optional[torch.Tensor] = None, head_dim: int = 256, norm_cols: int = 0, eps: float = 1e-6,
             out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
             device_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Fused FP8 GEMM: epilogue(a.ts * b.ts * A B^T + bias) -> out [M, N] (gated: [M, N/2])."""
    assert a.K == b.K
    M, N, K = a.rows, b.rows, a.K
    width = N // 2 if epilogue == "gated_silu" else N
    if out is None:
        out = torch.empty((M, width), dtype=out_dtype, device=a.codes.device)
    assert out.dtype == out_dtype and out.stride(1) == 1
    _check("fp8_gemm", lib().fp8_gemm(
        _ptr(a.codes), _ptr(a.ts), _ptr(b.codes), _ptr(b.ts), M, N, K, EPILOGUES[epilogue], _ptr(bias),
        _ptr(gamma), head_dim, norm_cols, eps, OUT_DTYPES[out_dtype], _ptr(out), out.stride(0),
        _ptr(device_error), _stream(stream)))
    return out


def attention(qkv: torch.Tensor, heads: int, head_dim: int = 256, out: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, device_error: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """Scaled dot-product attention over the QKV projection's output qkv bf16 [M, >= 3 H]
    (Q | K | V, heads of head_dim side by side; H = heads * head_dim) -> bf16 [M, H]."""
    assert qkv.dtype == torch.bfloat16 and qkv.dim() == 2 and qkv.stride(1) == 1
    M = qkv.shape[0]
    H = heads * head_dim
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=qkv.device)
    if workspace is None:
        workspace = torch.empty(max(lib().attention_workspace_bytes(M, heads), 16), dtype=torch.uint8,
                                device=qkv.device)
    _check("attention_fwd", lib().attention_fwd(
        _ptr(qkv), M, qkv.stride(0), heads, head_dim, _ptr(workspace), _ptr(out), out.stride(0),
        _ptr(device_error), _stream(stream)))
    return out


def nvfp4_get_device_error(device_error: torch.Tensor, stream=None) -> int:
    """Synchronizes the stream, returns the device error word and clears it."""
    code = ctypes.c_int(0)
    _check("nvfp4_get_device_error", lib().nvfp4_get_device_error(
        _ptr(device_error), ctypes.addressof(code), _stream(stream)))
    return code.value


def nvfp4_debug_wait_timeout(device_error: torch.Tensor, timeout_ns: int, stream=None) -> None:
    _check("nvfp4_debug_wait_timeout", lib().nvfp4_debug_wait_timeout(
        _ptr(device_error), timeout_ns, _stream(stream)))


def nvfp4_quantize_noalloc(x: torch.Tensor, out: Optional[Nvfp4Tensor] = None,
                           stream=None) -> Nvfp4Tensor:
    """nvfp4_quantize with a dynamic tensor scale, using the library's fixed scratch instead
    of a workspace (for callers that cannot allocate; calls that overlap on the GPU race)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = _alloc_nvfp4(M, K, x.device)
    _check("nvfp4_quantize_noalloc", lib().nvfp4_quantize_noalloc(
        _ptr(x), M, K, x.stride(0), _ptr(out.codes), _ptr(out.scales), _ptr(out.ts),
        _stream(stream)))
    return out


PROBE_KINDS = {"nvfp4": 0, "fp8": 1, "bf16": 2}
PROBE_K = {"nvfp4": 64, "fp8": 32, "bf16": 16}


def nvfp4_debug_mma_rate(kind: str, cta_group: int, n: int, iters: int, ctas: int,
                         device_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tensor-pipe rate probe: int64 [ctas, 2] of (SM cycles, ns) for `iters` back-to-back
    tcgen05.mma of `kind` ("nvfp4", "fp8", "bf16") at M = 128 * cta_group, N = n, per CTA (pair).
    Asynchronous on the stream; read the result after synchronizing."""
    out = torch.zeros((ctas, 2), dtype=torch.int64, device=torch.cuda.current_device())
    _check("nvfp4_debug_mma_rate", lib().nvfp4_debug_mma_rate(
        PROBE_KINDS[kind], cta_group, n, iters, ctas, _ptr(out), _ptr(device_error), _stream(stream)))
    return out
