"""The rule that every pointer handed to the library is memory of the current device
(include/nvfp4.h, conventions), checked without a GPU: the decision function the C ABI calls
after cudaPointerGetAttributes is compiled here with g++ and fed each kind of memory,
including another GPU's memory reached through unified addressing."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nvfp4_gemm_act_b300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdio>
#include "pointer_check.h"
int main() {
  using nvfp4::classify_pointer;
  const struct { const char* name; cudaMemoryType type; int owner; int current; } cases[] = {
    {"device_same", cudaMemoryTypeDevice, 0, 0},
    {"device_same_1", cudaMemoryTypeDevice, 3, 3},
    {"device_foreign", cudaMemoryTypeDevice, 1, 0},
    {"device_foreign_rev", cudaMemoryTypeDevice, 0, 7},
    {"managed_same", cudaMemoryTypeManaged, 2, 2},
    {"managed_foreign", cudaMemoryTypeManaged, 0, 1},
    {"host_pinned", cudaMemoryTypeHost, 0, 0},
    {"unregistered", cudaMemoryTypeUnregistered, -2, 0},
  };
  for (const auto& c : cases) std::printf("%s %d\n", c.name, (int)classify_pointer(c.type, c.owner, c.current));
  return 0;
}
"""


@pytest.fixture(scope="module")
def verdicts(tmp_path_factory):
    if shutil.which("g++") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime_api.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    d = tmp_path_factory.mktemp("ptr")
    src, exe = d / "t.cpp", d / "t"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", f"-I{CSRC}", f"-I{CUDA_INC}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (l.split() for l in out.splitlines())}


OK, ERR_ARG = 0, 7


def test_memory_of_the_current_device_is_accepted(verdicts):
    assert verdicts["device_same"] == OK
    assert verdicts["device_same_1"] == OK
    assert verdicts["managed_same"] == OK


def test_another_gpus_memory_is_refused(verdicts):
    assert verdicts["device_foreign"] == ERR_ARG
    assert verdicts["device_foreign_rev"] == ERR_ARG
    assert verdicts["managed_foreign"] == ERR_ARG


def test_host_memory_is_refused(verdicts):
    assert verdicts["host_pinned"] == ERR_ARG
    assert verdicts["unregistered"] == ERR_ARG


def test_every_compute_entry_point_checks_its_pointers():
    # each entry point that launches work calls check_pointers (directly or through the
    # quantize / GEMM validators) before its launch
    src = open(os.path.join(CSRC, "api.cu")).read()
    for fn in ("nvfp4_pack_weights", "fp8_quantize", "fp8_pack_weights", "attention_fwd",
               "nvfp4_debug_wait_timeout"):
        body = src[src.index(f"nvfp4_status {fn}("):]
        body = body[:body.index("\n}\n")]
        assert "check_pointers(" in body, fn
    for fn, helper in (("nvfp4_quantize", "check_quantize_args("), ("nvfp4_gemm", "gemm_memory_ok("),
                       ("nvfp4_gemm_nvfp4_out", "gemm_memory_ok("), ("fp8_gemm", "gemm_memory_ok(")):
        body = src[src.index(f"nvfp4_status {fn}("):]
        body = body[:body.index("\n}\n")]
        assert helper in body, fn
    noalloc = open(os.path.join(CSRC, "noalloc.cu")).read()
    assert "check_quantize_args(" in noalloc
