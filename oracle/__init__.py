"""CPU oracle for the fused NVFP4 GEMM path (test infrastructure; see nvfp4_ref)."""
from .nvfp4_ref import *  # noqa: F401,F403
