"""GB300 (sm_103a) routed FP8 block-scaled MoE FFN.

The compute lives in libmoe_fp8.so (hand-written CUDA, C ABI in include/moe_fp8.h). This
package holds the build script, the ctypes binding (``_lib``) and the seeded workload
generators (``inputs``). Importing the package does not load the library; the first call
through the binding does, and fails loudly if it has not been built.
"""
from ._lib import (MoEError, Shape, make_shape, moe_fp8_combine, moe_fp8_down, moe_fp8_forward,
                   moe_fp8_gate_up, moe_fp8_prepare, moe_fp8_read_status, moe_fp8_version,
                   moe_fp8_workspace_bytes, moe_fp8_workspace_init, moe_fp8_workspace_view,
                   moe_route)

__all__ = ["MoEError", "Shape", "make_shape", "moe_route", "moe_fp8_forward", "moe_fp8_prepare",
           "moe_fp8_gate_up", "moe_fp8_down", "moe_fp8_combine", "moe_fp8_workspace_bytes",
           "moe_fp8_workspace_init", "moe_fp8_workspace_view", "moe_fp8_read_status",
           "moe_fp8_version"]
