"""Tile-signalled grouped MoE expert-combine path for GB300 (sm_103a).

The compute path is the CUDA library libmoe_tsg.so (include/moe_tsg.h); this
package holds its ctypes binding (capi), a small owner of the torch
allocations (runtime.ExpertCombine), the build script and the workload shapes.
"""
from . import workloads  # noqa: F401

__all__ = ["capi", "runtime", "workloads", "build"]
