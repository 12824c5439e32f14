"""GB300-native sparse Mixture-of-Experts forward (sm_103a).

The compute path lives in the CUDA library ``libmoe.so`` (built from ``csrc/``) behind a
C ABI declared in ``include/moe.h``; ``moe`` is its thin ctypes binding.  Importing this
package does not load the library: ``top_routing_grouped_gb300.moe`` does, and it raises
if the library is missing.
"""
__all__ = ["workloads"]
