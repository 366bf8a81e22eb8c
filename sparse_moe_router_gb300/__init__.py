"""GB300-native top-k routed Mixture-of-Experts FFN layer.

The compute path is the C-ABI library ``libmoe.so`` (hand-written sm_103a CUDA kernels),
declared in ``include/moe.h`` and bound by ``sparse_moe_router_gb300.abi``.  Importing the
binding raises if the library has not been built: there is no fallback.
"""

__all__ = ["abi", "inputs"]
