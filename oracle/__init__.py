"""CPU oracle for the top-k routed MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import, call, link or execute anything in this package.  It shares no
code with the CUDA library (``sparse_moe_router_gb300``), and neither imports the other.
"""
