"""GB300-native Diffuser hot path: sparse attention on a fixed window/global/
random (or BigBird block) graph, followed by K personalized-PageRank diffusion
hops, behind the C-ABI library ``libdiffuser.so`` (see ``include/diffuser.h``).

The CUDA library is loaded on first use of ``sparse_long_sequence_gb300.binding``;
importing this package alone needs no GPU.
"""
__all__ = ["binding", "synthetic", "workloads"]
