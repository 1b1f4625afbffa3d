"""MoE FFN layer (router -> top-k -> group -> SwiGLU experts -> combine) for GB300.

The compute path is the CUDA library ``libmoe.so`` (C ABI, declared in
include/moe.h).  ``binding`` is its thin Python wrapper; importing it fails
loudly when the library has not been built.  ``workloads`` makes seeded
synthetic inputs and ``counters`` counts the algorithmic FLOPs and bytes.
"""

__all__ = ["binding", "workloads", "counters"]
