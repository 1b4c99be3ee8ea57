"""GB300-native (sm_103a) continuous-batching transformer decode step over a paged KV cache.

The compute path is libns.so (hand-written CUDA: tcgen05 projection GEMMs with fused
RMSNorm/RoPE/KV-write/SwiGLU/residual epilogues, a paged grouped-query decode-attention kernel
with split-K, an embedding + RoPE-table kernel), behind the C ABI in include/ns.h.  This
package is the thin Python binding (``_lib``), the build script (``_build``) and the roofline
arithmetic the benchmark reports (``roofline``).
"""
from . import roofline  # noqa: F401

__all__ = ["roofline"]
