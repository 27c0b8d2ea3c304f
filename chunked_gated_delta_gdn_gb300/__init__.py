"""GB300-native (sm_103a) gated delta rule: chunkwise forward and slot-indexed decode.

The kernels live in ``libgdn.so`` (C ABI in ``include/gdn.h``); this package is
its thin PyTorch binding:

* :func:`chunk_gated_delta_rule` -- chunkwise forward (training / prefill,
  packed varlen via ``cu_seqlens``, optional slot-cache state I/O).
* :func:`gated_delta_decode` -- one token per request on a slot-indexed
  recurrent-state cache, ``-1`` = padding.
"""
from .api import (GdnError, chunk_fwd_path, chunk_gated_delta_rule,
                  chunk_gated_delta_rule_fused_gates, chunk_workspace_size, gated_delta_decode,
                  gated_delta_decode_fused_gates, gated_delta_decode_multi)

__all__ = ["chunk_gated_delta_rule", "gated_delta_decode", "gated_delta_decode_multi",
           "chunk_gated_delta_rule_fused_gates",
           "gated_delta_decode_fused_gates", "chunk_workspace_size", "chunk_fwd_path", "GdnError"]
__version__ = "0.1.0"
