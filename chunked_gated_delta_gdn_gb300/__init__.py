"""GB300-native (sm_103a) gated delta rule: chunkwise forward and slot-indexed decode.

The kernels live in ``libgdn.so`` (C ABI in ``include/gdn.h``); this package is
its thin PyTorch binding:

* :func:`chunk_gated_delta_rule` -- chunkwise forward (training / prefill,
  packed varlen via ``cu_seqlens``, optional slot-cache state I/O).
* :func:`gated_delta_decode` -- one token per request on a slot-indexed
  recurrent-state cache, ``-1`` = padding; :func:`gated_delta_decode_multi` for
  several tokens per request.
* ``*_fused_gates`` -- the same with g and beta computed in the kernels.
* :func:`chunk_gated_delta_product`, :func:`gated_delta_product_decode` -- the Gated
  Delta Product (several delta-rule writes per token).
* :func:`chunk_gated_delta_rule_bwd` -- the backward (dq, dk, dv, dg, dbeta, d_initial_state);
  :func:`chunk_gated_delta_rule_trainable` -- forward + backward as a torch autograd op;
  :func:`chunk_gated_delta_rule_bwd_fused_gates` and
  :func:`chunk_gated_delta_rule_fused_gates_trainable` -- the same through the fused gates
  (gradients w.r.t. a, b, A_log, dt_bias).

Device-side errors (bad slot, bad ``cu_seqlens``, a timed-out in-kernel wait) reach the
caller only through a ``dev_status`` tensor, or as :class:`GdnDeviceError` with ``check=True``.
"""
from .api import (GdnDeviceError, GdnError, chunk_fwd_path, chunk_gated_delta_product, chunk_gated_delta_rule,
                  chunk_gated_delta_rule_bwd, chunk_gated_delta_rule_bwd_fused_gates,
                  chunk_gated_delta_rule_fused_gates, chunk_gated_delta_rule_fused_gates_trainable,
                  chunk_gated_delta_rule_trainable, chunk_workspace_size, gated_delta_decode,
                  gated_delta_decode_fused_gates, gated_delta_decode_multi,
                  gated_delta_product_decode)

__all__ = ["chunk_gated_delta_rule", "gated_delta_decode", "gated_delta_decode_multi",
           "chunk_gated_delta_rule_fused_gates", "gated_delta_decode_fused_gates",
           "chunk_gated_delta_product", "gated_delta_product_decode",
           "chunk_gated_delta_rule_bwd", "chunk_gated_delta_rule_trainable",
           "chunk_gated_delta_rule_bwd_fused_gates", "chunk_gated_delta_rule_fused_gates_trainable",
           "chunk_workspace_size", "chunk_fwd_path", "GdnError", "GdnDeviceError"]
__version__ = "0.1.0"
