"""Python binding of libgdn: argument marshalling around the C ABI, nothing else.

Every step of the computation runs in the CUDA kernels behind ``gdn_chunk_fwd``
and ``gdn_decode``; this module checks tensors, allocates outputs and scratch
with PyTorch (device memory only), and passes raw pointers plus torch's current
CUDA stream.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _lib

__all__ = ["chunk_gated_delta_rule", "gated_delta_decode", "gated_delta_decode_multi",
           "chunk_gated_delta_rule_fused_gates", "chunk_gated_delta_product",
           "gated_delta_product_decode", "chunk_gated_delta_rule_bwd",
           "chunk_gated_delta_rule_trainable",
           "gated_delta_decode_fused_gates", "chunk_gated_delta_rule_bwd_fused_gates",
           "chunk_gated_delta_rule_fused_gates_trainable", "chunk_workspace_size", "chunk_fwd_path",
           "GdnError",
           "GdnDeviceError"]

GdnError = _lib.GdnError

_DT = {torch.float32: _lib.GDN_F32, torch.bfloat16: _lib.GDN_BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor (got %s)" % (name, t.device))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _scale(scale) -> float:
    return float("nan") if scale is None else float(scale)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class GdnDeviceError(RuntimeError):
    """A kernel reported bad data or a timed-out wait through its device status word
    (GDN_DEV_* bits; raised by ``check=True``)."""

    NAMES = {1: "GDN_DEV_BAD_SLOT", 2: "GDN_DEV_BAD_CU_SEQLENS", 4: "GDN_DEV_TIMEOUT"}

    def __init__(self, fn: str, bits: int):
        self.bits = bits
        names = [n for b, n in self.NAMES.items() if bits & b] or ["0x%x" % bits]
        super().__init__("%s reported %s" % (fn, " | ".join(names)))


def _status(dev_status, check, dev):
    """The device status word passed to the C ABI: the caller's, else a fresh one when
    ``check`` asks for the call's device-side errors, else none."""
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
        return dev_status
    if check:
        return torch.zeros(1, dtype=torch.int32, device=dev)
    return None


def _raise_on_status(fn, status, check):
    """With ``check``: wait for the call (its stream) and raise GdnDeviceError if any GDN_DEV_*
    bit is set.  Without it the status is left for the caller to read."""
    if check and status is not None:
        bits = int(status.item())   # synchronises with the call's stream
        if bits:
            raise GdnDeviceError(fn, bits)


DEVICE_ERRORS_DOC = """
    Device-side errors -- a slot index out of range, a cu_seqlens that is not monotone
    within [0, T], a bounded in-kernel wait that timed out -- skip the affected unit (its
    outputs are then left partly written) and are reported only through the device status
    word: pass ``dev_status`` (a [1] int32 CUDA tensor; GDN_DEV_* bits are OR-ed into it) and
    read it after the stream has run, or pass ``check=True`` to have this call synchronise
    and raise GdnDeviceError.  Without either, such errors are silent.
"""


def chunk_fwd_path(K: int, V: int, dtype=torch.bfloat16, beta_dtype=None) -> int:
    """1: fused tcgen05 kernel; 0: fp32 CUDA-core chunk kernels; -1: rejected."""
    return _lib.load().gdn_chunk_fwd_path(K, V, _DT[dtype], _DT[beta_dtype or dtype])


def chunk_workspace_size(B, T, Hqk, Hv, K, V, num_seqs, dtype=torch.bfloat16,
                         beta_dtype=None) -> int:
    n = _lib.load().gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, K, V, num_seqs, _DT[dtype],
                                                 _DT[beta_dtype or dtype])
    if n == (1 << 64) - 1:
        raise ValueError("sizes rejected by gdn_chunk_fwd")
    return int(n)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, chunk_size=64, initial_state=None,
                           output_final_state=False, use_qk_l2norm_in_kernel=False,
                           cu_seqlens=None, *, state_indices=None, out=None, final_state=None,
                           workspace=None, dev_status=None, check=False,
                           **kwargs) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunkwise gated delta rule forward through ``gdn_chunk_fwd``.

    Signature of torch_chunk_gated_delta_rule ("Megatron-Core API:
    core.ssm.gated_delta_net.gdn"): q, k [B, T, Hqk, K]; v [B, T, Hv, V];
    g [B, T, Hv] fp32; beta [B, T, Hv]; scale None -> 1/sqrt(K); chunk_size 64;
    returns ``(o, final_state or None)``.  Extra keyword arguments are accepted and
    ignored, as that function does.

    ``state_indices`` ([N] int32): ``initial_state`` is then a slot cache
    [num_slots, Hv, K, V]; sequence n starts from slot ``state_indices[n]`` and,
    with ``output_final_state``, writes its final state back into that slot of
    ``final_state`` (default: the same cache, updated in place).  Slot -1 marks a
    padding sequence: zero output, no state access.
    """
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 4:
        raise ValueError("q must be [B, T, Hqk, K]")
    B, T, Hqk, K = q.shape
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev)
    if v.dim() != 4 or v.shape[:2] != q.shape[:2]:
        raise ValueError("v must be [B, T, Hv, V]")
    Hv, V = v.shape[2], v.shape[3]
    _need(g, "g", torch.float32, dev, (B, T, Hv))
    _need(beta, "beta", (dt, torch.float32), dev, (B, T, Hv))
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    num_slots = 0
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32, dev, (N,))
        cache = initial_state if initial_state is not None else final_state
        if cache is None:
            raise ValueError("state_indices needs initial_state or final_state (the slot cache)")
        num_slots = cache.shape[0]
        st_shape = (num_slots, Hv, K, V)
        if output_final_state and final_state is None:
            final_state = initial_state
    else:
        st_shape = (N, Hv, K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, st_shape)
    if output_final_state:
        if final_state is None:
            final_state = torch.empty(st_shape, dtype=torch.float32, device=dev)
        _need(final_state, "final_state", torch.float32, dev, st_shape)
    else:
        final_state = None
    if out is None:
        out = torch.empty((B, T, Hv, V), dtype=dt, device=dev)
    _need(out, "out", dt, dev, (B, T, Hv, V))
    L = _lib.load()
    bdt = _DT[beta.dtype]
    need = chunk_workspace_size(B, T, Hqk, Hv, K, V, N, dt, beta.dtype)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev_status = _status(dev_status, check, dev)
    st = L.gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B, T, Hqk, Hv, K, V,
                         _DT[dt], bdt, _scale(scale), int(chunk_size), _ptr(initial_state),
                         int(bool(output_final_state)), _ptr(final_state),
                         int(bool(use_qk_l2norm_in_kernel)), _ptr(cu_seqlens), N,
                         _ptr(state_indices), num_slots, _ptr(out), _ptr(workspace), ws_bytes,
                         _ptr(dev_status), _stream(dev))
    _lib.check("gdn_chunk_fwd", st)
    _raise_on_status("gdn_chunk_fwd", dev_status, check)
    return out, final_state


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, d_o, d_final_state=None, scale=None,
                               chunk_size=64, initial_state=None, use_qk_l2norm_in_kernel=False,
                               cu_seqlens=None, *, need_d_initial_state=True, workspace=None,
                               dev_status=None, check=False):
    """Gradients of :func:`chunk_gated_delta_rule` through ``gdn_chunk_bwd``.

    Takes the forward's inputs (no slot cache) plus ``d_o`` [B, T, Hv, V] (the
    output gradient, q's dtype) and ``d_final_state`` [N, Hv, K, V] fp32 or None.
    Returns ``(dq, dk, dv, dg, dbeta, d_initial_state)``: dq, dk, dv in q's dtype,
    dg and dbeta fp32, d_initial_state fp32 [N, Hv, K, V] (None when
    ``need_d_initial_state`` is False).
    """
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 4:
        raise ValueError("q must be [B, T, Hqk, K]")
    B, T, Hqk, K = q.shape
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev)
    if v.dim() != 4 or v.shape[:2] != q.shape[:2]:
        raise ValueError("v must be [B, T, Hv, V]")
    Hv, V = v.shape[2], v.shape[3]
    _need(g, "g", torch.float32, dev, (B, T, Hv))
    _need(beta, "beta", (dt, torch.float32), dev, (B, T, Hv))
    _need(d_o, "d_o", dt, dev, (B, T, Hv, V))
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    st_shape = (N, Hv, K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, st_shape)
    if d_final_state is not None:
        _need(d_final_state, "d_final_state", torch.float32, dev, st_shape)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty((B, T, Hv), dtype=torch.float32, device=dev)
    dbeta = torch.empty((B, T, Hv), dtype=torch.float32, device=dev)
    dh0 = torch.empty(st_shape, dtype=torch.float32, device=dev) if need_d_initial_state else None
    L = _lib.load()
    bdt = _DT[beta.dtype]
    need = L.gdn_chunk_bwd_workspace_size(B, T, Hqk, Hv, K, V, N, _DT[dt], bdt)
    if need == (1 << 64) - 1:
        raise ValueError("sizes rejected by gdn_chunk_bwd")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(int(need), 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    dev_status = _status(dev_status, check, dev)
    st = L.gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B, T, Hqk, Hv, K, V,
                         _DT[dt], bdt, _scale(scale), int(chunk_size), _ptr(initial_state),
                         int(bool(use_qk_l2norm_in_kernel)), _ptr(cu_seqlens), N, _ptr(d_o),
                         _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                         _ptr(dbeta), _ptr(dh0), _ptr(workspace), ws_bytes, _ptr(dev_status),
                         _stream(dev))
    _lib.check("gdn_chunk_bwd", st)
    _raise_on_status("gdn_chunk_bwd", dev_status, check)
    return dq, dk, dv, dg, dbeta, dh0


class _ChunkGatedDeltaRule(torch.autograd.Function):
    """gdn_chunk_fwd forward, gdn_chunk_bwd backward."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, scale, output_final_state, use_l2,
                cu_seqlens):
        o, fin = chunk_gated_delta_rule(q, k, v, g, beta, scale=scale,
                                        initial_state=initial_state,
                                        output_final_state=output_final_state,
                                        use_qk_l2norm_in_kernel=use_l2, cu_seqlens=cu_seqlens)
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens)
        ctx.scale, ctx.use_l2 = scale, use_l2
        return o, fin

    @staticmethod
    def backward(ctx, d_o, d_fin):
        q, k, v, g, beta, init, cu = ctx.saved_tensors
        dq, dk, dv, dg, db, dh0 = chunk_gated_delta_rule_bwd(
            q, k, v, g, beta, d_o.contiguous(),
            None if d_fin is None else d_fin.contiguous(), scale=ctx.scale,
            initial_state=init, use_qk_l2norm_in_kernel=ctx.use_l2, cu_seqlens=cu,
            need_d_initial_state=init is not None and ctx.needs_input_grad[5])
        return dq, dk, dv, dg, db.to(beta.dtype), dh0, None, None, None, None


def chunk_gated_delta_rule_trainable(q, k, v, g, beta, scale=None, initial_state=None,
                                     output_final_state=False, use_qk_l2norm_in_kernel=False,
                                     cu_seqlens=None):
    """:func:`chunk_gated_delta_rule` as a differentiable op (torch autograd): the
    forward runs ``gdn_chunk_fwd`` and the backward ``gdn_chunk_bwd``.  Returns
    ``(o, final_state or None)``."""
    return _ChunkGatedDeltaRule.apply(q, k, v, g, beta, initial_state, scale,
                                      bool(output_final_state), bool(use_qk_l2norm_in_kernel),
                                      cu_seqlens)


def gated_delta_decode(q, k, v, g, beta, ssm_state, batch_indices=None, scale=None,
                       use_qk_l2norm_in_kernel=True, *, out=None, dev_status=None, check=False) -> torch.Tensor:
    """One decode token per request through ``gdn_decode``; ``ssm_state`` is updated in place.

    q, k [n, Hqk, K]; v [n, Hv, V]; g [n, Hv] fp32; beta [n, Hv];
    ssm_state [num_slots, Hv, K, V] fp32; batch_indices [n] int32 (-1 = padding) or
    None (request i uses slot i).  Returns o [n, Hv, V].
    """
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 3:
        raise ValueError("q must be [n, Hqk, K]")
    n, Hqk, K = q.shape
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev)
    if v.dim() != 3 or v.shape[0] != n:
        raise ValueError("v must be [n, Hv, V]")
    Hv, V = v.shape[1], v.shape[2]
    _need(g, "g", torch.float32, dev, (n, Hv))
    _need(beta, "beta", (dt, torch.float32), dev, (n, Hv))
    _need(ssm_state, "ssm_state", torch.float32, dev)
    if ssm_state.dim() != 4 or tuple(ssm_state.shape[1:]) != (Hv, K, V):
        raise ValueError("ssm_state must be [num_slots, Hv, K, V]")
    if batch_indices is not None:
        _need(batch_indices, "batch_indices", torch.int32, dev, (n,))
    if out is None:
        out = torch.empty((n, Hv, V), dtype=dt, device=dev)
    _need(out, "out", dt, dev, (n, Hv, V))
    dev_status = _status(dev_status, check, dev)
    st = _lib.load().gdn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ssm_state),
                                ssm_state.shape[0], _ptr(batch_indices), n, Hqk, Hv, K, V,
                                _DT[dt], _DT[beta.dtype], _scale(scale),
                                int(bool(use_qk_l2norm_in_kernel)), _ptr(out), _ptr(dev_status),
                                _stream(dev))
    _lib.check("gdn_decode", st)
    _raise_on_status("gdn_decode", dev_status, check)
    return out


def _gate_args(a, b, A_log, dt_bias, dev, dt, lead_shape, Hv):
    _need(a, "a", (dt, torch.float32), dev, tuple(lead_shape) + (Hv,))
    _need(b, "b", a.dtype, dev, tuple(lead_shape) + (Hv,))
    _need(A_log, "A_log", torch.float32, dev, (Hv,))
    _need(dt_bias, "dt_bias", torch.float32, dev, (Hv,))
    return _DT[a.dtype]


def chunk_gated_delta_rule_fused_gates(q, k, v, a, b, A_log, dt_bias, scale=None, chunk_size=64,
                                       initial_state=None, output_final_state=False,
                                       use_qk_l2norm_in_kernel=False, cu_seqlens=None, *,
                                       state_indices=None, out=None, final_state=None,
                                       workspace=None, dev_status=None, check=False, **kwargs):
    """Chunked forward with the gates computed in the kernels (``gdn_chunk_fwd_gated``):
    g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b), with a, b [B, T, Hv]
    and A_log, dt_bias [Hv] fp32.  Everything else as :func:`chunk_gated_delta_rule`."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q must be [B, T, Hqk, K] and v [B, T, Hv, V]")
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev)
    ab_dt = _gate_args(a, b, A_log, dt_bias, dev, dt, (B, T), Hv)
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    num_slots = 0
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32, dev, (N,))
        cache = initial_state if initial_state is not None else final_state
        num_slots = cache.shape[0]
        st_shape = (num_slots, Hv, K, V)
        if output_final_state and final_state is None:
            final_state = initial_state
    else:
        st_shape = (N, Hv, K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, st_shape)
    if output_final_state:
        if final_state is None:
            final_state = torch.empty(st_shape, dtype=torch.float32, device=dev)
        _need(final_state, "final_state", torch.float32, dev, st_shape)
    else:
        final_state = None
    if out is None:
        out = torch.empty((B, T, Hv, V), dtype=dt, device=dev)
    _need(out, "out", dt, dev, (B, T, Hv, V))
    need = chunk_workspace_size(B, T, Hqk, Hv, K, V, N, dt, dt)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev_status = _status(dev_status, check, dev)
    st = _lib.load().gdn_chunk_fwd_gated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), ab_dt, _ptr(A_log), _ptr(dt_bias), B, T,
        Hqk, Hv, K, V, _DT[dt], _scale(scale), int(chunk_size), _ptr(initial_state),
        int(bool(output_final_state)), _ptr(final_state), int(bool(use_qk_l2norm_in_kernel)),
        _ptr(cu_seqlens), N, _ptr(state_indices), num_slots, _ptr(out), _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream(dev))
    _lib.check("gdn_chunk_fwd_gated", st)
    _raise_on_status("gdn_chunk_fwd_gated", dev_status, check)
    return out, final_state


def chunk_gated_delta_rule_bwd_fused_gates(q, k, v, a, b, A_log, dt_bias, d_o,
                                           d_final_state=None, scale=None, chunk_size=64,
                                           initial_state=None, use_qk_l2norm_in_kernel=False,
                                           cu_seqlens=None, *, need_d_initial_state=True,
                                           workspace=None, dev_status=None, check=False):
    """Gradients of :func:`chunk_gated_delta_rule_fused_gates` through ``gdn_chunk_bwd_gated``.

    Returns ``(dq, dk, dv, da, db, dA_log, ddt_bias, d_initial_state)``: dq, dk, dv in q's
    dtype; da, db [B, T, Hv] and dA_log, ddt_bias [Hv] fp32; d_initial_state fp32
    [N, Hv, K, V] (None when ``need_d_initial_state`` is False).  No slot cache."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q must be [B, T, Hqk, K] and v [B, T, Hv, V]")
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev)
    ab_dt = _gate_args(a, b, A_log, dt_bias, dev, dt, (B, T), Hv)
    _need(d_o, "d_o", dt, dev, (B, T, Hv, V))
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    st_shape = (N, Hv, K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, st_shape)
    if d_final_state is not None:
        _need(d_final_state, "d_final_state", torch.float32, dev, st_shape)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    da = torch.empty((B, T, Hv), dtype=torch.float32, device=dev)
    db = torch.empty((B, T, Hv), dtype=torch.float32, device=dev)
    dA_log = torch.empty(Hv, dtype=torch.float32, device=dev)
    ddt_bias = torch.empty(Hv, dtype=torch.float32, device=dev)
    dh0 = torch.empty(st_shape, dtype=torch.float32, device=dev) if need_d_initial_state else None
    L = _lib.load()
    need = L.gdn_chunk_bwd_gated_workspace_size(B, T, Hqk, Hv, K, V, N, _DT[dt])
    if need == (1 << 64) - 1:
        raise ValueError("sizes rejected by gdn_chunk_bwd_gated")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(int(need), 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    dev_status = _status(dev_status, check, dev)
    st = L.gdn_chunk_bwd_gated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), ab_dt, _ptr(A_log), _ptr(dt_bias), B, T,
        Hqk, Hv, K, V, _DT[dt], _scale(scale), int(chunk_size), _ptr(initial_state),
        int(bool(use_qk_l2norm_in_kernel)), _ptr(cu_seqlens), N, _ptr(d_o), _ptr(d_final_state),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da), _ptr(db), _ptr(dA_log), _ptr(ddt_bias),
        _ptr(dh0), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(dev))
    _lib.check("gdn_chunk_bwd_gated", st)
    _raise_on_status("gdn_chunk_bwd_gated", dev_status, check)
    return dq, dk, dv, da, db, dA_log, ddt_bias, dh0


class _ChunkGatedDeltaRuleFusedGates(torch.autograd.Function):
    """gdn_chunk_fwd_gated forward, gdn_chunk_bwd_gated backward."""

    @staticmethod
    def forward(ctx, q, k, v, a, b, A_log, dt_bias, initial_state, scale, output_final_state,
                use_l2, cu_seqlens):
        o, fin = chunk_gated_delta_rule_fused_gates(
            q, k, v, a, b, A_log, dt_bias, scale=scale, initial_state=initial_state,
            output_final_state=output_final_state, use_qk_l2norm_in_kernel=use_l2,
            cu_seqlens=cu_seqlens)
        ctx.save_for_backward(q, k, v, a, b, A_log, dt_bias, initial_state, cu_seqlens)
        ctx.scale, ctx.use_l2 = scale, use_l2
        return o, fin

    @staticmethod
    def backward(ctx, d_o, d_fin):
        q, k, v, a, b, A_log, dt_bias, init, cu = ctx.saved_tensors
        dq, dk, dv, da, db, dA, ddt, dh0 = chunk_gated_delta_rule_bwd_fused_gates(
            q, k, v, a, b, A_log, dt_bias, d_o.contiguous(),
            None if d_fin is None else d_fin.contiguous(), scale=ctx.scale, initial_state=init,
            use_qk_l2norm_in_kernel=ctx.use_l2, cu_seqlens=cu,
            need_d_initial_state=init is not None and ctx.needs_input_grad[7])
        return (dq, dk, dv, da.to(a.dtype), db.to(b.dtype), dA, ddt, dh0, None, None, None, None)


def chunk_gated_delta_rule_fused_gates_trainable(q, k, v, a, b, A_log, dt_bias, scale=None,
                                                 initial_state=None, output_final_state=False,
                                                 use_qk_l2norm_in_kernel=False, cu_seqlens=None):
    """:func:`chunk_gated_delta_rule_fused_gates` as a differentiable op (torch autograd): the
    forward is gdn_chunk_fwd_gated, the backward gdn_chunk_bwd_gated, so gradients reach the
    gate features a, b and the parameters A_log, dt_bias."""
    return _ChunkGatedDeltaRuleFusedGates.apply(q, k, v, a, b, A_log, dt_bias, initial_state,
                                                scale, output_final_state,
                                                use_qk_l2norm_in_kernel, cu_seqlens)


def gated_delta_decode_fused_gates(q, k, v, a, b, A_log, dt_bias, ssm_state, batch_indices=None,
                                   scale=None, use_qk_l2norm_in_kernel=True, *, out=None,
                                   dev_status=None, check=False):
    """Decode step with the gates computed in the kernel (``gdn_decode_gated``); a, b [n, Hv]."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    n, Hqk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev)
    ab_dt = _gate_args(a, b, A_log, dt_bias, dev, dt, (n,), Hv)
    _need(ssm_state, "ssm_state", torch.float32, dev)
    if batch_indices is not None:
        _need(batch_indices, "batch_indices", torch.int32, dev, (n,))
    if out is None:
        out = torch.empty((n, Hv, V), dtype=dt, device=dev)
    dev_status = _status(dev_status, check, dev)
    st = _lib.load().gdn_decode_gated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), ab_dt, _ptr(A_log), _ptr(dt_bias),
        _ptr(ssm_state), ssm_state.shape[0], _ptr(batch_indices), n, Hqk, Hv, K, V, _DT[dt],
        _scale(scale), int(bool(use_qk_l2norm_in_kernel)), _ptr(out), _ptr(dev_status),
        _stream(dev))
    _lib.check("gdn_decode_gated", st)
    _raise_on_status("gdn_decode_gated", dev_status, check)
    return out


def gated_delta_decode_multi(q, k, v, g, beta, ssm_state, batch_indices=None, scale=None,
                             use_qk_l2norm_in_kernel=True, output_intermediate_states=False, *,
                             out=None, intermediate_states=None, dev_status=None, check=False):
    """L decode tokens per request through ``gdn_decode_multi``.

    q, k [n, L, Hqk, K]; v [n, L, Hv, V]; g [n, L, Hv] fp32; beta [n, L, Hv];
    ssm_state [num_slots, Hv, K, V] fp32 (updated in place to the state after the last
    token).  Returns ``(o [n, L, Hv, V], intermediate_states [n, L, Hv, K, V] or None)``.
    """
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q must be [n, L, Hqk, K] and v [n, L, Hv, V]")
    n, L, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev, (n, L, Hv, V))
    _need(g, "g", torch.float32, dev, (n, L, Hv))
    _need(beta, "beta", (dt, torch.float32), dev, (n, L, Hv))
    _need(ssm_state, "ssm_state", torch.float32, dev)
    if batch_indices is not None:
        _need(batch_indices, "batch_indices", torch.int32, dev, (n,))
    if out is None:
        out = torch.empty((n, L, Hv, V), dtype=dt, device=dev)
    if output_intermediate_states and intermediate_states is None:
        intermediate_states = torch.empty((n, L, Hv, K, V), dtype=torch.float32, device=dev)
    if intermediate_states is not None:
        _need(intermediate_states, "intermediate_states", torch.float32, dev, (n, L, Hv, K, V))
    dev_status = _status(dev_status, check, dev)
    st = _lib.load().gdn_decode_multi(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ssm_state), ssm_state.shape[0],
        _ptr(batch_indices), n, L, Hqk, Hv, K, V, _DT[dt], _DT[beta.dtype], _scale(scale),
        int(bool(use_qk_l2norm_in_kernel)), _ptr(out), _ptr(intermediate_states),
        _ptr(dev_status), _stream(dev))
    _lib.check("gdn_decode_multi", st)
    _raise_on_status("gdn_decode_multi", dev_status, check)
    return out, intermediate_states


def chunk_gated_delta_product(q, k, v, g, beta, scale=None, chunk_size=64, initial_state=None,
                              output_final_state=False, use_qk_l2norm_in_kernel=False,
                              cu_seqlens=None, *, state_indices=None, out=None, final_state=None,
                              workspace=None, dev_status=None, check=False,
                              **kwargs) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Gated Delta Product forward through ``gdn_product_chunk_fwd``: n_h delta-rule writes
    per token ("Megatron-Core API: core.ssm.gated_delta_product", GatedDeltaProductMixer).

    q [B, T, Hqk, K]; k [B, T, n_h, Hqk, K]; v [B, T, n_h, Hv, V]; g [B, T, Hv] fp32;
    beta [B, T, n_h, Hv].  Every other argument as :func:`chunk_gated_delta_rule`.
    Returns ``(o [B, T, Hv, V], final_state or None)``.
    """
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 4 or k.dim() != 5 or v.dim() != 5:
        raise ValueError("q must be [B, T, Hqk, K], k [B, T, n_h, Hqk, K], v [B, T, n_h, Hv, V]")
    B, T, Hqk, K = q.shape
    n_h = k.shape[2]
    Hv, V = v.shape[3], v.shape[4]
    _need(k, "k", dt, dev, (B, T, n_h, Hqk, K))
    _need(v, "v", dt, dev, (B, T, n_h, Hv, V))
    _need(g, "g", torch.float32, dev, (B, T, Hv))
    _need(beta, "beta", (dt, torch.float32), dev, (B, T, n_h, Hv))
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    num_slots = 0
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32, dev, (N,))
        cache = initial_state if initial_state is not None else final_state
        if cache is None:
            raise ValueError("state_indices needs initial_state or final_state (the slot cache)")
        num_slots = cache.shape[0]
        st_shape = (num_slots, Hv, K, V)
        if output_final_state and final_state is None:
            final_state = initial_state
    else:
        st_shape = (N, Hv, K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, st_shape)
    if output_final_state:
        if final_state is None:
            final_state = torch.empty(st_shape, dtype=torch.float32, device=dev)
        _need(final_state, "final_state", torch.float32, dev, st_shape)
    else:
        final_state = None
    if out is None:
        out = torch.empty((B, T, Hv, V), dtype=dt, device=dev)
    _need(out, "out", dt, dev, (B, T, Hv, V))
    L = _lib.load()
    need = L.gdn_product_chunk_fwd_workspace_size(B, T, n_h, Hqk, Hv, K, V, N, _DT[dt],
                                                  _DT[beta.dtype])
    if need == (1 << 64) - 1:
        raise ValueError("sizes rejected by gdn_product_chunk_fwd")
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev_status = _status(dev_status, check, dev)
    st = L.gdn_product_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B, T, n_h, Hqk,
                                 Hv, K, V, _DT[dt], _DT[beta.dtype], _scale(scale),
                                 int(chunk_size), _ptr(initial_state),
                                 int(bool(output_final_state)), _ptr(final_state),
                                 int(bool(use_qk_l2norm_in_kernel)), _ptr(cu_seqlens), N,
                                 _ptr(state_indices), num_slots, _ptr(out), _ptr(workspace),
                                 ws_bytes, _ptr(dev_status), _stream(dev))
    _lib.check("gdn_product_chunk_fwd", st)
    _raise_on_status("gdn_product_chunk_fwd", dev_status, check)
    return out, final_state


def gated_delta_product_decode(q, k, v, g, beta, ssm_state, batch_indices=None, scale=None,
                               use_qk_l2norm_in_kernel=True, output_intermediate_states=False, *,
                               out=None, intermediate_states=None, dev_status=None, check=False):
    """One Gated Delta Product token per request through ``gdn_product_decode``.

    q [n, Hqk, K]; k [n, n_h, Hqk, K]; v [n, n_h, Hv, V]; g [n, Hv] fp32; beta [n, n_h, Hv];
    ssm_state [num_slots, Hv, K, V] fp32, updated in place.  Returns ``(o [n, Hv, V],
    intermediate_states [n, n_h, Hv, K, V] or None)``.
    """
    _need(q, "q", (torch.float32, torch.bfloat16))
    dev, dt = q.device, q.dtype
    if q.dim() != 3 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q must be [n, Hqk, K], k [n, n_h, Hqk, K], v [n, n_h, Hv, V]")
    n, Hqk, K = q.shape
    n_h = k.shape[1]
    Hv, V = v.shape[2], v.shape[3]
    _need(k, "k", dt, dev, (n, n_h, Hqk, K))
    _need(v, "v", dt, dev, (n, n_h, Hv, V))
    _need(g, "g", torch.float32, dev, (n, Hv))
    _need(beta, "beta", (dt, torch.float32), dev, (n, n_h, Hv))
    _need(ssm_state, "ssm_state", torch.float32, dev)
    if batch_indices is not None:
        _need(batch_indices, "batch_indices", torch.int32, dev, (n,))
    if out is None:
        out = torch.empty((n, Hv, V), dtype=dt, device=dev)
    _need(out, "out", dt, dev, (n, Hv, V))
    if output_intermediate_states and intermediate_states is None:
        intermediate_states = torch.empty((n, n_h, Hv, K, V), dtype=torch.float32, device=dev)
    if intermediate_states is not None:
        _need(intermediate_states, "intermediate_states", torch.float32, dev, (n, n_h, Hv, K, V))
    dev_status = _status(dev_status, check, dev)
    st = _lib.load().gdn_product_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ssm_state), ssm_state.shape[0],
        _ptr(batch_indices), n, n_h, Hqk, Hv, K, V, _DT[dt], _DT[beta.dtype], _scale(scale),
        int(bool(use_qk_l2norm_in_kernel)), _ptr(out), _ptr(intermediate_states),
        _ptr(dev_status), _stream(dev))
    _lib.check("gdn_product_decode", st)
    _raise_on_status("gdn_product_decode", dev_status, check)
    return out, intermediate_states


for _fn in (chunk_gated_delta_rule, chunk_gated_delta_rule_bwd, gated_delta_decode,
            chunk_gated_delta_rule_fused_gates, gated_delta_decode_fused_gates,
            gated_delta_decode_multi, chunk_gated_delta_product, gated_delta_product_decode):
    _fn.__doc__ = (_fn.__doc__ or "").rstrip() + "\n" + DEVICE_ERRORS_DOC
