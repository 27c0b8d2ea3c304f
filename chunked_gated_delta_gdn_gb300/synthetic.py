"""Seeded synthetic inputs for the gated delta rule workloads.

This module only draws random numbers with the shapes and value distributions of
the workloads; it holds none of the method's arithmetic, and both the CUDA path
and the CPU oracle are fed from it.  Every tensor is drawn on the CPU with a
``torch.Generator`` seeded per workload (so the values are identical on every
host), in fp32, then cast to the I/O dtype; callers hand the oracle the cast
values (``.double()`` of them), so both sides see identical numbers.

Distributions (the pages fix the argument names and defaults only):

* q, k, v ~ N(0, 1).
* g = -softplus(N(0, 1)) (a log-decay in (-inf, 0)), except ``long_context``
  where g = -exp(A_log) * softplus(a + dt_bias) with A_log = log U(1, 16) per
  value head (the GatedDeltaNet ``A_init_range=(1, 16)`` default on
  "Megatron-Core API: core.ssm.gated_delta_net.gdn"), a ~ N(0, 1) per
  (token, head) and dt_bias ~ 0.5 * N(0, 1) per head.
* beta = sigmoid(N(0, 1)).
* initial / cached states ~ 0.1 * N(0, 1), fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

__all__ = ["ChunkInputs", "DecodeInputs", "ProductInputs", "chunk_inputs", "decode_inputs",
           "product_inputs", "product_decode_inputs", "output_grads", "WORKLOADS",
           "varlen_lengths"]


@dataclasses.dataclass
class ChunkInputs:
    q: torch.Tensor            # [B, T, Hqk, K]
    k: torch.Tensor            # [B, T, Hqk, K]
    v: torch.Tensor            # [B, T, Hv, V]
    g: torch.Tensor            # [B, T, Hv] fp32
    beta: torch.Tensor         # [B, T, Hv]
    initial_state: Optional[torch.Tensor]   # [N, Hv, K, V] fp32 or slot cache [S, Hv, K, V]
    cu_seqlens: Optional[torch.Tensor]      # [N + 1] int32
    state_indices: Optional[torch.Tensor]   # [N] int32 (slot per sequence) or None
    use_qk_l2norm: bool
    scale: Optional[float]


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor            # [n, Hqk, K]
    k: torch.Tensor
    v: torch.Tensor            # [n, Hv, V]
    g: torch.Tensor            # [n, Hv] fp32
    beta: torch.Tensor         # [n, Hv]
    ssm_state: torch.Tensor    # [num_slots, Hv, K, V] fp32
    batch_indices: Optional[torch.Tensor]   # [n] int32, -1 = padding
    use_qk_l2norm: bool
    scale: Optional[float]


# Workload table: name -> keyword arguments of chunk_inputs / decode_inputs.
WORKLOADS = {
    # tiny fp32 chunked forward
    "tiny_fp32": dict(kind="chunk", B=1, T=256, Hqk=2, Hv=2, K=64, V=64, dtype=torch.float32,
                      init="zeros", seed=1001),
    # one long sequence, bf16 I/O, fp32 state, grouped value heads
    "single_seq_bf16": dict(kind="chunk", B=1, T=8192, Hqk=16, Hv=32, K=128, V=128,
                            dtype=torch.bfloat16, init="randn", seed=1002),
    # 32 packed sequences of 100..4096 tokens, states from / to a 64-slot cache
    "varlen_prefill_bf16": dict(kind="chunk", num_seqs=32, min_len=100, max_len=4096, Hqk=16,
                                Hv=32, K=128, V=128, dtype=torch.bfloat16, init="slots",
                                num_slots=64, seed=1003),
    # batched decode, 256 requests (10% padding) on a 512-slot cache
    "decode_bf16": dict(kind="decode", n=256, Hqk=16, Hv=32, K=128, V=128, dtype=torch.bfloat16,
                        num_slots=512, pad_frac=0.1, seed=1004),
    # long-context training shape with the GatedDeltaNet gate parameterisation
    "long_context_bf16": dict(kind="chunk", B=4, T=32768, Hqk=16, Hv=32, K=128, V=128,
                              dtype=torch.bfloat16, init="none", gates="mixer", seed=1005),
}


def _randn(gen, shape, chunk=1 << 24):
    """N(0,1) fp32 drawn in fixed-size pieces (same values regardless of total size order)."""
    out = torch.empty(shape, dtype=torch.float32)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32)
    return out


def varlen_lengths(num_seqs: int, min_len: int, max_len: int, seed: int) -> list:
    """Sequence lengths drawn uniformly from [min_len, max_len] (inclusive)."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(min_len, max_len + 1, (num_seqs,), generator=gen).tolist()


def chunk_inputs(B=1, T=None, Hqk=2, Hv=2, K=64, V=64, dtype=torch.float32, init="zeros",
                 gates="plain", seed=0, num_seqs=None, min_len=None, max_len=None,
                 lengths=None, num_slots=None, use_qk_l2norm=True, scale=None,
                 beta_dtype=None, kind=None) -> ChunkInputs:
    """Inputs for the chunked forward.

    Either ``B, T`` (batched layout) or packed varlen: ``lengths`` (explicit) or
    ``num_seqs, min_len, max_len`` (drawn), giving B = 1, T = sum(lengths) and
    ``cu_seqlens``.  ``init``: "zeros", "randn" ([N, Hv, K, V]), "none" (no
    initial state) or "slots" (a ``num_slots`` cache plus ``state_indices``, a
    seeded random choice of distinct slots).
    """
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is None and num_seqs is not None:
        lengths = varlen_lengths(num_seqs, min_len, max_len, seed + 7919)
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        B, T = 1, int(cu[-1])
        N = len(lengths)
    else:
        N = B
    q = _randn(gen, (B, T, Hqk, K)).to(dtype)
    k = _randn(gen, (B, T, Hqk, K)).to(dtype)
    v = _randn(gen, (B, T, Hv, V)).to(dtype)
    if gates == "mixer":
        A_log = torch.log(torch.rand(Hv, generator=gen) * 15.0 + 1.0)
        a = _randn(gen, (B, T, Hv))
        dt_bias = 0.5 * _randn(gen, (Hv,))
        g = -torch.exp(A_log) * torch.nn.functional.softplus(a + dt_bias)
    else:
        g = -torch.nn.functional.softplus(_randn(gen, (B, T, Hv)))
    beta = torch.sigmoid(_randn(gen, (B, T, Hv))).to(beta_dtype or dtype)
    g = g.to(torch.float32).contiguous()
    init_state = None
    state_indices = None
    if init == "zeros":
        init_state = torch.zeros(N, Hv, K, V, dtype=torch.float32)
    elif init == "randn":
        init_state = 0.1 * _randn(gen, (N, Hv, K, V))
    elif init == "slots":
        init_state = 0.1 * _randn(gen, (num_slots, Hv, K, V))
        state_indices = torch.randperm(num_slots, generator=gen)[:N].to(torch.int32)
    elif init != "none":
        raise ValueError("unknown init %r" % init)
    return ChunkInputs(q=q, k=k, v=v, g=g, beta=beta, initial_state=init_state, cu_seqlens=cu,
                       state_indices=state_indices, use_qk_l2norm=use_qk_l2norm, scale=scale)


def decode_inputs(n=256, Hqk=16, Hv=32, K=128, V=128, dtype=torch.bfloat16, num_slots=512,
                  pad_frac=0.1, seed=0, identity=False, use_qk_l2norm=True, scale=None,
                  beta_dtype=None, kind=None) -> DecodeInputs:
    """Inputs for one decode step: ``n`` requests on a ``num_slots`` cache.

    ``batch_indices``: the first ``n`` entries of a seeded permutation of the
    slots, with round(pad_frac * n) seeded positions set to -1 (padding).
    ``identity=True`` gives ``batch_indices=None`` (static batching).
    """
    gen = torch.Generator().manual_seed(seed)
    q = _randn(gen, (n, Hqk, K)).to(dtype)
    k = _randn(gen, (n, Hqk, K)).to(dtype)
    v = _randn(gen, (n, Hv, V)).to(dtype)
    g = -torch.nn.functional.softplus(_randn(gen, (n, Hv)))
    beta = torch.sigmoid(_randn(gen, (n, Hv))).to(beta_dtype or dtype)
    state = 0.1 * _randn(gen, (num_slots, Hv, K, V))
    idx = None
    if not identity:
        if n > num_slots:
            raise ValueError("n > num_slots needs repeated slots")
        idx = torch.randperm(num_slots, generator=gen)[:n].to(torch.int32)
        n_pad = int(round(pad_frac * n))
        if n_pad:
            pos = torch.randperm(n, generator=gen)[:n_pad]
            idx[pos] = -1
    return DecodeInputs(q=q, k=k, v=v, g=g.contiguous(), beta=beta, ssm_state=state,
                        batch_indices=idx, use_qk_l2norm=use_qk_l2norm, scale=scale)


def workload(name: str, **overrides):
    """Inputs for a named workload of :data:`WORKLOADS` (keyword overrides allowed)."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    if spec.get("kind") == "decode":
        return decode_inputs(**spec)
    return chunk_inputs(**spec)


@dataclasses.dataclass
class ProductInputs:
    q: torch.Tensor            # [B, T, Hqk, K]          (decode: [n, Hqk, K])
    k: torch.Tensor            # [B, T, n_h, Hqk, K]     (decode: [n, n_h, Hqk, K])
    v: torch.Tensor            # [B, T, n_h, Hv, V]      (decode: [n, n_h, Hv, V])
    g: torch.Tensor            # [B, T, Hv] fp32         (decode: [n, Hv])
    beta: torch.Tensor         # [B, T, n_h, Hv]         (decode: [n, n_h, Hv])
    state: Optional[torch.Tensor]           # initial states [N, ...], or the slot cache
    cu_seqlens: Optional[torch.Tensor]
    slots: Optional[torch.Tensor]           # state_indices (chunk) / batch_indices (decode)


def product_inputs(n_h=2, B=1, T=None, Hqk=2, Hv=4, K=128, V=128, dtype=torch.bfloat16,
                   lengths=None, init="randn", num_slots=None, seed=0) -> ProductInputs:
    """Inputs for the Gated Delta Product chunked forward: n_h writes per token, each with its
    own key, value and beta (same distributions as :func:`chunk_inputs`).  ``lengths`` gives
    packed varlen sequences; ``init``: "none", "randn" or "slots" (a ``num_slots`` cache)."""
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is not None:
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        B, T = 1, int(cu[-1])
        N = len(lengths)
    else:
        N = B
    q = _randn(gen, (B, T, Hqk, K)).to(dtype)
    k = _randn(gen, (B, T, n_h, Hqk, K)).to(dtype)
    v = _randn(gen, (B, T, n_h, Hv, V)).to(dtype)
    g = (-torch.nn.functional.softplus(_randn(gen, (B, T, Hv)))).to(torch.float32).contiguous()
    beta = torch.sigmoid(_randn(gen, (B, T, n_h, Hv))).to(dtype)
    state, slots = None, None
    if init == "randn":
        state = 0.1 * _randn(gen, (N, Hv, K, V))
    elif init == "slots":
        state = 0.1 * _randn(gen, (num_slots, Hv, K, V))
        slots = torch.randperm(num_slots, generator=gen)[:N].to(torch.int32)
    elif init != "none":
        raise ValueError("unknown init %r" % init)
    return ProductInputs(q=q, k=k, v=v, g=g, beta=beta, state=state, cu_seqlens=cu, slots=slots)


def product_decode_inputs(n_h=2, n=32, Hqk=2, Hv=4, K=128, V=128, dtype=torch.bfloat16,
                          num_slots=48, pad_frac=0.125, seed=0) -> ProductInputs:
    """One Gated Delta Product token per request on a ``num_slots`` cache; batch_indices as
    in :func:`decode_inputs` (a seeded permutation prefix with padding entries set to -1)."""
    gen = torch.Generator().manual_seed(seed)
    q = _randn(gen, (n, Hqk, K)).to(dtype)
    k = _randn(gen, (n, n_h, Hqk, K)).to(dtype)
    v = _randn(gen, (n, n_h, Hv, V)).to(dtype)
    g = (-torch.nn.functional.softplus(_randn(gen, (n, Hv)))).to(torch.float32).contiguous()
    beta = torch.sigmoid(_randn(gen, (n, n_h, Hv))).to(dtype)
    cache = 0.1 * _randn(gen, (num_slots, Hv, K, V))
    idx = torch.randperm(num_slots, generator=gen)[:n].to(torch.int32)
    npad = int(round(pad_frac * n))
    if npad:
        idx[torch.randperm(n, generator=gen)[:npad]] = -1
    return ProductInputs(q=q, k=k, v=v, g=g, beta=beta, state=cache, cu_seqlens=None, slots=idx)


def output_grads(inp: ChunkInputs, seed=0, d_final=True):
    """Upstream gradients for the backward of a ChunkInputs batch: d_o ~ N(0, 1) in the
    inputs' dtype, shaped like the output, and d_final_state ~ N(0, 1) fp32 [N, Hv, K, V]
    (None when ``d_final`` is False)."""
    gen = torch.Generator().manual_seed(seed)
    B, T = inp.q.shape[:2]
    Hv, V = inp.v.shape[2:]
    K = inp.q.shape[3]
    N = B if inp.cu_seqlens is None else inp.cu_seqlens.numel() - 1
    d_o = _randn(gen, (B, T, Hv, V)).to(inp.q.dtype)
    dfin = _randn(gen, (N, Hv, K, V)) if d_final else None
    return d_o, dfin
