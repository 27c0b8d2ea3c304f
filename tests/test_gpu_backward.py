"""GPU parity of the chunked backward (gdn_chunk_bwd) against the fp64 adjoint oracle:
every gradient (dq, dk, dv, dg, dbeta, d_initial_state) by relative L2 error, on multi-chunk
inputs with ragged tails, packed varlen with empty and one-token sequences, grouped value
heads, odd head dims, L2 norm on and off, fp32 and bf16 I/O; plus determinism, zero gradients
past the last sequence, the autograd op, and a sampled check at the long-context training
shape (4 x 32768 tokens, 32 value heads)."""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdn_gb300 import (chunk_gated_delta_rule_bwd,
                                           chunk_gated_delta_rule_trainable, synthetic)
from tests.parity import TOL, f64, rel_l2

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")


def gpu_bwd(inp, d_o, dfin, **kw):
    d = lambda x: None if x is None else x.cuda()
    out = chunk_gated_delta_rule_bwd(d(inp.q), d(inp.k), d(inp.v), d(inp.g), d(inp.beta),
                                     d(d_o), d(dfin), scale=inp.scale,
                                     initial_state=d(inp.initial_state),
                                     use_qk_l2norm_in_kernel=inp.use_qk_l2norm,
                                     cu_seqlens=d(inp.cu_seqlens), **kw)
    torch.cuda.synchronize()
    return out


def oracle_bwd(inp, d_o, dfin):
    return oracle.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, d_o, dfin, scale=inp.scale,
                           initial_state=inp.initial_state,
                           use_qk_l2norm_in_kernel=inp.use_qk_l2norm, cu_seqlens=inp.cu_seqlens)


def check(inp, d_o, dfin, tol, label):
    got = gpu_bwd(inp, d_o, dfin)
    ref = oracle_bwd(inp, d_o, dfin)
    errs = {name: rel_l2(f64(x), r) for name, x, r in zip(NAMES, got, ref)}
    print("%s: %s (tol %.0e)" % (label, " ".join("%s=%.2e" % kv for kv in errs.items()), tol))
    for name, e in errs.items():
        assert e <= tol, (name, e)
    return got


CASES = {
    # several chunks, ragged tail, batched rows, initial state and final-state gradient
    "fp32_batched_ragged": dict(B=2, T=150, Hqk=1, Hv=2, K=64, V=64, dtype=torch.float32,
                                init="randn", seed=3101),
    # packed varlen with an empty and a one-token sequence, grouped heads, largest dims
    "fp32_varlen_gva_k128": dict(lengths=[100, 0, 1, 257, 64], Hqk=2, Hv=4, K=128, V=128,
                                 dtype=torch.float32, init="randn", seed=3102),
    # no L2 norm, explicit scale, no initial state
    "fp32_no_l2_no_init": dict(B=1, T=200, Hqk=2, Hv=2, K=64, V=64, dtype=torch.float32,
                               init="none", use_qk_l2norm=False, scale=0.3, seed=3103),
    # head dims that are not multiples of 32 (padded tiles, partial V tile)
    "fp32_odd_dims": dict(B=1, T=129, Hqk=1, Hv=3, K=36, V=20, dtype=torch.float32,
                          init="randn", seed=3104),
    # bf16 I/O at the production head shape
    "bf16_varlen_k128": dict(lengths=[130, 65, 7], Hqk=2, Hv=4, K=128, V=128,
                             dtype=torch.bfloat16, init="randn", seed=3105),
    # the GatedDeltaNet gate parameterisation (strong decays)
    "bf16_mixer_gates": dict(B=2, T=300, Hqk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16,
                             init="randn", gates="mixer", seed=3106),
    # tensor-core path edges: many short sequences (partial chunks, TMA boxes reaching into the
    # next sequence), empty sequences first and last, equal head counts
    "bf16_many_short": dict(lengths=[0, 1, 2, 63, 64, 65, 5, 127, 0], Hqk=2, Hv=2, K=128, V=128,
                            dtype=torch.bfloat16, init="randn", seed=3114),
    # tensor-core path without an initial state or a final-state gradient
    "bf16_no_init_no_dfinal": dict(B=1, T=200, Hqk=2, Hv=4, K=128, V=128, dtype=torch.bfloat16,
                                   init="none", seed=3115),
    # tensor-core path with four value heads per query/key head (one grad CTA sums them all)
    "bf16_group_of_four": dict(lengths=[190, 64, 33], Hqk=1, Hv=4, K=128, V=128,
                               dtype=torch.bfloat16, init="randn", seed=3117),
    # tensor-core path without the in-kernel norm (unit-norm rows given), explicit scale
    "bf16_no_l2": dict(B=1, T=130, Hqk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16,
                       init="randn", use_qk_l2norm=False, scale=0.2, seed=3116),
}


def unit_rows(x):
    """Rows scaled to unit L2 norm: what a caller hands in when the kernel does not
    normalise q and k (raw N(0, 1) keys give |k|^2 beta >> 2 and a diverging recurrence,
    whose fp32 rounding no tolerance of 1e-4 survives)."""
    xf = x.float()
    return (xf / xf.norm(dim=-1, keepdim=True)).to(x.dtype)


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_oracle(case):
    inp = synthetic.chunk_inputs(**CASES[case])
    if not inp.use_qk_l2norm:
        inp.q, inp.k = unit_rows(inp.q), unit_rows(inp.k)
    d_o, dfin = synthetic.output_grads(inp, seed=CASES[case]["seed"] + 1,
                                       d_final=case not in ("fp32_no_l2_no_init",
                                                            "bf16_no_init_no_dfinal"))
    check(inp, d_o, dfin, TOL[inp.q.dtype], case)


def test_backward_is_bitwise_deterministic():
    inp = synthetic.chunk_inputs(lengths=[300, 77], Hqk=2, Hv=4, K=128, V=128,
                                 dtype=torch.bfloat16, init="randn", seed=3107)
    d_o, dfin = synthetic.output_grads(inp, seed=3108)
    a = gpu_bwd(inp, d_o, dfin)
    b = gpu_bwd(inp, d_o, dfin)
    for name, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), name


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tokens_past_the_last_sequence_get_zero_gradients(dtype):
    inp = synthetic.chunk_inputs(lengths=[70, 50], Hqk=1, Hv=2, K=128, V=128,
                                 dtype=dtype, init="randn", seed=3109)
    T = inp.q.shape[1]
    pad = 40   # 40 trailing tokens that belong to no sequence
    grow = lambda x, fill=0.0: torch.cat([x, torch.full((1, pad) + tuple(x.shape[2:]), fill,
                                                        dtype=x.dtype)], 1)
    padded = synthetic.ChunkInputs(q=grow(inp.q, 1.0), k=grow(inp.k, 1.0), v=grow(inp.v, 1.0),
                                   g=grow(inp.g, -0.5), beta=grow(inp.beta, 0.5),
                                   initial_state=inp.initial_state, cu_seqlens=inp.cu_seqlens,
                                   state_indices=None, use_qk_l2norm=True, scale=None)
    d_o, dfin = synthetic.output_grads(padded, seed=3110)
    got = gpu_bwd(padded, d_o, dfin)
    ref = oracle_bwd(inp, d_o[:, :T], dfin)
    for name, x, r in zip(NAMES, got, ref):
        if name != "d_initial_state":
            assert torch.count_nonzero(x[:, T:]).item() == 0, name
            x = x[:, :T]
        assert rel_l2(f64(x), r) <= TOL[dtype], name


def test_autograd_op_runs_the_backward_kernel():
    """chunk_gated_delta_rule_trainable's gradients are gdn_chunk_bwd's, bit for bit."""
    inp = synthetic.chunk_inputs(lengths=[90, 200], Hqk=2, Hv=4, K=128, V=128,
                                 dtype=torch.bfloat16, init="randn", seed=3111)
    d_o, dfin = synthetic.output_grads(inp, seed=3112)
    d = lambda x: x.cuda()
    leaves = [d(inp.q), d(inp.k), d(inp.v), d(inp.g), d(inp.beta), d(inp.initial_state)]
    for t in leaves:
        t.requires_grad_(True)
    o, fin = chunk_gated_delta_rule_trainable(*leaves[:5], initial_state=leaves[5],
                                              output_final_state=True,
                                              use_qk_l2norm_in_kernel=True,
                                              cu_seqlens=d(inp.cu_seqlens))
    torch.autograd.backward([o, fin], [d(d_o), d(dfin)])
    torch.cuda.synchronize()
    ref = gpu_bwd(inp, d_o, dfin)
    for name, leaf, r in zip(NAMES, leaves, ref):
        assert torch.equal(leaf.grad, r.to(leaf.grad.dtype)), name


def test_backward_sampled_at_long_context_training_shape():
    """B = 4, T = 32768, Hqk = 16, Hv = 32, K = V = 128, bf16, GatedDeltaNet gates: the GPU
    runs the whole batch; the oracle recomputes one query/key head group (its two value
    heads) of the last sequence over all 32768 tokens."""
    inp = synthetic.chunk_inputs(**{**synthetic.WORKLOADS["long_context_bf16"], "kind": None,
                                    "init": "randn"})
    d_o, dfin = synthetic.output_grads(inp, seed=3113)
    got = gpu_bwd(inp, d_o, dfin)
    b, hq = 3, 5
    hv = slice(2 * hq, 2 * hq + 2)
    sub = lambda x, hs: x[b:b + 1, :, hs].contiguous()
    ref = oracle.backward(sub(inp.q, slice(hq, hq + 1)), sub(inp.k, slice(hq, hq + 1)),
                          sub(inp.v, hv), sub(inp.g, hv), sub(inp.beta, hv), sub(d_o, hv),
                          dfin[b:b + 1, hv], initial_state=inp.initial_state[b:b + 1, hv],
                          use_qk_l2norm_in_kernel=True)
    picks = [got[0][b:b + 1, :, hq:hq + 1], got[1][b:b + 1, :, hq:hq + 1], got[2][b:b + 1, :, hv],
             got[3][b:b + 1, :, hv], got[4][b:b + 1, :, hv], got[5][b:b + 1, hv]]
    errs = {name: rel_l2(f64(x), r) for name, x, r in zip(NAMES, picks, ref)}
    print("long context sampled: %s" % " ".join("%s=%.2e" % kv for kv in errs.items()))
    for name, e in errs.items():
        assert e <= TOL[torch.bfloat16], (name, e)
    for x in got:
        assert torch.isfinite(x.float()).all()
