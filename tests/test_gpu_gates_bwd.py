"""GPU parity of the backward through the fused gates (gdn_chunk_bwd_gated) against the fp64
oracle: the adjoint's dg, dbeta carried through oracle.gates.gates_backward (pinned by finite
differences in tests/test_oracle_backward_pins.py) give da, db, dA_log, ddt_bias; dq, dk, dv and
the initial-state gradient come from the adjoint directly.  Also: zero gate gradients past the
last sequence, bitwise determinism, and the autograd op."""
import numpy as np
import pytest
import torch

import oracle
from oracle import gates as ogates
from chunked_gated_delta_gdn_gb300 import (chunk_gated_delta_rule_bwd_fused_gates,
                                           chunk_gated_delta_rule_fused_gates_trainable)
from tests.parity import TOL, f64, rel_l2

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "da", "db", "dA_log", "ddt_bias", "d_initial_state")


def make_case(dtype, KV, lengths=None, B=1, T=None, Hqk=2, Hv=4, seed=0, pad=0):
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is not None:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
        B, T, N = 1, int(sum(lengths)) + pad, len(lengths)
    else:
        N = B
    rnd = lambda *s: torch.randn(*s, generator=gen)
    case = dict(q=rnd(B, T, Hqk, KV).to(dtype), k=rnd(B, T, Hqk, KV).to(dtype),
                v=rnd(B, T, Hv, KV).to(dtype), a=rnd(B, T, Hv).to(dtype), b=rnd(B, T, Hv).to(dtype),
                A_log=torch.log(torch.rand(Hv, generator=gen) * 15 + 1),
                dt_bias=0.5 * rnd(Hv), init=0.1 * rnd(N, Hv, KV, KV), cu=cu,
                d_o=rnd(B, T, Hv, KV).to(dtype), dfin=rnd(N, Hv, KV, KV))
    return case


def gpu(case, **kw):
    d = {k: (None if x is None else x.cuda()) for k, x in case.items()}
    out = chunk_gated_delta_rule_bwd_fused_gates(
        d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["d_o"], d["dfin"],
        initial_state=d["init"], use_qk_l2norm_in_kernel=True, cu_seqlens=d["cu"], **kw)
    torch.cuda.synchronize()
    return out


def reference(case, T_used=None):
    c = dict(case)
    if T_used is not None:   # the oracle sees only the tokens that belong to a sequence
        for key in ("q", "k", "v", "a", "b", "d_o"):
            c[key] = c[key][:, :T_used]
    g, beta = ogates.compute_gates(c["a"], c["b"], c["A_log"], c["dt_bias"])
    dq, dk, dv, dg, dbeta, dinit = oracle.backward(
        c["q"], c["k"], c["v"], g, beta, c["d_o"], c["dfin"], initial_state=c["init"],
        use_qk_l2norm_in_kernel=True, cu_seqlens=c["cu"])
    da, db, dA_log, ddt_bias = ogates.gates_backward(c["a"], c["b"], c["A_log"], c["dt_bias"],
                                                     dg, dbeta)
    return dq, dk, dv, da, db, dA_log, ddt_bias, dinit


@pytest.mark.parametrize("dtype,KV,layout", [(torch.bfloat16, 128, "varlen"),
                                             (torch.float32, 64, "batched")])
def test_gated_backward_matches_oracle(dtype, KV, layout):
    if layout == "varlen":
        case = make_case(dtype, KV, lengths=[200, 0, 64, 1, 131], seed=501)
    else:
        case = make_case(dtype, KV, B=2, T=150, Hqk=1, Hv=2, seed=502)
    got = gpu(case)
    ref = reference(case)
    errs = {n: rel_l2(f64(x), r) for n, x, r in zip(NAMES, got, ref)}
    print("gated bwd %s %s: %s" % (dtype, layout, " ".join("%s=%.2e" % kv for kv in errs.items())))
    for n, e in errs.items():
        assert e <= TOL[dtype], (n, e)


def test_gate_gradients_zero_past_the_last_sequence():
    case = make_case(torch.bfloat16, 128, lengths=[90, 40], seed=503, pad=30)
    got = gpu(case)
    T_used = 130
    for n in ("da", "db"):
        x = got[NAMES.index(n)]
        assert torch.count_nonzero(x[:, T_used:]).item() == 0, n
    ref = reference(case, T_used=T_used)
    for n, x, r in zip(NAMES, got, ref):
        if n in ("dq", "dk", "dv", "da", "db"):
            x = x[:, :T_used]
        assert rel_l2(f64(x), r) <= TOL[torch.bfloat16], n


def test_gated_backward_is_bitwise_deterministic():
    case = make_case(torch.bfloat16, 128, lengths=[300, 77], seed=504)
    a, b = gpu(case), gpu(case)
    for n, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), n


def test_fused_gates_autograd_op_runs_the_gated_backward():
    """chunk_gated_delta_rule_fused_gates_trainable's gradients are gdn_chunk_bwd_gated's."""
    case = make_case(torch.bfloat16, 128, lengths=[90, 200], seed=505)
    direct = gpu(case)
    leaves = {k: case[k].cuda().requires_grad_(True)
              for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "init")}
    o, fin = chunk_gated_delta_rule_fused_gates_trainable(
        leaves["q"], leaves["k"], leaves["v"], leaves["a"], leaves["b"], leaves["A_log"],
        leaves["dt_bias"], initial_state=leaves["init"], output_final_state=True,
        use_qk_l2norm_in_kernel=True, cu_seqlens=case["cu"].cuda())
    loss = (o.float() * case["d_o"].cuda().float()).sum() + (fin * case["dfin"].cuda()).sum()
    loss.backward()
    order = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "init")
    for name, key, x in zip(NAMES, order, direct):
        got = leaves[key].grad
        assert got is not None, name
        ref = x.to(got.dtype)
        assert torch.equal(got, ref), name
