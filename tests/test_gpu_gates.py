"""Fused gates on the GPU: g = -exp(A_log) softplus(a + dt_bias) and
beta = sigmoid(b) evaluated inside the kernels, against the fp64 oracle fed the
oracle's own gate values (the gate formula pinned in tests/test_oracle_pins.py)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import gates as ogates
from chunked_gated_delta_gdn_gb300 import (chunk_gated_delta_rule_fused_gates,
                                           gated_delta_decode_fused_gates)
from tests.parity import TOL, f64, rel_l2

pytestmark = pytest.mark.gpu


def gate_inputs(shape, Hv, seed, dtype):
    gen = torch.Generator().manual_seed(seed)
    a = torch.randn(shape + (Hv,), generator=gen).to(dtype)
    b = torch.randn(shape + (Hv,), generator=gen).to(dtype)
    A_log = torch.log(torch.rand(Hv, generator=gen) * 15 + 1)
    dt_bias = 0.5 * torch.randn(Hv, generator=gen)
    return a, b, A_log, dt_bias


@pytest.mark.parametrize("dtype,KV", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_chunk_fused_gates_match_oracle(dtype, KV):
    lengths = [200, 64, 1, 130]
    T = sum(lengths)
    Hqk, Hv = 2, 4
    gen = torch.Generator().manual_seed(31)
    q = torch.randn(1, T, Hqk, KV, generator=gen).to(dtype)
    k = torch.randn(1, T, Hqk, KV, generator=gen).to(dtype)
    v = torch.randn(1, T, Hv, KV, generator=gen).to(dtype)
    s0 = 0.1 * torch.randn(len(lengths), Hv, KV, KV, generator=gen)
    a, b, A_log, dt_bias = gate_inputs((1, T), Hv, 32, dtype)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    dev = "cuda"
    o, fin = chunk_gated_delta_rule_fused_gates(
        q.to(dev), k.to(dev), v.to(dev), a.to(dev), b.to(dev), A_log.to(dev), dt_bias.to(dev),
        initial_state=s0.to(dev), output_final_state=True, use_qk_l2norm_in_kernel=True,
        cu_seqlens=cu.to(dev))
    torch.cuda.synchronize()
    g, beta = ogates.compute_gates(a, b, A_log, dt_bias)
    o_ref, f_ref = oracle.recurrent(q, k, v, g, beta, initial_state=s0,
                                    use_qk_l2norm_in_kernel=True, cu_seqlens=cu)
    e_o, e_f = rel_l2(f64(o), o_ref), rel_l2(f64(fin), f_ref)
    print("fused gates chunk %s: o %.3e final %.3e" % (dtype, e_o, e_f))
    assert e_o <= TOL[dtype] and e_f <= TOL[dtype]


@pytest.mark.parametrize("dtype,KV", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_decode_fused_gates_match_oracle(dtype, KV):
    n, Hqk, Hv, slots = 24, 2, 4, 30
    gen = torch.Generator().manual_seed(41)
    q = torch.randn(n, Hqk, KV, generator=gen).to(dtype)
    k = torch.randn(n, Hqk, KV, generator=gen).to(dtype)
    v = torch.randn(n, Hv, KV, generator=gen).to(dtype)
    cache = 0.1 * torch.randn(slots, Hv, KV, KV, generator=gen)
    idx = torch.randperm(slots, generator=gen)[:n].to(torch.int32)
    idx[[3, 9]] = -1
    a, b, A_log, dt_bias = gate_inputs((n,), Hv, 42, dtype)
    dev = "cuda"
    state = cache.to(dev)
    o = gated_delta_decode_fused_gates(q.to(dev), k.to(dev), v.to(dev), a.to(dev), b.to(dev),
                                       A_log.to(dev), dt_bias.to(dev), state, idx.to(dev))
    torch.cuda.synchronize()
    g, beta = ogates.compute_gates(a, b, A_log, dt_bias)
    ref_cache = f64(cache).copy()
    o_ref = oracle.decode(q, k, v, g, beta, ref_cache, idx)
    e_o, e_s = rel_l2(f64(o), o_ref), rel_l2(f64(state), ref_cache)
    print("fused gates decode %s: o %.3e state %.3e" % (dtype, e_o, e_s))
    assert e_o <= TOL[dtype] and e_s <= TOL[dtype]
    assert torch.count_nonzero(o[[3, 9]].float()).item() == 0
