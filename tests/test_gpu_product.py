"""GPU parity of the Gated Delta Product ("Megatron-Core API: core.ssm.gated_delta_product",
GatedDeltaProductMixer: several delta-rule writes per token) against the fp64 oracle:
the chunked forward on both kernel paths (tensor-core bf16, CUDA-core fp32) with packed
varlen sequences and slot caches, the decode step with padding, prefill-then-decode
continuity, and n_h = 1 against the gated delta rule."""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdn_gb300 import (chunk_gated_delta_product, chunk_gated_delta_rule,
                                           gated_delta_product_decode, synthetic)
from tests.parity import TOL, f64, rel_l2

pytestmark = pytest.mark.gpu


def oracle_chunk(inp):
    """Oracle outputs for a ProductInputs batch; slot caches are gathered / scattered here."""
    init = None
    if inp.state is not None:
        init = inp.state[inp.slots.long()] if inp.slots is not None else inp.state
    return oracle.product(inp.q, inp.k, inp.v, inp.g, inp.beta, initial_state=init,
                          use_qk_l2norm_in_kernel=True, cu_seqlens=inp.cu_seqlens)


def gpu_chunk(inp):
    d = lambda x: None if x is None else x.cuda()
    cache = d(inp.state)
    o, f = chunk_gated_delta_product(d(inp.q), d(inp.k), d(inp.v), d(inp.g), d(inp.beta),
                                     initial_state=cache, output_final_state=True,
                                     use_qk_l2norm_in_kernel=True, cu_seqlens=d(inp.cu_seqlens),
                                     state_indices=d(inp.slots))
    torch.cuda.synchronize()
    return o, f


@pytest.mark.parametrize("case", ["bf16_tc_varlen_slots", "fp32_cuda_core_batched"])
def test_product_chunk_matches_oracle(case):
    if case == "bf16_tc_varlen_slots":
        inp = synthetic.product_inputs(n_h=2, Hqk=2, Hv=4, K=128, V=128, dtype=torch.bfloat16,
                                       lengths=[100, 1, 257, 64, 0, 130], init="slots",
                                       num_slots=9, seed=2101)
    else:
        inp = synthetic.product_inputs(n_h=3, B=2, T=150, Hqk=1, Hv=2, K=64, V=64,
                                       dtype=torch.float32, init="randn", seed=2102)
    o, f = gpu_chunk(inp)
    o_ref, f_ref = oracle_chunk(inp)
    tol = TOL[inp.q.dtype]
    e_o = rel_l2(f64(o), o_ref)
    if inp.slots is not None:
        e_f = rel_l2(f64(f[inp.slots.long().cuda()]), f_ref)
        untouched = sorted(set(range(inp.state.shape[0])) - set(inp.slots.tolist()))
        assert torch.equal(f[untouched].cpu(), inp.state[untouched])
    else:
        e_f = rel_l2(f64(f), f_ref)
    print("product chunk %s: rel-L2 o=%.3e final=%.3e (tol %.0e)" % (case, e_o, e_f, tol))
    assert e_o <= tol and e_f <= tol


def test_product_single_write_is_the_chunk_rule():
    """n_h = 1 gives exactly what chunk_gated_delta_rule gives on the same inputs."""
    inp = synthetic.product_inputs(n_h=1, B=2, T=200, Hqk=2, Hv=4, K=128, V=128,
                                   dtype=torch.bfloat16, init="randn", seed=2103)
    o, f = gpu_chunk(inp)
    d = lambda x: x.cuda()
    o2, f2 = chunk_gated_delta_rule(d(inp.q), d(inp.k[:, :, 0]).contiguous(),
                                    d(inp.v[:, :, 0]).contiguous(), d(inp.g),
                                    d(inp.beta[:, :, 0]).contiguous(), initial_state=d(inp.state),
                                    output_final_state=True, use_qk_l2norm_in_kernel=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(f, f2)


@pytest.mark.parametrize("case", ["bf16_k128", "fp32_k64_intermediate"])
def test_product_decode_matches_oracle(case):
    if case == "bf16_k128":
        inp = synthetic.product_decode_inputs(n_h=2, n=32, Hqk=2, Hv=4, K=128, V=128,
                                              dtype=torch.bfloat16, num_slots=48, seed=2104)
    else:
        inp = synthetic.product_decode_inputs(n_h=3, n=12, Hqk=1, Hv=2, K=64, V=64,
                                              dtype=torch.float32, num_slots=16, seed=2105)
    cache = inp.state.cuda()
    before = cache.clone()
    o, inter = gated_delta_product_decode(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(),
                                          inp.beta.cuda(), cache, inp.slots.cuda(),
                                          output_intermediate_states=(case != "bf16_k128"))
    torch.cuda.synchronize()
    ref_cache = f64(inp.state).copy()
    o_ref = oracle.product_decode(inp.q, inp.k, inp.v, inp.g, inp.beta, ref_cache, inp.slots)
    slots = inp.slots.tolist()
    real = [i for i, s in enumerate(slots) if s >= 0]
    pad = [i for i, s in enumerate(slots) if s < 0]
    tol = TOL[inp.q.dtype]
    used = sorted(slots[i] for i in real)
    e_o = rel_l2(f64(o[real]), o_ref[real])
    e_s = rel_l2(f64(cache[used]), ref_cache[used])
    print("product decode %s: rel-L2 o=%.3e state=%.3e (tol %.0e)" % (case, e_o, e_s, tol))
    assert e_o <= tol and e_s <= tol
    assert pad and torch.count_nonzero(o[pad].float()).item() == 0
    untouched = sorted(set(range(cache.shape[0])) - set(used))
    assert torch.equal(cache[untouched], before[untouched])
    if inter is not None:   # the state after the last write is the slot's new state
        for i in real:
            assert torch.equal(inter[i, -1], cache[slots[i]])


def test_product_prefill_then_decode_continues_the_sequence():
    """Prefill of T tokens then one decode token equals the prefill of all T + 1 tokens."""
    T = 129
    full = synthetic.product_inputs(n_h=2, B=1, T=T + 1, Hqk=2, Hv=4, K=128, V=128,
                                    dtype=torch.bfloat16, init="randn", seed=2106)
    d = lambda x: x.cuda()
    o_all, f_all = chunk_gated_delta_product(d(full.q), d(full.k), d(full.v), d(full.g),
                                             d(full.beta), initial_state=d(full.state),
                                             output_final_state=True, use_qk_l2norm_in_kernel=True)
    _, f_pre = chunk_gated_delta_product(d(full.q[:, :T]).contiguous(), d(full.k[:, :T]).contiguous(),
                                         d(full.v[:, :T]).contiguous(), d(full.g[:, :T]).contiguous(),
                                         d(full.beta[:, :T]).contiguous(),
                                         initial_state=d(full.state), output_final_state=True,
                                         use_qk_l2norm_in_kernel=True)
    cache = f_pre.clone()
    o_dec, _ = gated_delta_product_decode(d(full.q[0, T:]).contiguous(), d(full.k[0, T:]).contiguous(),
                                          d(full.v[0, T:]).contiguous(), d(full.g[0, T:]).contiguous(),
                                          d(full.beta[0, T:]).contiguous(), cache, None)
    torch.cuda.synchronize()
    tol = TOL[torch.bfloat16]
    assert rel_l2(f64(cache), f64(f_all)) <= tol
    assert rel_l2(f64(o_dec[0]), f64(o_all[0, T])) <= tol
