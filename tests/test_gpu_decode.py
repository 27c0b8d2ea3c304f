"""GPU parity of gdn_decode against the fp64 oracle, plus the exact properties:
padding rows are +0.0, slots not named are byte-identical, each request's state
lands in its own slot."""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdn_gb300 import gated_delta_decode, synthetic
from chunked_gated_delta_gdn_gb300._lib import GDN_DEV_BAD_SLOT
from tests.parity import TOL, f64, rel_l2

pytestmark = pytest.mark.gpu


def run_case(inp, label):
    dev = "cuda"
    state_gpu = inp.ssm_state.to(dev)
    before = state_gpu.clone()
    idx = None if inp.batch_indices is None else inp.batch_indices.to(dev)
    # the output lives between two canary rows, every element NaN before the call: padding
    # rows must come back as written zeros, the canaries bit-identical
    n_req, Hv, V = inp.v.shape
    buf = torch.full((n_req + 2, Hv, V), float("nan"), dtype=inp.v.dtype, device=dev)
    canary = buf[[0, n_req + 1]].clone()
    o = gated_delta_decode(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.g.to(dev),
                           inp.beta.to(dev), state_gpu, idx, scale=inp.scale,
                           use_qk_l2norm_in_kernel=inp.use_qk_l2norm, out=buf[1:n_req + 1])
    torch.cuda.synchronize()
    ibits = torch.int16 if buf.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(buf[[0, n_req + 1]].view(ibits), canary.view(ibits)), "decode wrote outside o"
    assert torch.isfinite(o.float()).all(), "decode left output rows unwritten"
    cache = f64(inp.ssm_state).copy()
    o_ref = oracle.decode(inp.q, inp.k, inp.v, inp.g, inp.beta, cache, inp.batch_indices,
                          scale=inp.scale, use_qk_l2norm_in_kernel=inp.use_qk_l2norm)
    tol = TOL[inp.q.dtype]
    n = inp.q.shape[0]
    slots = list(range(n)) if inp.batch_indices is None else inp.batch_indices.tolist()
    real = [i for i in range(n) if slots[i] >= 0]
    pad = [i for i in range(n) if slots[i] < 0]
    # o on real requests, and the written slots
    e_o = rel_l2(f64(o[real]), o_ref[real])
    used = sorted(slots[i] for i in real)
    e_s = rel_l2(f64(state_gpu[used]), cache[used])
    print("%s: rel-L2 o=%.3e state=%.3e (tol %.1e)" % (label, e_o, e_s, tol))
    assert e_o <= tol and e_s <= tol
    # each request's new state is in its own slot: compare per request
    for i in real[:: max(1, len(real) // 16)]:
        assert rel_l2(f64(state_gpu[slots[i]]), cache[slots[i]]) <= tol
    # padding rows are exactly +0.0 (bit pattern zero)
    if pad:
        bits = o[pad].contiguous().view(torch.int16 if o.dtype == torch.bfloat16 else torch.int32)
        assert torch.count_nonzero(bits).item() == 0
    # slots not named by any request are byte-identical (the canaries of the cache: every
    # neighbour of a written slot that no request names)
    untouched = sorted(set(range(state_gpu.shape[0])) - set(used))
    if untouched:
        assert torch.equal(state_gpu[untouched].view(torch.int32),
                           before[untouched].view(torch.int32))
    return o, state_gpu


def test_decode_workload_full_size():
    """256 requests (26 padding) on the 512-slot, 1 GiB fp32 cache, bf16 I/O."""
    inp = synthetic.workload("decode_bf16")
    assert int((inp.batch_indices < 0).sum()) == 26
    run_case(inp, "decode_bf16 full")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("KV", [(128, 128), (64, 64), (64, 128), (32, 16), (96, 96), (128, 32)])
def test_decode_shapes(dtype, KV):
    K, V = KV
    inp = synthetic.decode_inputs(n=37, Hqk=2, Hv=4, K=K, V=V, dtype=dtype, num_slots=50,
                                  pad_frac=0.2, seed=7 + K + V)
    run_case(inp, "decode %s K=%d V=%d" % (dtype, K, V))


def test_decode_identity_indices_and_options():
    inp = synthetic.decode_inputs(n=16, Hqk=4, Hv=4, K=128, V=128, dtype=torch.bfloat16,
                                  num_slots=20, identity=True, seed=3, use_qk_l2norm=False,
                                  scale=0.37, beta_dtype=torch.float32)
    run_case(inp, "decode identity/no-l2/fp32-beta")


def test_decode_bad_slot_is_skipped_and_reported():
    inp = synthetic.decode_inputs(n=8, Hqk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16,
                                  num_slots=10, pad_frac=0.0, seed=5)
    inp.batch_indices[3] = 10       # == num_slots: out of range
    inp.batch_indices[5] = -7       # below -1
    dev = "cuda"
    state = inp.ssm_state.to(dev)
    before = state.clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o = gated_delta_decode(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.g.to(dev),
                           inp.beta.to(dev), state, inp.batch_indices.to(dev),
                           dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & GDN_DEV_BAD_SLOT
    assert torch.count_nonzero(o[[3, 5]].float()).item() == 0
    named = set(int(x) for x in inp.batch_indices.tolist() if 0 <= x < 10)
    for s in range(10):
        if s not in named:
            assert torch.equal(state[s], before[s])


def test_decode_continues_a_prefill_state():
    """Decode steps fed from a cached state reproduce the oracle's token-by-token run."""
    torch.manual_seed(0)
    n_steps, Hqk, Hv, K, V = 5, 2, 4, 128, 128
    cache = 0.1 * torch.randn(3, Hv, K, V)
    dev = "cuda"
    c_gpu = cache.to(dev)
    c_ref = f64(cache).copy()
    idx = torch.tensor([2], dtype=torch.int32)
    for t in range(n_steps):
        q = torch.randn(1, Hqk, K).bfloat16(); k = torch.randn(1, Hqk, K).bfloat16()
        v = torch.randn(1, Hv, V).bfloat16()
        g = -torch.nn.functional.softplus(torch.randn(1, Hv))
        b = torch.sigmoid(torch.randn(1, Hv)).bfloat16()
        o = gated_delta_decode(q.to(dev), k.to(dev), v.to(dev), g.to(dev), b.to(dev), c_gpu,
                               idx.to(dev))
        o_ref = oracle.decode(q, k, v, g, b, c_ref, idx)
        assert rel_l2(f64(o), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(f64(c_gpu), c_ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype,KV", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_multi_token_decode_with_intermediate_states(dtype, KV):
    """L tokens per request on the slot cache: outputs, the final slot state and the
    state after every token match the oracle applied token by token."""
    from chunked_gated_delta_gdn_gb300 import gated_delta_decode_multi
    n, L, Hqk, Hv, slots = 12, 5, 2, 4, 20
    gen = torch.Generator().manual_seed(71)
    q = torch.randn(n, L, Hqk, KV, generator=gen).to(dtype)
    k = torch.randn(n, L, Hqk, KV, generator=gen).to(dtype)
    v = torch.randn(n, L, Hv, KV, generator=gen).to(dtype)
    g = -torch.nn.functional.softplus(torch.randn(n, L, Hv, generator=gen))
    beta = torch.sigmoid(torch.randn(n, L, Hv, generator=gen)).to(dtype)
    cache = 0.1 * torch.randn(slots, Hv, KV, KV, generator=gen)
    idx = torch.randperm(slots, generator=gen)[:n].to(torch.int32)
    idx[4] = -1
    dev = "cuda"
    state = cache.to(dev)
    before = state.clone()
    o, inter = gated_delta_decode_multi(q.to(dev), k.to(dev), v.to(dev), g.to(dev), beta.to(dev),
                                        state, idx.to(dev), output_intermediate_states=True)
    torch.cuda.synchronize()
    ref_cache = f64(cache).copy()
    o_ref = np.zeros((n, L, Hv, KV))
    inter_ref = np.zeros((n, L, Hv, KV, KV))
    for t in range(L):
        o_ref[:, t] = oracle.decode(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], ref_cache, idx)
        for i in range(n):
            if idx[i] >= 0:
                inter_ref[i, t] = ref_cache[idx[i]]
    real = [i for i in range(n) if idx[i] >= 0]
    tol = TOL[dtype]
    e_o = rel_l2(f64(o[real]), o_ref[real])
    e_s = rel_l2(f64(state), ref_cache)
    e_i = rel_l2(f64(inter[real]), inter_ref[real])
    print("multi-token decode %s: o %.3e state %.3e intermediates %.3e" % (dtype, e_o, e_s, e_i))
    assert e_o <= tol and e_s <= tol and e_i <= tol
    assert torch.count_nonzero(o[4].float()).item() == 0
    assert torch.equal(inter[real, L - 1], state[idx[real].long()])
    untouched = sorted(set(range(slots)) - set(int(x) for x in idx if x >= 0))
    assert torch.equal(state[untouched], before[untouched])
    # L = 1 is exactly the single-token entry point
    s1, s2 = before.clone(), before.clone()
    o1, _ = gated_delta_decode_multi(q[:, :1].contiguous().to(dev), k[:, :1].contiguous().to(dev),
                                     v[:, :1].contiguous().to(dev), g[:, :1].contiguous().to(dev),
                                     beta[:, :1].contiguous().to(dev), s1, idx.to(dev))
    o2 = gated_delta_decode(q[:, 0].contiguous().to(dev), k[:, 0].contiguous().to(dev),
                            v[:, 0].contiguous().to(dev), g[:, 0].contiguous().to(dev),
                            beta[:, 0].contiguous().to(dev), s2, idx.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(o1[:, 0], o2) and torch.equal(s1, s2)
