"""CUDA-graph capture of the two entry points.  Decode and packed-varlen prefill
must be replayable from a captured graph with new device-side indices: no host
synchronisation and no data-dependent shapes ("Megatron-Core API:
core.ssm.gated_delta_product", GatedDeltaProductMixer.ssm_decode / ssm_prefill).
Each test captures once, rewrites the index tensors in place, replays, and
compares with an eager call on the same inputs (bitwise: same kernels, same
arguments)."""
import pytest
import torch

from chunked_gated_delta_gdn_gb300 import chunk_gated_delta_rule, gated_delta_decode, synthetic

pytestmark = pytest.mark.gpu


def test_decode_graph_replay_with_new_batch_indices():
    dev = torch.device("cuda")
    inp = synthetic.decode_inputs(n=64, Hqk=16, Hv=32, K=128, V=128, dtype=torch.bfloat16,
                                  num_slots=96, pad_frac=0.1, seed=91)
    q, k, v, g, b = (getattr(inp, x).to(dev) for x in ("q", "k", "v", "g", "beta"))
    cache0 = inp.ssm_state.to(dev)
    idx = inp.batch_indices.to(dev)
    state = cache0.clone()
    out = torch.empty_like(v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gated_delta_decode(q, k, v, g, b, state, idx, out=out)      # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gated_delta_decode(q, k, v, g, b, state, idx, out=out)
    for trial in range(2):
        gen = torch.Generator().manual_seed(500 + trial)
        new_idx = torch.randperm(96, generator=gen)[:64].to(torch.int32)
        new_idx[torch.randperm(64, generator=gen)[:7]] = -1
        idx.copy_(new_idx.to(dev))
        state.copy_(cache0)
        graph.replay()
        torch.cuda.synchronize()
        ref_state = cache0.clone()
        ref = gated_delta_decode(q, k, v, g, b, ref_state, idx.clone())
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert torch.equal(state, ref_state)
        pad = (new_idx < 0).nonzero().flatten().tolist()
        assert torch.count_nonzero(out[pad].float()).item() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_varlen_prefill_graph_replay_with_new_cu_seqlens(dtype):
    """The same packed token count, re-split into different sequences and slots
    between replays."""
    dev = torch.device("cuda")
    K = V = 128 if dtype == torch.bfloat16 else 64
    lengths = [300, 17, 64, 500, 0, 143]
    inp = synthetic.chunk_inputs(lengths=lengths, Hqk=2, Hv=4, K=K, V=V, dtype=dtype,
                                 init="slots", num_slots=10, seed=92)
    q, k, v, g, b = (getattr(inp, x).to(dev) for x in ("q", "k", "v", "g", "beta"))
    cache0 = inp.initial_state.to(dev)
    cu = inp.cu_seqlens.to(dev)
    slots = inp.state_indices.to(dev)
    cache = cache0.clone()
    out = torch.empty_like(v)
    T = q.shape[1]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    kw = dict(initial_state=cache, output_final_state=True, use_qk_l2norm_in_kernel=True,
              cu_seqlens=cu, state_indices=slots, out=out)
    with torch.cuda.stream(s):
        chunk_gated_delta_rule(q, k, v, g, b, **kw)               # warm-up (and workspace)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chunk_gated_delta_rule(q, k, v, g, b, **kw)
    for trial, new_lengths in enumerate([[100, 100, 400, 200, 124, 100], [0, 1, 63, 65, 895, 0]]):
        assert sum(new_lengths) == T
        new_cu = torch.zeros(len(new_lengths) + 1, dtype=torch.int32)
        new_cu[1:] = torch.cumsum(torch.tensor(new_lengths), 0).to(torch.int32)
        cu.copy_(new_cu.to(dev))
        new_slots = torch.randperm(10, generator=torch.Generator().manual_seed(600 + trial))[:6]
        new_slots[2] = -1
        slots.copy_(new_slots.to(torch.int32).to(dev))
        cache.copy_(cache0)
        out.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        ref_cache = cache0.clone()
        ref_o, _ = chunk_gated_delta_rule(q, k, v, g, b, initial_state=ref_cache,
                                          output_final_state=True, use_qk_l2norm_in_kernel=True,
                                          cu_seqlens=cu.clone(), state_indices=slots.clone())
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o)
        assert torch.equal(cache, ref_cache)
