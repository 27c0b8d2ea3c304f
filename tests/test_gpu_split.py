"""GPU parity of the planned tensor-core launch: sequences split into segments that run
concurrently and are joined through the linearity of the chunk map (transition, contribution,
scan, second pass), against the fp64 oracle.  Covers a split whose last segment ends in a
partial chunk at the sequence end, varlen sequences whose segment boundaries fall inside the
64-token grid of the packed axis (sequences starting at arbitrary offsets), slot caches with
padding and empty sequences, the planned and the unplanned launch of the same inputs, and a
captured graph replayed with other lengths (the plan is rebuilt on the device)."""
import ctypes

import pytest
import torch

from chunked_gated_delta_gdn_gb300 import (_lib, chunk_fwd_path, chunk_gated_delta_rule,
                                           chunk_workspace_size, synthetic)
from tests.parity import TOL, compare_chunk, oracle_chunk, to_dev
from tests.test_gpu_chunk import run_gpu

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def tc_path():
    if chunk_fwd_path(128, 128, BF16) != 1:
        pytest.skip("the tensor-core path does not serve bf16 K = V = 128 here")


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def segments(num_chains):
    """Segments of a split sequence for this many (sequence, head) chains (the library's rule:
    2 s - 3 first-pass units per chain within one CTA per SM, at most 16, none below 3)."""
    s = min((sm_count() // num_chains + 3) // 2, 16)
    return s if s >= 3 else 1


def test_split_single_sequence_ragged_end():
    tc_path()
    s = segments(4)
    T = 64 * 2 * s + 64 * 7 + 29      # at least 2 s chunks; ends 29 tokens into a chunk
    assert s >= 3
    inp = synthetic.chunk_inputs(B=1, T=T, Hqk=2, Hv=4, K=128, V=128, dtype=BF16, init="randn",
                                 seed=301)
    # the plan carries segment matrices (64 KB each) only when the sequence splits
    assert chunk_workspace_size(1, T, 2, 4, 128, 128, 1, BF16) >= 4 * (3 * s - 5) * 65536
    o, fin = run_gpu(inp)
    compare_chunk(inp, o, fin, oracle_chunk(inp), TOL[BF16], "split single T=%d s=%d" % (T, s))


def test_split_varlen_offsets_slots_padding_empty():
    """Two long sequences split (one starting 2137 tokens into the packed axis, so its segment
    boundaries sit 25 tokens into the 64-token grid), a padding slot, an empty sequence."""
    tc_path()
    lengths = [2100, 37, 0, 1950, 300]
    inp = synthetic.chunk_inputs(lengths=lengths, Hqk=2, Hv=4, K=128, V=128, dtype=BF16,
                                 init="slots", num_slots=9, seed=302)
    inp.state_indices = torch.tensor([5, -1, 2, 0, 7], dtype=torch.int32)
    s = segments(len(lengths) * 4)
    assert s >= 3 and (2100 + 63) // 64 >= 2 * s and (1950 + 63) // 64 >= 2 * s
    cache_before = inp.initial_state.clone()
    o, cache = run_gpu(inp)
    compare_chunk(inp, o, cache, oracle_chunk(inp), TOL[BF16], "split varlen s=%d" % s)
    # the empty sequence passes its slot through; unnamed slots are untouched
    assert torch.equal(cache[2].cpu(), cache_before[2])
    for slot in (1, 3, 4, 6, 8):
        assert torch.equal(cache[slot].cpu(), cache_before[slot])


def raw_chunk_fwd(d, inp, workspace, nbytes):
    """gdn_chunk_fwd through the C ABI with an explicit workspace (None: no launch plan)."""
    B, T, Hqk, K = d["q"].shape
    Hv, V = d["v"].shape[2], d["v"].shape[3]
    N = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    o = torch.full((B, T, Hv, V), float("nan"), dtype=BF16, device="cuda")
    fin = torch.full((N, Hv, K, V), float("nan"), device="cuda")
    ptr = lambda x: None if x is None else x.data_ptr()
    st = _lib.load().gdn_chunk_fwd(
        ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]), ptr(d["beta"]), B, T, Hqk, Hv, K, V,
        _lib.GDN_BF16, _lib.GDN_BF16, float("nan"), 64, ptr(d["initial_state"]), 1, ptr(fin),
        1, ptr(d["cu_seqlens"]), N, None, 0, ptr(o), workspace, nbytes, None,
        torch.cuda.current_stream().cuda_stream)
    assert st == _lib.GDN_OK, _lib.status_string(st)
    torch.cuda.synchronize()
    return o, fin


def test_planned_and_unplanned_launch_agree_with_oracle():
    tc_path()
    s = segments(2)
    inp = synthetic.chunk_inputs(B=1, T=64 * (2 * s + 5), Hqk=1, Hv=2, K=128, V=128, dtype=BF16,
                                 init="randn", seed=303)
    d = to_dev(inp)
    ref = oracle_chunk(inp)
    need = chunk_workspace_size(1, inp.q.shape[1], 1, 2, 128, 128, 1, BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o1, f1 = raw_chunk_fwd(d, inp, ws.data_ptr(), need)
    o0, f0 = raw_chunk_fwd(d, inp, None, 0)
    compare_chunk(inp, o1, f1, ref, TOL[BF16], "planned (s=%d)" % s)
    compare_chunk(inp, o0, f0, ref, TOL[BF16], "unplanned")
    # the split changes only the rounding order
    assert (o1.float() - o0.float()).abs().max().item() < 0.1


def test_captured_graph_replans_for_new_lengths():
    tc_path()
    first, second = [2100, 37, 1950], [500, 3000, 587]
    assert sum(first) == sum(second)
    mk = lambda lengths: synthetic.chunk_inputs(lengths=lengths, Hqk=2, Hv=4, K=128, V=128,
                                                dtype=BF16, init="randn", seed=304)
    a, b = mk(first), mk(second)
    d = to_dev(a)
    N, Hv = len(first), 4
    out = torch.full_like(d["v"], float("nan"))
    fin = torch.full((N, Hv, 128, 128), float("nan"), device="cuda")
    need = chunk_workspace_size(1, sum(first), 2, Hv, 128, 128, N, BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    call = lambda: chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=a.scale,
                                          initial_state=d["initial_state"], output_final_state=True,
                                          use_qk_l2norm_in_kernel=True, cu_seqlens=d["cu_seqlens"],
                                          out=out, final_state=fin, workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()   # warm-up outside the capture (loads the library, sets kernel attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for inp in (a, b):
        src = to_dev(inp)
        for key in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens"):
            d[key].copy_(src[key])
        out.fill_(float("nan"))
        fin.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        compare_chunk(inp, out, fin, oracle_chunk(inp), TOL[BF16],
                      "graph replay lengths %s" % (inp.cu_seqlens.diff().tolist(),))
