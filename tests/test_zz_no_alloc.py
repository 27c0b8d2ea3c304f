"""gdn_chunk_fwd_noalloc: the entry point for callers that cannot allocate device
memory (plugins inside another runtime's memory budget, C callers without an
allocator, code that must not call cudaMalloc mid-step).  It runs the CUDA-core
chunk kernels with their scratch in one static device array instead of a
caller workspace.  Called here through the C ABI and checked against
gdn_chunk_fwd (with a torch-allocated workspace) on two calls in a row, so the
second call also shows that what the first left in the shared array does not
leak into its result.  Collected last: it runs after every other test, and also
passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from chunked_gated_delta_gdn_gb300 import _lib, chunk_gated_delta_rule, synthetic
from tests.parity import TOL, f64, rel_l2

pytestmark = pytest.mark.gpu

NOALLOC_MAX = 64 << 20


def noalloc_fn():
    lib = _lib.load()
    fn = lib.gdn_chunk_fwd_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, i, vp, i, vp, i, vp, i,
                   vp, vp, vp]
    fn.restype = i
    return fn


def call_noalloc(inp, dev):
    B, T, Hqk, K = inp.q.shape
    Hv, V = inp.v.shape[2], inp.v.shape[3]
    d = {k: getattr(inp, k).to(dev) for k in ("q", "k", "v", "g", "beta", "initial_state")}
    o = torch.full((B, T, Hv, V), float("nan"), dtype=inp.q.dtype, device=dev)
    fin = torch.full((B, Hv, K, V), float("nan"), dtype=torch.float32, device=dev)
    io = _lib.GDN_F32 if inp.q.dtype == torch.float32 else _lib.GDN_BF16
    st = noalloc_fn()(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
                      d["beta"].data_ptr(), B, T, Hqk, Hv, K, V, io, io, float("nan"), 64,
                      d["initial_state"].data_ptr(), 1, fin.data_ptr(), 1, None, B, None, 0,
                      o.data_ptr(), None, torch.cuda.current_stream(dev).cuda_stream)
    assert st == _lib.GDN_OK, _lib.status_string(st)
    torch.cuda.synchronize(dev)
    return o, fin


def call_existing(inp, dev):
    d = {k: getattr(inp, k).to(dev) for k in ("q", "k", "v", "g", "beta", "initial_state")}
    o, fin = chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                    initial_state=d["initial_state"], output_final_state=True,
                                    use_qk_l2norm_in_kernel=True)
    torch.cuda.synchronize(dev)
    return o, fin


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = torch.device("cuda", 0)
    # fp32 I/O runs the CUDA-core kernels, the ones that use scratch
    cases = [synthetic.workload("tiny_fp32"),
             synthetic.chunk_inputs(B=2, T=300, Hqk=1, Hv=2, K=64, V=64, dtype=torch.float32,
                                    init="randn", seed=77)]
    outs = [call_noalloc(inp, dev) for inp in cases]      # two no-alloc calls in a row
    for n, (inp, (o1, f1)) in enumerate(zip(cases, outs)):
        o2, f2 = call_existing(inp, dev)
        e_o, e_f = rel_l2(f64(o1), f64(o2)), rel_l2(f64(f1), f64(f2))
        print("no-alloc call %d: rel-L2 vs gdn_chunk_fwd o=%.3e final=%.3e" % (n + 1, e_o, e_f))
        assert np.isfinite(f64(o1)).all() and np.isfinite(f64(f1)).all()
        assert e_o <= TOL[torch.float32] and e_f <= TOL[torch.float32]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib.load()
    need = lib.gdn_chunk_fwd_workspace_size(1, 1 << 16, 4, 8, 128, 128, 1, _lib.GDN_F32,
                                            _lib.GDN_F32)
    assert need > NOALLOC_MAX
    # no tensors at all: a correct build rejects the size first (GDN_ERR_WORKSPACE); if that
    # check ever regressed, the NULL pointers stop the call in host code (GDN_ERR_NULL) before
    # any launch
    st = noalloc_fn()(None, None, None, None, None, 1, 1 << 16, 4, 8, 128, 128, _lib.GDN_F32,
                      _lib.GDN_F32, float("nan"), 64, None, 0, None, 1, None, 1, None, 0, None,
                      None, None)
    assert st == _lib.GDN_ERR_WORKSPACE
