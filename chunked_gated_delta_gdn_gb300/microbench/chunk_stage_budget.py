"""Per-chunk cycle budget of the fused chunk kernel, from stage timestamps.

    python -m chunked_gated_delta_gdn_gb300.microbench.chunk_stage_budget [--B 4] [--T 8192] [--record]

With --record the kernel runs in record mode, as the first launch of the backward (gdn_chunk_bwd):
the state group then also stages the entry state and U' of every chunk as bf16 tiles for the
backward's later kernels, inside its "S -> bf16" and "U' -> bf16" rows, and waits at the top of
each chunk until the previous chunk's tiles have left shared memory.

Builds the ``stamps`` variant of the library (the same sources with -DGDN_CHUNK_STAMPS: the
leader of each warp group records clock64 at its stage boundaries for chunks 32 .. 95 of the
first and the last CTA), runs the long-context shape at a smaller length through that library's
gdn_chunk_fwd, and prints the median cycles of every stage of the prep group and of the state
group, with the per-chunk period of each.  A "wait" row is time the group's leader spent
blocked on the other group (or on the TMA / tensor pipe), every other row is the group's own
work on the critical path of its chain.  The variant spills a few registers for the stamps, so
its period reads slightly above the production build's.
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np
import torch

from .. import build, synthetic

PREP = ["loop top", "wait: per-token vectors free, TMA stage landed", "D1 issue (8 MMAs)",
        "wait: D1 done, P buffer free", "norms, P, A from D1", "wait: Tw / Tu buffer free",
        "solve T = (I + A)^-1 -> Tw, Tu"]
STATE = ["loop top", "wait: chunk ready (prep)", "U issue (4 MMAs)", "S -> bf16 S^T, decay S",
         "[O1|Y] issue (8 MMAs)", "K~^T build", "wait: [O1|Y] done", "-Y -> bf16",
         "U' issue (4 MMAs)", "wait: U' done", "U' -> bf16", "O2, S^T issue (4 + 4 MMAs)",
         "wait: O2, S^T done", "output epilogue"]


def run(B: int, T: int, reps: int = 3, record: bool = False):
    path = build.build(variant="stamps")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.gdn_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, i, vp,
                                  i, vp, i, vp, i, vp, vp, sz, vp, vp]
    lib.gdn_chunk_fwd.restype = i
    lib.gdn_chunk_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, i, vp, i,
                                  vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.gdn_chunk_bwd.restype = i
    lib.gdn_chunk_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    lib.gdn_chunk_bwd_workspace_size.restype = sz
    lib.gdn_chunk_stamps_read.argtypes = [vp]
    lib.gdn_chunk_stamps_read.restype = i
    inp = synthetic.workload("long_context_bf16", B=B, T=T)
    dev = torch.device("cuda", 0)
    d = {k: getattr(inp, k).to(dev) for k in ("q", "k", "v", "g", "beta")}
    init = inp.initial_state.to(dev) if inp.initial_state is not None else None
    Hqk, K = inp.q.shape[2:]
    Hv, V = inp.v.shape[2:]
    o = torch.empty_like(d["v"])
    fin = torch.empty(B, Hv, K, V, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if record:
        d_o = torch.randn_like(d["v"], dtype=torch.float32).to(d["v"].dtype)
        grads = [torch.empty_like(d[x]) for x in ("q", "k", "v")]
        dg = torch.empty(B, T, Hv, device=dev)
        db = torch.empty(B, T, Hv, device=dev)
        need = lib.gdn_chunk_bwd_workspace_size(B, T, Hqk, Hv, K, V, B, 1, 1)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    for _ in range(reps):
        if record:
            st = lib.gdn_chunk_bwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                   d["g"].data_ptr(), d["beta"].data_ptr(), B, T, Hqk, Hv, K, V, 1,
                                   1, float("nan"), 64, None if init is None else init.data_ptr(),
                                   1, None, B, d_o.data_ptr(), None, grads[0].data_ptr(),
                                   grads[1].data_ptr(), grads[2].data_ptr(), dg.data_ptr(),
                                   db.data_ptr(), None, ws.data_ptr(), need, None, stream)
        else:
            st = lib.gdn_chunk_fwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                   d["g"].data_ptr(), d["beta"].data_ptr(), B, T, Hqk, Hv, K, V, 1,
                                   1, float("nan"), 64, None if init is None else init.data_ptr(), 1,
                                   fin.data_ptr(), 1, None, B, None, 0, o.data_ptr(), None, 0, None,
                                   stream)
        assert st == 0, st
    torch.cuda.synchronize(dev)
    buf = np.zeros((2, 2, 64, 16), dtype=np.uint64)
    assert lib.gdn_chunk_stamps_read(ctypes.c_void_p(buf.ctypes.data)) == 0
    return buf.astype(np.int64)


def budget(st, names):
    """Median cycles of every stage (stamp p-1 -> p) and of the tail (last stamp -> next top)."""
    n = len(names)
    rows = [(names[p], int(np.median(st[:, p] - st[:, p - 1]))) for p in range(1, n)]
    rows.append(("hand-off, loop", int(np.median(st[1:, 0] - st[:-1, n - 1]))))
    period = int(np.median(st[1:, 0] - st[:-1, 0]))
    return rows, period


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--record", action="store_true")
    args = ap.parse_args()
    assert args.T >= 96 * 64, "stamps cover chunks 32 .. 95"
    buf = run(args.B, args.T, record=args.record)
    mode = "record mode (the backward's forward recompute)" if args.record else "forward mode"
    for cta, label in ((0, "first CTA"), (1, "last CTA")):
        print("\n### %s, %s (B=%d, T=%d, chunks 32-95, median cycles)\n" % (mode, label, args.B, args.T))
        for grp, (gname, names) in enumerate((("prep group (warps 0-7)", PREP),
                                              ("state group (warps 8-11)", STATE))):
            rows, period = budget(buf[cta, grp], names)
            print("| %s | cycles |\n|---|---|" % gname)
            for name, cyc in rows:
                print("| %s | %d |" % (name, cyc))
            print("| **period per chunk** | **%d** |\n" % period)


if __name__ == "__main__":
    main()
