"""Stage budgets of the tensor-core backward's reverse and grad passes, from stage timestamps.

    python -m chunked_gated_delta_gdn_gb300.microbench.backward_stage_budget [--B 4] [--T 8192]

Builds the ``stamps`` variant of the library (the same sources with -DGDN_CHUNK_STAMPS), runs
gdn_chunk_bwd on the long-context shape at a smaller length through it, and prints:

- the reverse pass's per-chunk budget: thread 0 of the first eight CTAs (one per (sequence,
  value head)) records clock64 at every stage boundary of iterations 32 .. 95; the table gives
  the median cycles of each stage over those 512 chunks, and the period (loop top to loop top);
- the grad pass's budget per value head: its issuing thread (warp 8) in CTAs 4000 .. 4007 (one
  per (chunk, query/key head), taking its two value heads in turn) records the same for each head
  and for the epilogue; the table gives the median over the eight CTAs.

The recording thread issues the MMAs and the bulk copies (thread 0 in the reverse pass, the
issuer warp in the grad pass), so an "issue" row is the time it spends issuing (blocked at about
the tensor pipe's rate) while the other warps run the work named in the row; a stage done by the
other warps alone shows as the recording thread's wait for it; a "wait" row includes the barrier
that follows it.
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np
import torch

from .. import build, synthetic

REVERSE = [
    "wait: stage landed",
    "partial-chunk clearing",
    "Y, dUp issue (others: q scaling, the next stage's loads)",
    "wait: Y, dUp done",
    "dU' = dUp + Y diag(lambda r_k) -> bf16",
    "dX issue, wait",
    "dX, dv tiles staged, row dots",
    "dS tile staged, dS decayed",
    "bf16 dX operand",
    "stores issued (second thread), row dots out",
    "dS update issue, wait",
    "bf16 copy of dS",
]
GRAD = [
    "wait: the head's tiles landed",
    "(the issuer passes the norms)",
    "wait: q, k normalised in place (first head); partial-chunk clearing",
    "R1, R2 (R3) issue (warps 0-7: <S0, dS>)",
    "gamma, lambda factors",
    "wait: R1-R3 done",
    "row dots",
    "wait: R4's first operand built in TMEM; the next head's dO, dX, U' and R4 over [S0 | dS] issued (warps 0-7: F, E)",
    "wait: F, E done",
    "the rest of R4 issued (warps 2-3: dG, dbeta, dg)",
    "wait: R4 done",
    "next head's S0, dS issued",
]


def run(B: int, T: int, reps: int = 3):
    path = build.build(variant="stamps")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.gdn_chunk_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, i, vp, i,
                                  vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.gdn_chunk_bwd.restype = i
    lib.gdn_chunk_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    lib.gdn_chunk_bwd_workspace_size.restype = sz
    lib.gdn_bwd_stamps_read.argtypes = [vp, vp]
    lib.gdn_bwd_stamps_read.restype = i
    inp = synthetic.workload("long_context_bf16", B=B, T=T)
    dev = torch.device("cuda", 0)
    d = {k: getattr(inp, k).to(dev) for k in ("q", "k", "v", "g", "beta")}
    init = inp.initial_state.to(dev) if inp.initial_state is not None else None
    Hqk, K = inp.q.shape[2:]
    Hv, V = inp.v.shape[2:]
    stream = torch.cuda.current_stream(dev).cuda_stream
    d_o = torch.randn_like(d["v"], dtype=torch.float32).to(d["v"].dtype)
    grads = [torch.empty_like(d[x]) for x in ("q", "k", "v")]
    dg = torch.empty(B, T, Hv, device=dev)
    db = torch.empty(B, T, Hv, device=dev)
    need = lib.gdn_chunk_bwd_workspace_size(B, T, Hqk, Hv, K, V, B, 1, 1)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    for _ in range(reps):
        st = lib.gdn_chunk_bwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                               d["g"].data_ptr(), d["beta"].data_ptr(), B, T, Hqk, Hv, K, V, 1, 1,
                               float("nan"), 64, None if init is None else init.data_ptr(), 1, None,
                               B, d_o.data_ptr(), None, grads[0].data_ptr(), grads[1].data_ptr(),
                               grads[2].data_ptr(), dg.data_ptr(), db.data_ptr(), None,
                               ws.data_ptr(), need, None, stream)
        assert st == 0, st
    torch.cuda.synchronize(dev)
    rev = np.zeros((8, 64, 16), dtype=np.uint64)
    grad = np.zeros((8, 2, 16), dtype=np.uint64)
    assert lib.gdn_bwd_stamps_read(ctypes.c_void_p(rev.ctypes.data), ctypes.c_void_p(grad.ctypes.data)) == 0
    return rev.astype(np.int64), grad.astype(np.int64), Hqk


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--T", type=int, default=8192)
    args = ap.parse_args()
    assert args.T >= 96 * 64, "the reverse pass's stamps cover iterations 32 .. 95"
    rev, grad, Hqk = run(args.B, args.T)
    assert (args.B * args.T) // 64 * Hqk >= 4008, "the grad pass's stamps read CTAs 4000 .. 4007"

    print("\n### reverse pass (B=%d, T=%d): iterations 32-95 of 8 CTAs, median cycles\n" % (args.B, args.T))
    print("| stage | cycles |\n|---|---|")
    for p, name in enumerate(REVERSE, start=1):
        print("| %s | %d |" % (name, int(np.median(rev[:, :, p] - rev[:, :, p - 1]))))
    print("| loop | %d |" % int(np.median(rev[:, 1:, 0] - rev[:, :-1, 12])))
    print("| **period per chunk** | **%d** |" % int(np.median(rev[:, 1:, 0] - rev[:, :-1, 0])))

    print("\n### grad pass (B=%d, T=%d): CTAs 4000-4007, median cycles\n" % (args.B, args.T))
    print("| stage | first value head | second value head |\n|---|---|---|")
    for p, name in enumerate(GRAD, start=1):
        c = [int(np.median(grad[:, h, p] - grad[:, h, p - 1])) for h in range(2)]
        print("| %s | %d | %d |" % (name, c[0], c[1]))
    print("| from the second head's loads issued to its tiles landed | - | %d |"
          % int(np.median(grad[:, 1, 1] - grad[:, 0, 12])))
    print("| epilogue: L2-norm Jacobian, bf16 dq, dk staged | %d | |" % int(np.median(grad[:, 0, 14] - grad[:, 0, 13])))
    print("| **CTA, loads issued to epilogue staged** | **%d** | |" % int(np.median(grad[:, 0, 14] - grad[:, 0, 0])))


if __name__ == "__main__":
    main()
