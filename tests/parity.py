"""Helpers for the GPU parity tests: run the fp64 oracle on the same seeded inputs
the CUDA path receives, optionally on a sample of (sequence, value head) pairs,
and compare with relative L2 error."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Bars from the method's stated tolerances: relative L2 error of o and of the
# final state against the fp64 oracle.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def f64(t):
    return t.detach().cpu().double().numpy()


def to_dev(inp, device="cuda"):
    """Copy every tensor field of a ChunkInputs / DecodeInputs to the device."""
    out = {}
    for k, v in vars(inp).items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def seq_bounds(inp):
    B, T = inp.q.shape[:2]
    if inp.cu_seqlens is None:
        return [(b * T, (b + 1) * T) for b in range(B)]
    cu = inp.cu_seqlens.tolist()
    return [(cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def oracle_chunk(inp, pairs=None, nthreads=0, batch=256):
    """Oracle (token-by-token recurrence) outputs for a ChunkInputs.

    pairs: None (all) or a list of (sequence n, value head h).  Returns a dict
    {(n, h): (o [L, V], final [K, V])}; sequences whose slot is -1 map to None
    (padding: zero output, no state).  The requested pairs are packed as
    independent one-head sequences so one oracle call runs them in parallel.
    """
    B, T, Hqk, K = inp.q.shape
    Hv, V = inp.v.shape[2], inp.v.shape[3]
    grp = Hv // Hqk
    flat = lambda x: x.reshape((B * T,) + tuple(x.shape[2:]))
    q, k, v, g, beta = (flat(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    bounds = seq_bounds(inp)
    if pairs is None:
        pairs = [(n, h) for n in range(len(bounds)) for h in range(Hv)]
    res = {}
    todo = []
    for n, h in pairs:
        slot = n
        if inp.state_indices is not None:
            slot = int(inp.state_indices[n])
            if slot < 0:
                res[(n, h)] = None
                continue
        todo.append((n, h, slot))
    for i0 in range(0, len(todo), batch):
        part = todo[i0:i0 + batch]
        qs, ks, vs, gs, bs, inits, cu = [], [], [], [], [], [], [0]
        for n, h, slot in part:
            s, e = bounds[n]
            hq = h // grp
            qs.append(q[s:e, hq:hq + 1]); ks.append(k[s:e, hq:hq + 1])
            vs.append(v[s:e, h:h + 1]); gs.append(g[s:e, h:h + 1]); bs.append(beta[s:e, h:h + 1])
            if inp.initial_state is not None:
                inits.append(f64(inp.initial_state[slot, h])[None])
            cu.append(cu[-1] + (e - s))
        cat = lambda xs: f64(torch.cat(xs, 0))[None]
        init = np.stack(inits, 0) if inits else None
        o, fin = oracle.recurrent(cat(qs), cat(ks), cat(vs), cat(gs), cat(bs), scale=inp.scale,
                                  initial_state=init, use_qk_l2norm_in_kernel=inp.use_qk_l2norm,
                                  cu_seqlens=np.array(cu), nthreads=nthreads)
        for j, (n, h, slot) in enumerate(part):
            res[(n, h)] = (o[0, cu[j]:cu[j + 1], 0], fin[j, 0])
    return res


def chunk_rel_l2(x, ref, C=64):
    """Largest relative L2 error over the C-token chunks of a sequence ([L, V] arrays).  A
    fault confined to one chunk (a wrong buffer parity, one bad tile) moves the whole-sequence
    error of a 512-chunk sequence by only about 1/sqrt(512) of its local size; per chunk it
    shows at full size.  Chunks whose reference is exactly zero are compared in absolute terms."""
    worst = 0.0
    for c0 in range(0, len(ref), C):
        r, g = ref[c0:c0 + C], x[c0:c0 + C]
        den = np.linalg.norm(r)
        err = np.linalg.norm(g - r)
        worst = max(worst, err / den if den > 0 else err)
    return worst


def compare_chunk(inp, o_gpu, fin_gpu, ref, tol, label=""):
    """Compare (sequence, head) pairs: relative L2 of o over each whole sequence and over each
    of its 64-token chunks, and of the final state.  fin_gpu indexed by slot or by sequence.
    Returns (max rel-L2 of o, max per-chunk rel-L2 of o, max rel-L2 of the final state)."""
    B, T = inp.q.shape[:2]
    Hv, V = inp.v.shape[2], inp.v.shape[3]
    o_flat = o_gpu.reshape(B * T, Hv, V)
    bounds = seq_bounds(inp)
    worst_o, worst_c, worst_f = 0.0, 0.0, 0.0
    for (n, h), r in ref.items():
        s, e = bounds[n]
        og = f64(o_flat[s:e, h])
        if r is None:   # padding sequence: exact zeros
            assert np.all(og == 0.0), "%s: padding sequence %d has nonzero output" % (label, n)
            continue
        o_ref, f_ref = r
        if e > s:
            assert np.isfinite(og).all(), "%s: sequence %d head %d has unwritten output" % (label, n, h)
            worst_o = max(worst_o, rel_l2(og, o_ref))
            worst_c = max(worst_c, chunk_rel_l2(og, o_ref))
        if fin_gpu is not None:
            slot = n if inp.state_indices is None else int(inp.state_indices[n])
            fg = f64(fin_gpu[slot, h])
            assert np.isfinite(fg).all(), "%s: final state %d head %d unwritten" % (label, n, h)
            worst_f = max(worst_f, rel_l2(fg, f_ref))
    print("%s: max rel-L2 o=%.3e (per 64-token chunk %.3e) final=%.3e (tol %.1e)"
          % (label, worst_o, worst_c, worst_f, tol))
    assert worst_o <= tol, "%s: o rel-L2 %.3e > %.1e" % (label, worst_o, tol)
    assert worst_c <= tol, "%s: per-chunk o rel-L2 %.3e > %.1e" % (label, worst_c, tol)
    assert worst_f <= tol, "%s: final-state rel-L2 %.3e > %.1e" % (label, worst_f, tol)
    return worst_o, worst_c, worst_f
