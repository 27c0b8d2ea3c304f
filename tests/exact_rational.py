"""Exact rational brute force of the gated delta rule (test helper, pure Python).

Runs the recurrence in ``fractions.Fraction`` so the result carries no rounding
at all.  Decays are given directly as rationals a_t = exp(g_t) (a_t = 0 is a
full reset), L2 normalisation is not applied (callers pass keys that are already
unit-norm or switch the norm off), and value head h reads query/key head
h // (Hv // Hqk).  Used only to pin the fp64 oracle.
"""
from fractions import Fraction


def _matT_vec(S, x, K, V):
    return [sum(S[i][j] * x[i] for i in range(K)) for j in range(V)]


def run(q, k, v, a, beta, cu_seqlens, Hqk, Hv, scale, initial_state=None):
    """q, k: [T][Hqk][K]; v: [T][Hv][V]; a, beta: [T][Hv] (Fractions or ints).

    Returns (o [T][Hv][V], final [N][Hv][K][V]) as Fractions.
    """
    T = len(q)
    K = len(q[0][0])
    V = len(v[0][0])
    N = len(cu_seqlens) - 1
    grp = Hv // Hqk
    o = [[[Fraction(0)] * V for _ in range(Hv)] for _ in range(T)]
    final = []
    for n in range(N):
        per_head = []
        for h in range(Hv):
            if initial_state is None:
                S = [[Fraction(0)] * V for _ in range(K)]
            else:
                S = [[Fraction(x) for x in row] for row in initial_state[n][h]]
            hq = h // grp
            for t in range(cu_seqlens[n], cu_seqlens[n + 1]):
                at = Fraction(a[t][h])
                bt = Fraction(beta[t][h])
                kt = [Fraction(x) for x in k[t][hq]]
                qt = [Fraction(x) for x in q[t][hq]]
                vt = [Fraction(x) for x in v[t][h]]
                S = [[at * S[i][j] for j in range(V)] for i in range(K)]
                r = _matT_vec(S, kt, K, V)
                u = [bt * (vt[j] - r[j]) for j in range(V)]
                S = [[S[i][j] + kt[i] * u[j] for j in range(V)] for i in range(K)]
                ot = _matT_vec(S, qt, K, V)
                o[t][h] = [Fraction(scale) * x for x in ot]
            per_head.append(S)
        final.append(per_head)
    return o, final


def run_product(q, k, v, a, beta, cu_seqlens, Hqk, Hv, scale, initial_state=None):
    """Gated Delta Product in exact arithmetic: per token the decay a_t once, then the writes
    j = 0..n_h-1 with k[t][j], v[t][j], beta[t][j], then o_t = scale S^T q_t.
    q: [T][Hqk][K]; k: [T][n_h][Hqk][K]; v: [T][n_h][Hv][V]; a: [T][Hv]; beta: [T][n_h][Hv]."""
    T = len(q)
    K = len(q[0][0])
    V = len(v[0][0][0])
    n_h = len(k[0])
    N = len(cu_seqlens) - 1
    grp = Hv // Hqk
    o = [[[Fraction(0)] * V for _ in range(Hv)] for _ in range(T)]
    final = []
    for n in range(N):
        per_head = []
        for h in range(Hv):
            if initial_state is None:
                S = [[Fraction(0)] * V for _ in range(K)]
            else:
                S = [[Fraction(x) for x in row] for row in initial_state[n][h]]
            hq = h // grp
            for t in range(cu_seqlens[n], cu_seqlens[n + 1]):
                at = Fraction(a[t][h])
                S = [[at * S[i][j] for j in range(V)] for i in range(K)]
                for w in range(n_h):
                    kt = [Fraction(x) for x in k[t][w][hq]]
                    vt = [Fraction(x) for x in v[t][w][h]]
                    bt = Fraction(beta[t][w][h])
                    r = _matT_vec(S, kt, K, V)
                    u = [bt * (vt[j] - r[j]) for j in range(V)]
                    S = [[S[i][j] + kt[i] * u[j] for j in range(V)] for i in range(K)]
                qt = [Fraction(x) for x in q[t][hq]]
                ot = _matT_vec(S, qt, K, V)
                o[t][h] = [Fraction(scale) * x for x in ot]
            per_head.append(S)
        final.append(per_head)
    return o, final
