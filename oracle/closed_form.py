"""Unrolled closed form of the gated delta rule, fp64 numpy -- TEST INFRASTRUCTURE ONLY.

A second, independent statement of the recurrence for tiny shapes.  One token's
update is affine in the state:

    S_t = M_t S_{t-1} + B_t,   M_t = a_t (I - beta_t k_t k_t^T),   B_t = beta_t k_t v_t^T,

with a_t = exp(g_t).  Unrolled from the initial state S_0:

    S_t = (M_t ... M_1) S_0 + sum_{j<=t} (M_t ... M_{j+1}) B_j,    o_t = scale * S_t^T q_t.

Every product below is formed explicitly as a dense K x K matrix (no state is
carried from one step to the next), so the cost is O(T^2 K^3): tiny inputs only.
The method is the gated delta rule of "Megatron-Core API:
core.ssm.gated_delta_net.gdn" (GatedDeltaNet); this file shares no code with the
C oracle or with the CUDA path.
"""
from __future__ import annotations

import math

import numpy as np

L2_EPS = 1e-6


def _l2(x, use):
    if not use:
        return x
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def single_sequence(q, k, v, g, beta, scale=None, initial_state=None, use_qk_l2norm=False):
    """One sequence, one head: q, k [T, K]; v [T, V]; g, beta [T].  Returns (o [T, V], S_T)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, K = q.shape
    V = v.shape[1]
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    qn, kn = _l2(q, use_qk_l2norm), _l2(k, use_qk_l2norm)
    S0 = np.zeros((K, V)) if initial_state is None else np.asarray(initial_state, np.float64)
    eye = np.eye(K)
    M = [np.exp(g[t]) * (eye - beta[t] * np.outer(kn[t], kn[t])) for t in range(T)]
    Bm = [beta[t] * np.outer(kn[t], v[t]) for t in range(T)]

    def prod(hi, lo):
        """M_hi M_{hi-1} ... M_lo (identity when hi < lo), 0-based inclusive."""
        P = eye.copy()
        for t in range(lo, hi + 1):
            P = M[t] @ P
        return P

    o = np.zeros((T, V))
    S = S0
    for t in range(T):
        S = prod(t, 0) @ S0
        for j in range(t + 1):
            S = S + prod(t, j + 1) @ Bm[j]
        o[t] = scale * (S.T @ qn[t])
    return o, S


def batched(q, k, v, g, beta, scale=None, initial_state=None, use_qk_l2norm=False):
    """Batched layout q, k [B, T, Hqk, K]; v [B, T, Hv, V]; g, beta [B, T, Hv].
    Value head h reads query/key head h // (Hv // Hqk)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    grp = Hv // Hqk
    o = np.zeros((B, T, Hv, V))
    fin = np.zeros((B, Hv, K, V))
    for b in range(B):
        for h in range(Hv):
            init = None if initial_state is None else initial_state[b, h]
            o[b, :, h], fin[b, h] = single_sequence(
                q[b, :, h // grp], k[b, :, h // grp], v[b, :, h], g[b, :, h], beta[b, :, h],
                scale=scale, initial_state=init, use_qk_l2norm=use_qk_l2norm)
    return o, fin
