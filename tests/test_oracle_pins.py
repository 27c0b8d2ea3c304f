"""Pins for the fp64 CPU oracle: each test checks the oracle against something
other than itself -- hand-worked values, exact rational brute force, closed
forms, special cases that reduce to textbook results, autograd, and invariants
that any correct evaluation must satisfy.  CPU only.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import closed_form
from tests import exact_rational

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_examples.json")


def rel_err(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def rand_case(rng, B=1, T=37, Hqk=2, Hv=4, K=8, V=6, init=True):
    q = rng.standard_normal((B, T, Hqk, K))
    k = rng.standard_normal((B, T, Hqk, K))
    v = rng.standard_normal((B, T, Hv, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv))))
    s0 = 0.1 * rng.standard_normal((B, Hv, K, V)) if init else None
    return q, k, v, g, beta, s0


# --------------------------------------------------------------------------- golden

def test_hand_worked_prefill():
    ex = json.load(open(GOLDEN))["prefill"]
    T, K, V = len(ex["q"]), ex["K"], ex["V"]
    q = np.array(ex["q"], float).reshape(1, T, 1, K)
    k = np.array(ex["k"], float).reshape(1, T, 1, K)
    v = np.array(ex["v"], float).reshape(1, T, 1, V)
    g = np.log(np.array(ex["a"], float)).reshape(1, T, 1)
    beta = np.array(ex["beta"], float).reshape(1, T, 1)
    s0 = np.array(ex["initial_state"], float).reshape(1, 1, K, V)
    for fn in (oracle.recurrent, lambda *a, **kw: oracle.chunked(*a, chunk_size=2, **kw)):
        o, fin = fn(q, k, v, g, beta, scale=ex["scale"], initial_state=s0,
                    use_qk_l2norm_in_kernel=ex["use_qk_l2norm"])
        np.testing.assert_allclose(o[0, :, 0], ex["expected_o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(fin[0, 0], ex["expected_final_state"], rtol=0, atol=1e-12)


def test_hand_worked_decode():
    ex = json.load(open(GOLDEN))["decode"]
    n = len(ex["q"])
    q = np.array(ex["q"], float).reshape(n, 1, 1)
    k = np.array(ex["k"], float).reshape(n, 1, 1)
    v = np.array(ex["v"], float).reshape(n, 1, 1)
    g = np.log(np.array(ex["a"], float)).reshape(n, 1)
    beta = np.array(ex["beta"], float).reshape(n, 1)
    cache = np.array(ex["initial_cache"], float).reshape(-1, 1, 1, 1).copy()
    o = oracle.decode(q, k, v, g, beta, cache, np.array(ex["batch_indices"]), scale=ex["scale"],
                      use_qk_l2norm_in_kernel=ex["use_qk_l2norm"])
    np.testing.assert_allclose(o.reshape(-1), ex["expected_o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(cache.reshape(-1), ex["expected_cache"], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- exact brute force

DECAYS = [Fraction(1), Fraction(1, 2), Fraction(3, 4), Fraction(0)]
BETAS = [Fraction(0), Fraction(1, 4), Fraction(1, 2), Fraction(1)]


def _exact_case(seed, lengths, Hqk, Hv, K, V, with_init):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q = rng.integers(-3, 4, (T, Hqk, K))
    k = rng.integers(-3, 4, (T, Hqk, K))
    v = rng.integers(-3, 4, (T, Hv, V))
    a = [[DECAYS[x] for x in row] for row in rng.integers(0, 4, (T, Hv))]
    b = [[BETAS[x] for x in row] for row in rng.integers(0, 4, (T, Hv))]
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    N = len(lengths)
    s0 = rng.integers(-2, 3, (N, Hv, K, V)) if with_init else None
    return q, k, v, a, b, cu, s0


@pytest.mark.parametrize("seed", range(6))
def test_exact_rational_brute_force(seed):
    lengths = [5, 7] if seed % 2 else [12]
    Hqk, Hv, K, V = (1, 2, 3, 4) if seed < 3 else (2, 2, 4, 2)
    q, k, v, a, b, cu, s0 = _exact_case(seed, lengths, Hqk, Hv, K, V, with_init=seed % 3 != 0)
    scale = Fraction(1, 2)
    o_ex, fin_ex = exact_rational.run(q.tolist(), k.tolist(), v.tolist(), a, b, cu, Hqk, Hv,
                                      scale, None if s0 is None else s0.tolist())
    with np.errstate(divide="ignore"):
        g = np.log(np.array([[float(x) for x in row] for row in a]))  # a = 0 -> g = -inf
    beta = np.array([[float(x) for x in row] for row in b])
    T = cu[-1]
    o, fin = oracle.recurrent(q.reshape(1, T, Hqk, K), k.reshape(1, T, Hqk, K),
                              v.reshape(1, T, Hv, V), g.reshape(1, T, Hv),
                              beta.reshape(1, T, Hv), scale=0.5, initial_state=s0,
                              use_qk_l2norm_in_kernel=False, cu_seqlens=np.array(cu))
    o_ref = np.array([[[float(x) for x in row] for row in tok] for tok in o_ex])
    fin_ref = np.array([[[[float(x) for x in r] for r in hd] for hd in seq] for seq in fin_ex])
    assert rel_err(o[0], o_ref) < 1e-12
    assert rel_err(fin, fin_ref) < 1e-12
    # decode, token by token, through the same slots
    if len(lengths) == 1 and s0 is not None:
        cache = s0.astype(np.float64).copy()
        outs = []
        for t in range(T):
            outs.append(oracle.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                      beta[t:t + 1], cache, np.array([0]), scale=0.5,
                                      use_qk_l2norm_in_kernel=False)[0])
        assert rel_err(np.stack(outs), o_ref) < 1e-12
        assert rel_err(cache, fin_ref) < 1e-12


def test_exact_rational_unit_keys_with_l2norm():
    """Keys with integer norms: normalised keys are exact rationals (up to eps=1e-6)."""
    vecs = [(3, 4, 0), (1, 2, 2), (2, 3, 6), (0, 0, 1), (1, 4, 8), (4, 4, 7), (2, 6, 9)]
    norms = [5, 3, 7, 1, 9, 9, 11]
    rng = np.random.default_rng(11)
    T, K, V = 9, 3, 2
    ki = rng.integers(0, len(vecs), T)
    qi = rng.integers(0, len(vecs), T)
    kk = [[[Fraction(x, norms[i]) for x in vecs[i]]] for i in ki]
    qq = [[[Fraction(x, norms[i]) for x in vecs[i]]] for i in qi]
    vv = rng.integers(-4, 5, (T, 1, V))
    a = [[DECAYS[x]] for x in rng.integers(0, 3, T)]
    b = [[BETAS[x]] for x in rng.integers(1, 4, T)]
    o_ex, fin_ex = exact_rational.run(qq, kk, vv.tolist(), a, b, [0, T], 1, 1, Fraction(1))
    # oracle sees the raw (unnormalised) integer vectors and normalises them itself
    # a positive multiple of a raw query normalises to the same q-hat
    q = np.array([[vecs[i]] for i in qi], float).reshape(1, T, 1, K) * 2.5
    k = np.array([[vecs[i]] for i in ki], float).reshape(1, T, 1, K)
    with np.errstate(divide="ignore"):
        g = np.log(np.array([[float(x[0])] for x in a])).reshape(1, T, 1)
    beta = np.array([[float(x[0])] for x in b]).reshape(1, T, 1)
    o, fin = oracle.recurrent(q, k, vv.reshape(1, T, 1, V).astype(float), g, beta, scale=1.0,
                              use_qk_l2norm_in_kernel=True)
    o_ref = np.array([[float(x) for x in tok[0]] for tok in o_ex])
    assert rel_err(o[0, :, 0], o_ref) < 1e-6   # eps = 1e-6 inside the square root
    assert rel_err(fin[0, 0], np.array([[float(x) for x in r] for r in fin_ex[0][0]])) < 1e-6


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("l2", [False, True])
def test_unrolled_closed_form(l2):
    rng = np.random.default_rng(3)
    q, k, v, g, beta, s0 = rand_case(rng, B=2, T=9, Hqk=1, Hv=2, K=4, V=3)
    o, fin = oracle.recurrent(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=l2)
    o2, fin2 = closed_form.batched(q, k, v, g, beta, initial_state=s0, use_qk_l2norm=l2)
    assert rel_err(o, o2) < 1e-12
    assert rel_err(fin, fin2) < 1e-12


def test_delta_rule_is_a_gradient_step():
    """S_t = X - beta * grad_X 1/2 ||X^T k - v||^2 at X = a S_{t-1} (torch autograd)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    K, V = 5, 4
    S0 = rng.standard_normal((K, V))
    k = rng.standard_normal(K)
    k = k / np.sqrt(np.sum(k * k) + 1e-6)   # oracle with l2norm on sees the raw key
    kraw = k * 2.5
    v = rng.standard_normal(V)
    q = rng.standard_normal(K)
    a, b = 0.7, 0.3
    X = torch.tensor(a * S0, requires_grad=True)
    loss = 0.5 * torch.sum((X.T @ torch.tensor(k) - torch.tensor(v)) ** 2)
    loss.backward()
    S1 = (X - b * X.grad).detach().numpy()
    cache = S0.reshape(1, 1, K, V).copy()
    qn = q / np.sqrt(np.sum(q * q) + 1e-6)
    o = oracle.decode(q.reshape(1, 1, K), kraw.reshape(1, 1, K), v.reshape(1, 1, V),
                      np.array([[math.log(a)]]), np.array([[b]]), cache, None, scale=1.0,
                      use_qk_l2norm_in_kernel=True)
    # k-hat of the raw key differs from k only through eps: tolerance 1e-7
    assert rel_err(cache[0, 0], S1) < 1e-7
    assert rel_err(o[0, 0], S1.T @ qn) < 1e-7


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(7)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=20, Hqk=2, Hv=2, K=5, V=3)
    beta[:] = 0.0
    o, fin = oracle.recurrent(q, k, v, g, beta, scale=0.5, initial_state=s0,
                              use_qk_l2norm_in_kernel=False)
    G = np.cumsum(g[0], axis=0)                   # [T, Hv]
    for h in range(2):
        for t in range(20):
            exp_o = 0.5 * math.exp(G[t, h]) * (s0[0, h].T @ q[0, t, h])
            np.testing.assert_allclose(o[0, t, h], exp_o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(fin[0, h], math.exp(G[-1, h]) * s0[0, h], rtol=1e-12)


def test_zero_decay_resets_state():
    """a_t = 0 (g = -inf): S_t = beta k v^T, o_t = scale beta (q.k) v."""
    rng = np.random.default_rng(8)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=6, Hqk=1, Hv=1, K=4, V=3)
    g[:] = -np.inf
    o, fin = oracle.recurrent(q, k, v, g, beta, scale=1.0, initial_state=s0,
                              use_qk_l2norm_in_kernel=False)
    for t in range(6):
        exp_o = beta[0, t, 0] * float(q[0, t, 0] @ k[0, t, 0]) * v[0, t, 0]
        np.testing.assert_allclose(o[0, t, 0], exp_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], beta[0, -1, 0] * np.outer(k[0, -1, 0], v[0, -1, 0]),
                               rtol=1e-12, atol=1e-14)


def test_orthonormal_keys_store_and_retrieve():
    """g = 0, beta = 1, orthonormal keys: writing v_j under k_j, then querying k_j returns v_j."""
    rng = np.random.default_rng(9)
    K, V = 6, 4
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm.T                                   # rows orthonormal
    vals = rng.standard_normal((K, V))
    T = 2 * K
    k = np.zeros((1, T, 1, K)); q = np.zeros((1, T, 1, K)); v = np.zeros((1, T, 1, V))
    g = np.zeros((1, T, 1)); beta = np.zeros((1, T, 1))
    for j in range(K):                            # write phase
        k[0, j, 0] = keys[j]; q[0, j, 0] = keys[j]; v[0, j, 0] = vals[j]; beta[0, j, 0] = 1.0
    for j in range(K):                            # read phase: beta = 0 leaves S unchanged
        k[0, K + j, 0] = keys[j]; q[0, K + j, 0] = keys[j]
    o, fin = oracle.recurrent(q, k, v, g, beta, scale=1.0, use_qk_l2norm_in_kernel=False)
    np.testing.assert_allclose(o[0, K:, 0], vals, rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0], keys.T @ vals, rtol=0, atol=1e-12)


def test_scalar_state_closed_form():
    """K = V = 1: s_t = c_t s_{t-1} + d_t with c = a (1 - beta k^2), d = beta k v, so
    s_T = (prod c) s_0 + sum_j (prod_{m>j} c_m) d_j."""
    rng = np.random.default_rng(10)
    T = 15
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=T, Hqk=1, Hv=1, K=1, V=1)
    o, fin = oracle.recurrent(q, k, v, g, beta, scale=1.0, initial_state=s0,
                              use_qk_l2norm_in_kernel=False)
    a = np.exp(g[0, :, 0]); kk = k[0, :, 0, 0]; vv = v[0, :, 0, 0]; bb = beta[0, :, 0]
    c = a * (1 - bb * kk * kk)
    d = bb * kk * vv
    for t in range(T):
        s = np.prod(c[:t + 1]) * s0[0, 0, 0, 0] + sum(np.prod(c[j + 1:t + 1]) * d[j]
                                                      for j in range(t + 1))
        np.testing.assert_allclose(o[0, t, 0, 0], s * q[0, t, 0, 0], rtol=1e-11, atol=1e-13)


def test_delta_interpolation_property():
    """With unit keys: S_t^T k_t = (1 - beta_t) (a_t S_{t-1})^T k_t + beta_t v_t."""
    rng = np.random.default_rng(12)
    K, V = 7, 5
    cache = rng.standard_normal((1, 1, K, V))
    for _ in range(5):
        kraw = rng.standard_normal((1, 1, K))
        kn = kraw[0, 0] / np.sqrt(np.sum(kraw * kraw) + 1e-6)
        v = rng.standard_normal((1, 1, V))
        a, b = float(rng.uniform(0.2, 1.0)), float(rng.uniform(0.0, 1.0))
        before = a * cache[0, 0].T @ kn
        oracle.decode(kraw, kraw, v, np.array([[math.log(a)]]), np.array([[b]]), cache, None,
                      use_qk_l2norm_in_kernel=True)
        after = cache[0, 0].T @ kn
        knorm2 = float(kn @ kn)                   # 1 - O(eps)
        np.testing.assert_allclose(after, before + b * knorm2 * (v[0, 0] - before), rtol=1e-12,
                                   atol=1e-12)
        np.testing.assert_allclose(after, (1 - b) * before + b * v[0, 0], rtol=1e-6, atol=1e-6)


def test_l2norm_and_default_scale():
    """One token from a zero state with beta = 1, g = 0: o = (1/sqrt(K)) (q-hat . k-hat) v."""
    rng = np.random.default_rng(13)
    K, V = 16, 3
    q = rng.standard_normal((1, 1, 1, K)) * 3
    k = rng.standard_normal((1, 1, 1, K)) * 0.5
    v = rng.standard_normal((1, 1, 1, V))
    o, _ = oracle.recurrent(q, k, v, np.zeros((1, 1, 1)), np.ones((1, 1, 1)),
                            use_qk_l2norm_in_kernel=True)
    qh = q.ravel() / np.sqrt(np.sum(q ** 2) + 1e-6)
    kh = k.ravel() / np.sqrt(np.sum(k ** 2) + 1e-6)
    np.testing.assert_allclose(o.ravel(), (qh @ kh) / math.sqrt(K) * v.ravel(), rtol=1e-13)
    # without the norm: plain dot product
    o2, _ = oracle.recurrent(q, k, v, np.zeros((1, 1, 1)), np.ones((1, 1, 1)), scale=2.0)
    np.testing.assert_allclose(o2.ravel(), 2.0 * float(q.ravel() @ k.ravel()) * v.ravel(),
                               rtol=1e-13)


# --------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("C", [1, 2, 3, 5, 16, 63, 64, 65, 100, 1000])
def test_chunked_equals_recurrent(C):
    rng = np.random.default_rng(100 + C)
    lengths = [100, 1, 64, 65, 0, 37]
    T = sum(lengths)
    q, k, v, g, beta, _ = rand_case(rng, B=1, T=T, Hqk=2, Hv=4, K=8, V=6, init=False)
    s0 = 0.1 * rng.standard_normal((len(lengths), 4, 8, 6))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    for l2 in (False, True):
        o1, f1 = oracle.recurrent(q, k, v, g, beta, initial_state=s0, cu_seqlens=cu,
                                  use_qk_l2norm_in_kernel=l2)
        o2, f2 = oracle.chunked(q, k, v, g, beta, chunk_size=C, initial_state=s0, cu_seqlens=cu,
                                use_qk_l2norm_in_kernel=l2)
        assert rel_err(o2, o1) < 1e-11
        assert rel_err(f2, f1) < 1e-11


def test_chunked_strong_decay_stays_finite():
    """Log-decays summing to about -5000 inside one chunk: only differences G_i - G_j
    are exponentiated, so nothing overflows."""
    rng = np.random.default_rng(21)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=130, Hqk=1, Hv=1, K=8, V=8)
    g[:] = -80.0 * rng.uniform(0.2, 1.0, g.shape)
    o1, f1 = oracle.recurrent(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True)
    o2, f2 = oracle.chunked(q, k, v, g, beta, chunk_size=64, initial_state=s0,
                            use_qk_l2norm_in_kernel=True)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(f2))
    assert rel_err(o2, o1) < 1e-12 and rel_err(f2, f1) < 1e-12


@pytest.mark.parametrize("split", [1, 17, 64, 99])
def test_prefill_then_decode_equals_whole(split):
    """State continuity: prefill of [0, t) then token-by-token decode of [t, L) equals
    prefill of [0, L), for every output and for the final state."""
    rng = np.random.default_rng(200 + split)
    L = 100
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=L, Hqk=2, Hv=4, K=8, V=6)
    o_all, f_all = oracle.chunked(q, k, v, g, beta, initial_state=s0, chunk_size=64,
                                  use_qk_l2norm_in_kernel=True)
    o_pre, f_pre = oracle.chunked(q[:, :split], k[:, :split], v[:, :split], g[:, :split],
                                  beta[:, :split], initial_state=s0, chunk_size=64,
                                  use_qk_l2norm_in_kernel=True)
    cache = np.concatenate([np.zeros_like(f_pre), f_pre], axis=0)   # slot 1 holds the state
    outs = [o_pre[0]]
    for t in range(split, L):
        outs.append(oracle.decode(q[0, t:t + 1], k[0, t:t + 1], v[0, t:t + 1], g[0, t:t + 1],
                                  beta[0, t:t + 1], cache, np.array([1])))
    o_cat = np.concatenate(outs, axis=0)
    assert rel_err(o_cat, o_all[0]) < 1e-12
    assert rel_err(cache[1], f_all[0]) < 1e-12
    assert np.all(cache[0] == 0)


def test_split_prefill_equals_whole():
    rng = np.random.default_rng(31)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=150, Hqk=1, Hv=2, K=8, V=8)
    o_all, f_all = oracle.chunked(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True)
    o1, f1 = oracle.chunked(q[:, :70], k[:, :70], v[:, :70], g[:, :70], beta[:, :70],
                            initial_state=s0, use_qk_l2norm_in_kernel=True)
    o2, f2 = oracle.chunked(q[:, 70:], k[:, 70:], v[:, 70:], g[:, 70:], beta[:, 70:],
                            initial_state=f1, use_qk_l2norm_in_kernel=True)
    assert rel_err(np.concatenate([o1, o2], axis=1), o_all) < 1e-12
    assert rel_err(f2, f_all) < 1e-12


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(41)
    lengths = [33, 64, 5, 90]
    T = sum(lengths)
    q, k, v, g, beta, _ = rand_case(rng, B=1, T=T, Hqk=2, Hv=2, K=8, V=4, init=False)
    s0 = rng.standard_normal((4, 2, 8, 4))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, fin = oracle.chunked(q, k, v, g, beta, initial_state=s0, cu_seqlens=cu,
                            use_qk_l2norm_in_kernel=True)
    for n in range(4):
        s, e = cu[n], cu[n + 1]
        o1, f1 = oracle.recurrent(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e],
                                  initial_state=s0[n:n + 1], use_qk_l2norm_in_kernel=True)
        assert rel_err(o[:, s:e], o1) < 1e-12
        assert rel_err(fin[n], f1[0]) < 1e-12


def test_batched_equals_uniform_varlen():
    rng = np.random.default_rng(42)
    q, k, v, g, beta, s0 = rand_case(rng, B=3, T=40, Hqk=1, Hv=2, K=4, V=4)
    o1, f1 = oracle.chunked(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True)
    flat = lambda x: x.reshape((1, 3 * 40) + x.shape[2:])
    o2, f2 = oracle.chunked(flat(q), flat(k), flat(v), flat(g), flat(beta), initial_state=s0,
                            cu_seqlens=np.array([0, 40, 80, 120]), use_qk_l2norm_in_kernel=True)
    assert rel_err(flat(o1), o2) < 1e-14 and rel_err(f1, f2) < 1e-14


def test_grouped_heads_equal_repeated_heads():
    """Value head h reads query/key head h // (Hv / Hqk): identical to repeating each
    query/key head Hv / Hqk times along the head axis."""
    rng = np.random.default_rng(51)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=50, Hqk=2, Hv=6, K=4, V=4)
    o1, f1 = oracle.chunked(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True)
    qr, kr = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    o2, f2 = oracle.recurrent(qr, kr, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True)
    assert rel_err(o1, o2) < 1e-12 and rel_err(f1, f2) < 1e-12


def test_empty_sequences_leave_state():
    rng = np.random.default_rng(52)
    q, k, v, g, beta, _ = rand_case(rng, B=1, T=10, Hqk=1, Hv=1, K=4, V=4, init=False)
    s0 = rng.standard_normal((3, 1, 4, 4))
    cu = np.array([0, 0, 10, 10])
    o, fin = oracle.chunked(q, k, v, g, beta, initial_state=s0, cu_seqlens=cu)
    assert np.array_equal(fin[0], s0[0]) and np.array_equal(fin[2], s0[2])


# --------------------------------------------------------------------------- decode semantics

def test_decode_padding_untouched_and_permutation():
    rng = np.random.default_rng(61)
    n, Hqk, Hv, K, V, S = 12, 2, 4, 8, 6, 20
    q = rng.standard_normal((n, Hqk, K)); k = rng.standard_normal((n, Hqk, K))
    v = rng.standard_normal((n, Hv, V)); g = -np.log1p(np.exp(rng.standard_normal((n, Hv))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((n, Hv))))
    cache0 = rng.standard_normal((S, Hv, K, V))
    idx = rng.permutation(S)[:n]
    idx[[2, 7]] = -1
    cache = cache0.copy()
    o = oracle.decode(q, k, v, g, beta, cache, idx)
    assert np.all(o[[2, 7]] == 0.0)
    used = set(int(x) for x in idx if x >= 0)
    for s in range(S):
        if s not in used:
            assert np.array_equal(cache[s], cache0[s])
    # same requests in another order: outputs permute, the cache ends identical
    perm = rng.permutation(n)
    cache2 = cache0.copy()
    o2 = oracle.decode(q[perm], k[perm], v[perm], g[perm], beta[perm], cache2, idx[perm])
    assert np.array_equal(o2, o[perm])
    assert np.array_equal(cache2, cache)
    # each request equals a one-sequence prefill from its slot
    for i in range(n):
        if idx[i] < 0:
            continue
        oi, fi = oracle.recurrent(q[None, i:i + 1], k[None, i:i + 1], v[None, i:i + 1],
                                  g[None, i:i + 1], beta[None, i:i + 1],
                                  initial_state=cache0[idx[i]][None], use_qk_l2norm_in_kernel=True)
        assert rel_err(o[i], oi[0, 0]) < 1e-13
        assert rel_err(cache[idx[i]], fi[0]) < 1e-13


def test_decode_bad_slot_is_reported_and_skipped():
    rng = np.random.default_rng(62)
    cache = rng.standard_normal((3, 1, 2, 2))
    before = cache.copy()
    args = (rng.standard_normal((2, 1, 2)), rng.standard_normal((2, 1, 2)),
            rng.standard_normal((2, 1, 2)), -np.ones((2, 1)), 0.5 * np.ones((2, 1)))
    with pytest.raises(RuntimeError):
        oracle.decode(*args, cache, np.array([5, 1]))
    o = oracle.decode(*args, before.copy(), np.array([5, 1]), allow_bad_slots=True)
    assert np.all(o[0] == 0)


# --------------------------------------------------------------------------- gate computation

def test_gate_functions_against_textbook_values():
    from oracle import gates
    # softplus: log 2 at 0, identity asymptote, e^x asymptote, symmetry softplus(x) - softplus(-x) = x
    assert gates.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert gates.softplus(40.0) == pytest.approx(40.0, rel=1e-15)
    assert gates.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)
    xs = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(gates.softplus(xs) - gates.softplus(-xs), xs, atol=1e-12)
    np.testing.assert_allclose(gates.softplus(xs), np.log1p(np.exp(xs)), rtol=1e-13)
    # sigmoid: 1/2 at 0, sigmoid(x) + sigmoid(-x) = 1, derivative identity s' = s (1 - s)
    assert gates.sigmoid(0.0) == 0.5
    np.testing.assert_allclose(gates.sigmoid(xs) + gates.sigmoid(-xs), 1.0, atol=1e-15)
    h = 1e-6
    num = (gates.sigmoid(xs + h) - gates.sigmoid(xs - h)) / (2 * h)
    s = gates.sigmoid(xs)
    np.testing.assert_allclose(num, s * (1 - s), atol=1e-9)
    assert gates.sigmoid(800.0) == 1.0 and gates.sigmoid(-800.0) == 0.0


def test_gates_formula_and_ranges():
    from oracle import gates
    rng = np.random.default_rng(14)
    Hv = 6
    A_log = np.log(rng.uniform(1, 16, Hv))
    dt_bias = 0.5 * rng.standard_normal(Hv)
    a = rng.standard_normal((3, 5, Hv))
    b = rng.standard_normal((3, 5, Hv))
    g, beta = gates.compute_gates(a, b, A_log, dt_bias)
    assert np.all(g < 0) and np.all((beta > 0) & (beta < 1))
    # a = -dt_bias gives softplus(0) = log 2: g = -exp(A_log) log 2 exactly
    g0, _ = gates.compute_gates(np.broadcast_to(-dt_bias, (1, Hv)), np.zeros((1, Hv)), A_log,
                                dt_bias)
    np.testing.assert_allclose(g0[0], -np.exp(A_log) * math.log(2.0), rtol=1e-15)
    # decay of one step = exp(g) = (1 + e^{a + dt})^{-exp(A_log)}
    np.testing.assert_allclose(np.exp(g), (1 + np.exp(a + dt_bias)) ** (-np.exp(A_log)),
                               rtol=1e-12)
