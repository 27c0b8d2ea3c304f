"""Planted mistakes: each test compiles a copy of the oracle's C source with one
plausible error (a dropped term, a wrong sign or index, a transposed operand, a
missing mask) and checks that the pins catch it -- at least one of the
independent checks below must fail on the mutant while all pass on the real
oracle.  CPU only; the mutants live in a temporary directory."""
import json
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import closed_form
from tests import exact_rational

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_examples.json")

MUTANTS = {
    "no_decay": ("for (int i = 0; i < K * V; ++i) S[i] *= a;",
                 "for (int i = 0; i < K * V; ++i) S[i] *= 1.0;"),
    "delta_sign": ("u[j] = beta * (v[j] - r[j]);", "u[j] = beta * (v[j] + r[j]);"),
    "readout_before_write": ("o[j] += S[i * V + j] * qn[i];",
                             "o[j] += (S[i * V + j] - kn[i] * u[j]) * qn[i];"),
    "read_with_query": ("r[j] += S[i * V + j] * kn[i];", "r[j] += S[i * V + j] * qn[i];"),
    "scale_twice": ("for (int j = 0; j < V; ++j) o[j] *= scale;",
                    "for (int j = 0; j < V; ++j) o[j] *= scale * scale;"),
    "head_map_modulo": ("const int hq = h / group;\n      for (int64_t t",
                        "const int hq = h % Hqk;\n      for (int64_t t"),
    "chunk_decay_reversed": ("val = bt[i] * kk * exp(G[i] - G[j]);",
                             "val = bt[i] * kk * exp(G[j] - G[i]);"),
    "chunk_no_diagonal": ("for (int j = 0; j <= i; ++j) {\n            double qk",
                          "for (int j = 0; j < i; ++j) {\n            double qk"),
    "chunk_state_no_decay": ("for (size_t x = 0; x < (size_t)K * V; ++x) S[x] *= gl;",
                             "for (size_t x = 0; x < (size_t)K * V; ++x) S[x] *= 1.0;"),
    "chunk_w_without_decay": ("const double sw = bt[i] * exp(G[i]);",
                              "const double sw = bt[i];"),
    "decode_padding_not_zeroed": ("for (int e = 0; e < V; ++e) oi[e] = 0.0;\n        if (s != -1)",
                                  "for (int e = 0; e < V; ++e) oi[e] = oi[e];\n        if (s != -1)"),
    "l2norm_skipped": ("const double r = 1.0 / sqrt(ss + GDN_ORACLE_L2_EPS);",
                       "const double r = 1.0;"),
}


def build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site for %s not unique" % name
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(src.replace(old, new))
    so = tmp_path / ("libmut_%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(path), "-o", str(so), "-lm"], check=True)
    return oracle.load_library(str(so))


def rel(x, ref):
    d = np.linalg.norm(np.asarray(ref))
    return float(np.linalg.norm(np.asarray(x) - np.asarray(ref)) / (d if d > 0 else 1.0))


# ---------------------------------------------------------------- the checks

def check_hand_prefill(lib):
    ex = json.load(open(GOLDEN))["prefill"]
    q = np.array(ex["q"], float).reshape(1, 2, 1, 2)
    k = np.array(ex["k"], float).reshape(1, 2, 1, 2)
    v = np.array(ex["v"], float).reshape(1, 2, 1, 2)
    g = np.log(np.array(ex["a"])).reshape(1, 2, 1)
    b = np.array(ex["beta"]).reshape(1, 2, 1)
    s0 = np.array(ex["initial_state"], float).reshape(1, 1, 2, 2)
    ok = True
    for fn in (oracle.recurrent, oracle.chunked):
        kw = {"chunk_size": 2} if fn is oracle.chunked else {}
        o, f = fn(q, k, v, g, b, scale=1.0, initial_state=s0, lib=lib, **kw)
        ok &= np.allclose(o[0, :, 0], ex["expected_o"], atol=1e-12)
        ok &= np.allclose(f[0, 0], ex["expected_final_state"], atol=1e-12)
    return bool(ok)


def check_hand_decode(lib):
    ex = json.load(open(GOLDEN))["decode"]
    n = 3
    cache = np.array(ex["initial_cache"], float).reshape(-1, 1, 1, 1).copy()
    o = oracle.decode(np.array(ex["q"], float).reshape(n, 1, 1),
                      np.array(ex["k"], float).reshape(n, 1, 1),
                      np.array(ex["v"], float).reshape(n, 1, 1),
                      np.log(np.array(ex["a"])).reshape(n, 1), np.array(ex["beta"]).reshape(n, 1),
                      cache, np.array(ex["batch_indices"]), scale=1.0,
                      use_qk_l2norm_in_kernel=False, lib=lib)
    return bool(np.allclose(o.ravel(), ex["expected_o"], atol=1e-12)
                and np.allclose(cache.ravel(), ex["expected_cache"], atol=1e-12))


def check_exact(lib):
    rng = np.random.default_rng(4)
    lengths, Hqk, Hv, K, V = [5, 7], 1, 2, 3, 4
    T = sum(lengths)
    q = rng.integers(-3, 4, (T, Hqk, K)); k = rng.integers(-3, 4, (T, Hqk, K))
    v = rng.integers(-3, 4, (T, Hv, V))
    dec = [Fraction(1), Fraction(1, 2), Fraction(3, 4)]
    bet = [Fraction(1, 4), Fraction(1, 2), Fraction(1)]
    a = [[dec[x] for x in row] for row in rng.integers(0, 3, (T, Hv))]
    b = [[bet[x] for x in row] for row in rng.integers(0, 3, (T, Hv))]
    s0 = rng.integers(-2, 3, (2, Hv, K, V))
    o_ex, f_ex = exact_rational.run(q.tolist(), k.tolist(), v.tolist(), a, b, [0, 5, 12], Hqk, Hv,
                                    Fraction(1, 2), s0.tolist())
    g = np.log(np.array([[float(x) for x in r] for r in a]))
    beta = np.array([[float(x) for x in r] for r in b])
    o, f = oracle.recurrent(q.reshape(1, T, Hqk, K), k.reshape(1, T, Hqk, K), v.reshape(1, T, Hv, V),
                            g.reshape(1, T, Hv), beta.reshape(1, T, Hv), scale=0.5,
                            initial_state=s0, cu_seqlens=np.array([0, 5, 12]), lib=lib)
    o_ref = np.array([[[float(x) for x in r] for r in tok] for tok in o_ex])
    f_ref = np.array([[[[float(x) for x in r] for r in hd] for hd in sq] for sq in f_ex])
    return rel(o[0], o_ref) < 1e-12 and rel(f, f_ref) < 1e-12


def rand_inputs(seed, T=70, Hqk=1, Hv=2, K=6, V=5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, Hqk, K)); k = rng.standard_normal((1, T, Hqk, K))
    v = rng.standard_normal((1, T, Hv, V))
    g = -np.log1p(np.exp(rng.standard_normal((1, T, Hv))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((1, T, Hv))))
    s0 = 0.5 * rng.standard_normal((1, Hv, K, V))
    return q, k, v, g, beta, s0


def check_chunked_vs_recurrent(lib):
    q, k, v, g, beta, s0 = rand_inputs(7)
    o1, f1 = oracle.recurrent(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True,
                              lib=lib)
    o2, f2 = oracle.chunked(q, k, v, g, beta, initial_state=s0, chunk_size=16,
                            use_qk_l2norm_in_kernel=True, lib=lib)
    return rel(o2, o1) < 1e-11 and rel(f2, f1) < 1e-11


def check_closed_form(lib):
    q, k, v, g, beta, s0 = rand_inputs(8, T=7, Hqk=1, Hv=2, K=4, V=3)
    ok = True
    for fn in (oracle.recurrent, oracle.chunked):
        o, f = fn(q, k, v, g, beta, initial_state=s0, use_qk_l2norm_in_kernel=True, lib=lib)
        o2, f2 = closed_form.batched(q, k, v, g, beta, initial_state=s0, use_qk_l2norm=True)
        ok &= rel(o, o2) < 1e-12 and rel(f, f2) < 1e-12
    return bool(ok)


def check_grouped_heads(lib):
    q, k, v, g, beta, s0 = rand_inputs(9, T=20, Hqk=2, Hv=4)
    o1, _ = oracle.recurrent(q, k, v, g, beta, initial_state=s0, lib=lib)
    o2, _ = closed_form.batched(q, k, v, g, beta, initial_state=s0)
    return rel(o1, o2) < 1e-12


def check_decode_padding(lib):
    rng = np.random.default_rng(10)
    cache = rng.standard_normal((4, 1, 3, 3))
    o = oracle.decode(rng.standard_normal((2, 1, 3)), rng.standard_normal((2, 1, 3)),
                      rng.standard_normal((2, 1, 3)), -np.ones((2, 1)), 0.5 * np.ones((2, 1)),
                      cache, np.array([-1, 2]), lib=lib)
    return bool(np.all(o[0] == 0.0))


def check_l2norm(lib):
    rng = np.random.default_rng(11)
    q = 3 * rng.standard_normal((1, 1, 1, 8)); k = 0.5 * rng.standard_normal((1, 1, 1, 8))
    v = rng.standard_normal((1, 1, 1, 2))
    o, _ = oracle.recurrent(q, k, v, np.zeros((1, 1, 1)), np.ones((1, 1, 1)), scale=1.0,
                            use_qk_l2norm_in_kernel=True, lib=lib)
    qh = q.ravel() / np.linalg.norm(q); kh = k.ravel() / np.linalg.norm(k)
    return bool(np.allclose(o.ravel(), (qh @ kh) * v.ravel(), rtol=1e-6))


CHECKS = [check_hand_prefill, check_hand_decode, check_exact, check_chunked_vs_recurrent,
          check_closed_form, check_grouped_heads, check_decode_padding, check_l2norm]


def test_real_oracle_passes_every_check():
    lib = oracle._load()
    for c in CHECKS:
        assert c(lib), c.__name__


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    lib = build_mutant(tmp_path, name)
    with np.errstate(all="ignore"):
        failed = []
        for c in CHECKS:
            try:
                if not c(lib):
                    failed.append(c.__name__)
            except (RuntimeError, FloatingPointError, ValueError):
                failed.append(c.__name__)
    assert failed, "mutant %s passed every check" % name
