"""Pins for the Gated Delta Product oracle (several delta-rule writes per token,
"Megatron-Core API: core.ssm.gated_delta_product", GatedDeltaProductMixer), CPU only.

Each pin ties the oracle to something other than itself: exact rational arithmetic on tiny
inputs, the single-write special case (the pinned gated delta rule), the identity with the
gated delta rule over the sequence of writes (decay on the first, query on the last), the
beta = 0 closed form, and the decode step against the sequence form.  Planted mistakes in a
copy of the C source must each fail at least one pin."""
import math
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import exact_rational

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")


def rand_product(seed, B=1, T=7, n_h=2, Hqk=1, Hv=2, K=4, V=3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hqk, K))
    k = rng.standard_normal((B, T, n_h, Hqk, K))
    v = rng.standard_normal((B, T, n_h, Hv, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, n_h, Hv))))
    return q, k, v, g, beta


def expand(q, k, v, g, beta):
    """The same inputs as one gated-delta-rule sequence of T * n_h writes."""
    B, T, n_h, Hqk, K = k.shape
    Hv = v.shape[3]
    qe = np.zeros((B, T, n_h, Hqk, K))
    qe[:, :, -1] = q
    ge = np.zeros((B, T, n_h, Hv))
    ge[:, :, 0] = g
    r = lambda x: x.reshape((B, T * n_h) + x.shape[3:])
    return r(qe), r(k), r(v), r(ge), r(beta)


def check_all(lib=None):
    """Every pin at once; returns the list of failed pin names (empty on the real oracle)."""
    failed = []
    # exact rational, n_h = 2 and 3, two sequences, initial state, two value heads
    for n_h in (2, 3):
        T, Hqk, Hv, K, V = 4, 1, 2, 3, 2
        rng = np.random.default_rng(10 + n_h)
        ints = lambda shape: rng.integers(-3, 4, size=shape).astype(np.float64)
        q, k, v = ints((T, Hqk, K)), ints((T, n_h, Hqk, K)) / 4, ints((T, n_h, Hv, V))
        a = rng.choice([0.5, 0.75, 1.0], size=(T, Hv))
        beta = rng.choice([0.25, 0.5, 1.0], size=(T, n_h, Hv))
        init = ints((2, Hv, K, V)) / 8
        cu = [0, 1, 4]
        o_ex, f_ex = exact_rational.run_product(
            q.tolist(), k.tolist(), v.tolist(), [[Fraction(x) for x in row] for row in a],
            beta.tolist(), cu, Hqk, Hv, Fraction(1, 2), init.tolist())
        o, f = oracle.product(q[None], k[None], v[None], np.log(a)[None], beta[None], scale=0.5,
                              initial_state=init, cu_seqlens=np.array(cu), lib=lib)
        o_ex = np.array([[[float(x) for x in row] for row in t] for t in o_ex])
        f_ex = np.array([[[[float(x) for x in r] for r in hh] for hh in nn] for nn in f_ex])
        if not (np.allclose(o[0], o_ex, rtol=1e-12, atol=1e-12) and
                np.allclose(f, f_ex, rtol=1e-12, atol=1e-12)):
            failed.append("exact_rational_nh%d" % n_h)
    # the gated delta rule over the sequence of writes
    q, k, v, g, beta = rand_product(1, B=2, T=9, n_h=3, Hqk=2, Hv=4, K=5, V=3)
    init = np.random.default_rng(2).standard_normal((2, 4, 5, 3)) * 0.1
    o, f = oracle.product(q, k, v, g, beta, initial_state=init, use_qk_l2norm_in_kernel=True,
                          lib=lib)
    qe, ke, ve, ge, be = expand(q, k, v, g, beta)
    oe, fe = oracle.recurrent(qe, ke, ve, ge, be, initial_state=init,
                              use_qk_l2norm_in_kernel=True)
    oe = oe.reshape(2, 9, 3, 4, 3)[:, :, -1]
    if not (np.allclose(o, oe, rtol=1e-12, atol=1e-13) and np.allclose(f, fe, rtol=1e-12, atol=1e-13)):
        failed.append("expanded_rule")
    # beta = 0: pure decay of the initial state
    q, k, v, g, beta = rand_product(3, T=6, n_h=2)
    init = np.random.default_rng(4).standard_normal((1, 2, 4, 3))
    o, f = oracle.product(q, k, v, g, np.zeros_like(beta), scale=0.7, initial_state=init,
                          use_qk_l2norm_in_kernel=True, lib=lib)
    G = np.cumsum(g[0], axis=0)
    qn = q[0, :, 0] / np.sqrt((q[0, :, 0] ** 2).sum(-1, keepdims=True) + 1e-6)
    o_cf = 0.7 * np.exp(G)[:, :, None] * np.einsum("hkv,tk->thv", init[0], qn)
    f_cf = np.exp(G[-1])[:, None, None] * init[0]
    if not (np.allclose(o[0], o_cf, rtol=1e-12, atol=1e-13) and np.allclose(f[0], f_cf, rtol=1e-12)):
        failed.append("zero_beta")
    # decode: one token per request against the sequence form, with padding
    q, k, v, g, beta = rand_product(5, B=1, T=5, n_h=2, Hqk=1, Hv=2, K=4, V=3)
    cache = np.random.default_rng(6).standard_normal((7, 2, 4, 3))
    idx = np.array([3, -1, 0, 6, 2])
    cache0 = cache.copy()
    od = oracle.product_decode(q[0], k[0], v[0], g[0], beta[0], cache, idx, lib=lib)
    ok = np.all(od[1] == 0.0) and np.array_equal(cache[[1, 4, 5]], cache0[[1, 4, 5]])
    for i, s in enumerate(idx):
        if s < 0:
            continue
        o1, f1 = oracle.product(q[:, i:i + 1], k[:, i:i + 1], v[:, i:i + 1], g[:, i:i + 1],
                                beta[:, i:i + 1], initial_state=cache0[s:s + 1],
                                use_qk_l2norm_in_kernel=True)
        ok = ok and np.allclose(od[i], o1[0, 0], rtol=1e-13, atol=1e-14) and np.allclose(
            cache[s], f1[0], rtol=1e-13, atol=1e-14)
    if not ok:
        failed.append("decode_vs_sequence")
    return failed


def test_single_write_is_the_gated_delta_rule():
    """n_h = 1 reduces to the pinned token-by-token rule (varlen, grouped heads, norms)."""
    rng = np.random.default_rng(0)
    q, k, v, g, beta = rand_product(0, B=1, T=11, n_h=1, Hqk=2, Hv=4, K=5, V=3)
    init = rng.standard_normal((3, 4, 5, 3)) * 0.1
    cu = np.array([0, 4, 4, 11])
    o, f = oracle.product(q, k, v, g, beta, initial_state=init, cu_seqlens=cu,
                          use_qk_l2norm_in_kernel=True)
    o2, f2 = oracle.recurrent(q, k[:, :, 0], v[:, :, 0], g, beta[:, :, 0], initial_state=init,
                              cu_seqlens=cu, use_qk_l2norm_in_kernel=True)
    np.testing.assert_allclose(o, o2, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(f, f2, rtol=1e-14, atol=1e-15)


def test_real_oracle_passes_every_pin():
    assert check_all() == []


MUTANTS = {
    "only_first_write": ("(size_t)Hv, n_h, K, V,\n                              use_qk_l2norm, kn, r);",
                         "(size_t)Hv, 1, K, V,\n                              use_qk_l2norm, kn, r);"),
    "decay_per_write": ("S[x] *= a;\n        oracle_product_writes",
                        "S[x] *= pow(a, n_h);\n        oracle_product_writes"),
    "first_beta_for_all": ("const double bj = bb[(size_t)j * bs];", "const double bj = bb[0];"),
    "read_with_first_key": ("oracle_l2norm(q + ((size_t)t * Hqk + hq) * K, K, use_qk_l2norm, qn);\n        oracle_readout",
                            "oracle_l2norm(k + (((size_t)t * n_h) * Hqk + hq) * K, K, use_qk_l2norm, qn);\n        oracle_readout"),
    "decode_no_decay": ("const double a = exp(g[(size_t)i * Hv + h]);",
                        "const double a = 1.0 + 0.0 * g[(size_t)i * Hv + h];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_product_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site for %s not unique" % name
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(src.replace(old, new))
    so = tmp_path / ("libmut_%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(path), "-o", str(so), "-lm"], check=True)
    assert check_all(oracle.load_library(str(so))) != []
