"""Pins for the backward oracle (the reverse-mode adjoint of the gated delta rule), CPU only.

The adjoint is tied to two things other than itself: central finite differences of the
pinned forward recurrence, and torch autograd through an independent fp64 restatement of
the recurrence written here.  Planted mistakes in a copy of the C source must each fail."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")


def rand_case(seed, T=6, Hqk=1, Hv=2, K=3, V=2, N=1):
    rng = np.random.default_rng(seed)
    mk = lambda *s: rng.standard_normal(s)
    q, k, v = mk(1, T, Hqk, K), mk(1, T, Hqk, K), mk(1, T, Hv, V)
    g = -np.log1p(np.exp(mk(1, T, Hv)))
    beta = 1.0 / (1.0 + np.exp(-mk(1, T, Hv)))
    init = 0.3 * mk(N, Hv, K, V)
    do, dfin = mk(1, T, Hv, V), mk(N, Hv, K, V)
    return q, k, v, g, beta, init, do, dfin


def finite_difference_errors(lib=None, l2=True, seed=0):
    """Max relative error of the adjoint against central differences, over every input."""
    q, k, v, g, beta, init, do, dfin = rand_case(seed, T=7, Hqk=1, Hv=2, K=3, V=2, N=3)
    cu = np.array([0, 3, 3, 7])    # a zero-length sequence in the middle

    def loss(q, k, v, g, beta, init):
        o, f = oracle.recurrent(q, k, v, g, beta, initial_state=init, cu_seqlens=cu,
                                use_qk_l2norm_in_kernel=l2, scale=0.7)
        return float((o * do).sum() + (f * dfin).sum())

    grads = oracle.backward(q, k, v, g, beta, do, dfin, initial_state=init, cu_seqlens=cu,
                            use_qk_l2norm_in_kernel=l2, scale=0.7, lib=lib)
    args = [q, k, v, g, beta, init]
    errs = []
    for ai, (x, gx) in enumerate(zip(args, grads)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1e-6
            xm[idx] -= 1e-6
            ap, am = list(args), list(args)
            ap[ai], am[ai] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / 2e-6
        errs.append(float(np.abs(num - gx).max() / max(1e-12, np.abs(num).max())))
    return errs


def torch_recurrence(q, k, v, g, beta, init, cu, scale, l2):
    """The gated delta rule in plain fp64 torch (autograd-ready), independent of the oracle."""
    T, Hqk, K = q.shape[1:]
    Hv, V = v.shape[2:]
    grp = Hv // Hqk
    outs = [None] * T
    finals = []
    for n in range(len(cu) - 1):
        per_head = []
        for h in range(Hv):
            S = init[n, h]
            for t in range(int(cu[n]), int(cu[n + 1])):
                qt, kt = q[0, t, h // grp], k[0, t, h // grp]
                if l2:
                    qt = qt / torch.sqrt((qt * qt).sum() + 1e-6)
                    kt = kt / torch.sqrt((kt * kt).sum() + 1e-6)
                S = torch.exp(g[0, t, h]) * S
                u = beta[0, t, h] * (v[0, t, h] - S.t() @ kt)
                S = S + torch.outer(kt, u)
                if outs[t] is None:
                    outs[t] = [None] * Hv
                outs[t][h] = scale * (S.t() @ qt)
            per_head.append(S)
        finals.append(torch.stack(per_head))
    o = torch.stack([torch.stack(row) for row in outs])[None]
    return o, torch.stack(finals)


def test_adjoint_matches_finite_differences():
    for l2 in (False, True):
        errs = finite_difference_errors(l2=l2)
        assert max(errs) < 1e-7, errs


def test_adjoint_matches_torch_autograd_of_the_recurrence():
    q, k, v, g, beta, init, do, dfin = rand_case(3, T=40, Hqk=2, Hv=4, K=8, V=8, N=3)
    cu = np.array([0, 17, 18, 40])
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v, g, beta, init)]
    o, f = torch_recurrence(*ts, cu, 0.5, True)
    (o * torch.tensor(do)).sum().add((f * torch.tensor(dfin)).sum()).backward()
    grads = oracle.backward(q, k, v, g, beta, do, dfin, initial_state=init, cu_seqlens=cu,
                            use_qk_l2norm_in_kernel=True, scale=0.5)
    for t, gx in zip(ts, grads):
        np.testing.assert_allclose(gx, t.grad.numpy(), rtol=1e-10, atol=1e-11)


MUTANTS = {
    "da_without_state_term": ("da += dS[i * V + c] * Sp[i * V + c];", "da += 0.0 * Sp[i * V + c];"),
    "dstate_without_read_term": ("dS[i * V + c] = a * (dS[i * V + c] + kn[i] * dr[c]);",
                                 "dS[i * V + c] = a * dS[i * V + c];"),
    "dq_without_write_term": ("dqh[i] = scale * (a * s + udo * kn[i]);", "dqh[i] = scale * a * s;"),
    "norm_backward_without_projection": (
        "dx[i] = rho * dxh[i] - rho * rho * rho * xd * x[i];", "dx[i] = rho * dxh[i];"),
    "dbeta_sign": ("db += du[c] * (vt[c] - a * r[c]);", "db -= du[c] * (vt[c] - a * r[c]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site for %s not unique" % name
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(src.replace(old, new))
    so = tmp_path / ("libmut_%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(path), "-o", str(so), "-lm"], check=True)
    lib = oracle.load_library(str(so))
    assert max(finite_difference_errors(lib=lib, l2=True)) > 1e-4


def test_gates_backward_matches_finite_differences():
    """oracle.gates.gates_backward composed with the adjoint gives the gradient of a loss of the
    fused-gate forward w.r.t. the raw features a, b and the per-head parameters A_log, dt_bias:
    central differences of that loss through oracle.gates.compute_gates and the recurrence."""
    from oracle import gates
    rng = np.random.default_rng(41)
    T, Hqk, Hv, K, V = 7, 1, 2, 3, 2
    cu = np.array([0, 3, 3, 7])
    q, k = rng.standard_normal((1, T, Hqk, K)), rng.standard_normal((1, T, Hqk, K))
    v = rng.standard_normal((1, T, Hv, V))
    init = 0.3 * rng.standard_normal((3, Hv, K, V))
    a, b = rng.standard_normal((1, T, Hv)), rng.standard_normal((1, T, Hv))
    A_log = np.log(rng.uniform(1.0, 16.0, Hv))
    dt_bias = 0.5 * rng.standard_normal(Hv)
    do, dfin = rng.standard_normal((1, T, Hv, V)), rng.standard_normal((3, Hv, K, V))

    def loss(a, b, A_log, dt_bias):
        g, beta = gates.compute_gates(a, b, A_log, dt_bias)
        o, f = oracle.recurrent(q, k, v, g, beta, initial_state=init, cu_seqlens=cu,
                                use_qk_l2norm_in_kernel=True)
        return float((o * do).sum() + (f * dfin).sum())

    g, beta = gates.compute_gates(a, b, A_log, dt_bias)
    _, _, _, dg, dbeta, _ = oracle.backward(q, k, v, g, beta, do, dfin, initial_state=init,
                                            cu_seqlens=cu, use_qk_l2norm_in_kernel=True)
    grads = gates.gates_backward(a, b, A_log, dt_bias, dg, dbeta)
    args = [a, b, A_log, dt_bias]
    for ai, (x, gx) in enumerate(zip(args, grads)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1e-6
            xm[idx] -= 1e-6
            ap, am = list(args), list(args)
            ap[ai], am[ai] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / 2e-6
        err = float(np.abs(num - gx).max() / max(1e-12, np.abs(num).max()))
        assert err < 1e-6, (("da", "db", "dA_log", "ddt_bias")[ai], err)


def test_gates_backward_special_values():
    """Closed forms: at a + dt_bias = 0 the softplus slope is 1/2, at b = 0 the sigmoid slope
    is 1/4, and the parameter gradients are the sums over every token of one head."""
    from oracle import gates
    Hv = 3
    dt_bias = np.array([0.2, -1.0, 0.7])
    a = np.broadcast_to(-dt_bias, (2, 5, Hv)).copy()
    b = np.zeros((2, 5, Hv))
    A_log = np.log(np.array([1.0, 2.0, 8.0]))
    dg = np.arange(30.0).reshape(2, 5, Hv) / 7.0
    dbeta = np.ones((2, 5, Hv))
    da, db, dA_log, ddt_bias = gates.gates_backward(a, b, A_log, dt_bias, dg, dbeta)
    np.testing.assert_allclose(da, -dg * np.exp(A_log) * 0.5, rtol=1e-15)
    np.testing.assert_allclose(db, 0.25, rtol=1e-15)
    g = -np.exp(A_log) * np.log(2.0)
    np.testing.assert_allclose(dA_log, dg.sum(axis=(0, 1)) * g, rtol=1e-14)
    np.testing.assert_allclose(ddt_bias, da.sum(axis=(0, 1)), rtol=1e-14)
