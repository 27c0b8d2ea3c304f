"""Gate computation of the GDN mixer, fp64 numpy -- TEST INFRASTRUCTURE ONLY.

The mixer computes "the per-head log-decay g and the write strength beta" from
its projected gate features and two per-head parameters, A_log and dt_bias
("Megatron-Core API: core.ssm.gated_delta_net.gdn", GatedDeltaNet._compute_gates;
A_init_range=(1, 16) on the same class).  The pages print no formula; the
reading used here is the plain one for that parameterisation:

    g    = -exp(A_log[h]) * softplus(a + dt_bias[h])      (a log-decay, always < 0)
    beta = sigmoid(b)                                     (a write strength in (0, 1))

with softplus(x) = log(1 + exp(x)) and sigmoid(x) = 1 / (1 + exp(-x)), both
evaluated in forms that neither overflow nor lose the tail.
"""
from __future__ import annotations

import numpy as np


def softplus(x):
    """log(1 + e^x) = max(x, 0) + log1p(e^{-|x|}), exact in fp64 for every x."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    """1 / (1 + e^{-x}) without overflow for large |x|."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def compute_gates(a, b, A_log, dt_bias):
    """a, b: [..., Hv]; A_log, dt_bias: [Hv].  Returns (g, beta) as float64 arrays."""
    f64 = lambda x: (x.detach().cpu().double().numpy() if hasattr(x, "detach")
                     else np.asarray(x, dtype=np.float64))
    a, b, A_log, dt_bias = (f64(x) for x in (a, b, A_log, dt_bias))
    g = -np.exp(A_log) * softplus(a + dt_bias)
    beta = sigmoid(b)
    return g, beta


def gates_backward(a, b, A_log, dt_bias, dg, dbeta):
    """Gradients of a loss through the gates, given its gradients dg, dbeta w.r.t. g and beta
    ([..., Hv]).  With x = a + dt_bias[h]:
        d softplus(x) / dx = sigmoid(x),     d sigmoid(b) / db = sigmoid(b) (1 - sigmoid(b)),
        dg / da = dg / d dt_bias = -exp(A_log) sigmoid(x),     dg / dA_log = g,
    so da = dg * (-exp(A_log) sigmoid(x)), db = dbeta * beta (1 - beta), and the per-head
    parameters collect over every leading index: dA_log[h] = sum dg * g,
    ddt_bias[h] = sum da.  Returns (da, db, dA_log, ddt_bias) as float64 arrays."""
    f64 = lambda x: (x.detach().cpu().double().numpy() if hasattr(x, "detach")
                     else np.asarray(x, dtype=np.float64))
    a, b, A_log, dt_bias, dg, dbeta = (f64(x) for x in (a, b, A_log, dt_bias, dg, dbeta))
    x = a + dt_bias
    g = -np.exp(A_log) * softplus(x)
    beta = sigmoid(b)
    da = dg * (-np.exp(A_log) * sigmoid(x))
    db = dbeta * beta * (1.0 - beta)
    lead = tuple(range(da.ndim - 1))
    return da, db, (dg * g).sum(axis=lead), da.sum(axis=lead)
