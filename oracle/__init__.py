"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product (the CUDA library and its
Python binding in ``chunked_gated_delta_gdn_gb300``) never imports it, and it
imports nothing from the product.

Three functions wrap the C library built from ``gdn_oracle.c``:

* :func:`recurrent` -- the definition, token by token (the gated delta rule of
  "Megatron-Core API: core.ssm.gated_delta_net.gdn", GatedDeltaNet; arguments
  follow torch_chunk_gated_delta_rule on the same page).
* :func:`chunked` -- the chunkwise (WY / UT-transform) evaluation for any chunk
  size, an independent second form.
* :func:`decode` -- one token per request on a slot-indexed cache with ``-1``
  padding ("Megatron-Core API: core.ssm.gated_delta_product",
  GatedDeltaProductMixer.ssm_decode).

:func:`product` and :func:`product_decode` evaluate the Gated Delta Product (several
delta-rule writes per token, "Megatron-Core API: core.ssm.gated_delta_product",
GatedDeltaProductMixer) by its recurrence.

:func:`backward` returns the gradients of every input of :func:`recurrent` for given
output / final-state gradients (the reverse-mode adjoint of the recurrence).

:mod:`oracle.closed_form` adds the unrolled product form for tiny inputs.

Pinned by ``tests/test_oracle_pins.py`` (the gated delta rule),
``tests/test_oracle_product_pins.py`` (the product) and
``tests/test_oracle_backward_pins.py`` (the adjoint); see the header of
``gdn_oracle.c`` for the exact update rule and the readings it takes.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK, ORACLE_ERR_ARG, ORACLE_ERR_NOMEM, ORACLE_ERR_SLOT = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``oracle/_build/libgdn_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str) -> ctypes.CDLL:
    """Open an oracle shared library built from gdn_oracle.c and declare its entry points."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_int64)
    i, d = ctypes.c_int, ctypes.c_double
    lib.gdn_oracle_recurrent.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, lp, i, d, i,
                                         dp, dp, dp, i]
    lib.gdn_oracle_chunked.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, lp, i, d, i, i,
                                       dp, dp, dp, i]
    lib.gdn_oracle_decode.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, dp, i, lp, d, i,
                                      dp, i]
    lib.gdn_oracle_product.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, lp, i, d, i,
                                       dp, dp, dp, i]
    lib.gdn_oracle_product_decode.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, dp, i, lp,
                                              d, i, dp, i]
    lib.gdn_oracle_backward.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, lp, i, d, i, dp, dp, dp,
                                        dp, dp, dp, dp, dp, dp, i]
    for f in (lib.gdn_oracle_recurrent, lib.gdn_oracle_chunked, lib.gdn_oracle_decode,
              lib.gdn_oracle_product, lib.gdn_oracle_product_decode, lib.gdn_oracle_backward):
        f.restype = ctypes.c_int
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle uses when ``nthreads`` is 0."""
    return int(_load().gdn_oracle_max_threads())


def _f64(x):
    """Lossless conversion to a C-contiguous float64 numpy array (torch or numpy input)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a, typ=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(typ))


def _prep_seq(q, k, v, g, beta, cu_seqlens, initial_state):
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4:
        raise ValueError("q, k must be [B, T, Hqk, K] and v [B, T, Hv, V]")
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    if v.shape[:2] != (B, T) or g.shape != (B, T, Hv) or beta.shape != (B, T, Hv):
        raise ValueError("g and beta must be [B, T, Hv]")
    if Hv % Hqk != 0:
        raise ValueError("Hv must be a multiple of Hqk")
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = _i64(cu_seqlens)
    N = cu.shape[0] - 1
    init = _f64(initial_state)
    if init is not None and init.shape != (N, Hv, K, V):
        raise ValueError("initial_state must be [N, Hv, K, V]")
    return q, k, v, g, beta, cu, init, (B, T, Hqk, Hv, K, V, N)


def _scale(scale, K):
    return 1.0 / math.sqrt(K) if scale is None else float(scale)


def recurrent(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=True,
              use_qk_l2norm_in_kernel=False, cu_seqlens=None, nthreads=0, lib=None):
    """Token-by-token gated delta rule.  Returns ``(o, final_state | None)`` as float64 numpy."""
    q, k, v, g, beta, cu, init, (B, T, Hqk, Hv, K, V, N) = _prep_seq(
        q, k, v, g, beta, cu_seqlens, initial_state)
    o = np.full((B, T, Hv, V), np.nan)   # every row a sequence covers is written
    fin = np.zeros((N, Hv, K, V), dtype=np.float64) if output_final_state else None
    rc = (lib or _load()).gdn_oracle_recurrent(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B * T, Hqk, Hv, K, V,
        _ptr(cu, ctypes.c_int64), N, _scale(scale, K), int(bool(use_qk_l2norm_in_kernel)),
        _ptr(init), _ptr(o), _ptr(fin), int(nthreads))
    if rc != ORACLE_OK:
        raise RuntimeError("gdn_oracle_recurrent failed with code %d" % rc)
    return o, fin


def chunked(q, k, v, g, beta, scale=None, chunk_size=64, initial_state=None,
            output_final_state=True, use_qk_l2norm_in_kernel=False, cu_seqlens=None, nthreads=0,
            lib=None):
    """Chunkwise (WY / UT-transform) evaluation for any ``chunk_size >= 1``."""
    q, k, v, g, beta, cu, init, (B, T, Hqk, Hv, K, V, N) = _prep_seq(
        q, k, v, g, beta, cu_seqlens, initial_state)
    o = np.full((B, T, Hv, V), np.nan)   # every row a sequence covers is written
    fin = np.zeros((N, Hv, K, V), dtype=np.float64) if output_final_state else None
    rc = (lib or _load()).gdn_oracle_chunked(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B * T, Hqk, Hv, K, V,
        _ptr(cu, ctypes.c_int64), N, _scale(scale, K), int(bool(use_qk_l2norm_in_kernel)),
        int(chunk_size), _ptr(init), _ptr(o), _ptr(fin), int(nthreads))
    if rc != ORACLE_OK:
        raise RuntimeError("gdn_oracle_chunked failed with code %d" % rc)
    return o, fin


def decode(q, k, v, g, beta, ssm_state, batch_indices=None, scale=None,
           use_qk_l2norm_in_kernel=True, nthreads=0, allow_bad_slots=False, lib=None):
    """One token per request.  ``ssm_state`` ([num_slots, Hv, K, V] float64 numpy) is
    updated in place; returns ``o`` [n, Hv, V].  ``-1`` slots give zero rows."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if not (isinstance(ssm_state, np.ndarray) and ssm_state.dtype == np.float64
            and ssm_state.flags.c_contiguous):
        raise TypeError("ssm_state must be a C-contiguous float64 numpy array (updated in place)")
    n, Hqk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    if ssm_state.ndim != 4 or ssm_state.shape[1:] != (Hv, K, V):
        raise ValueError("ssm_state must be [num_slots, Hv, K, V]")
    idx = _i64(batch_indices)
    o = np.full((n, Hv, V), np.nan)      # every row is written (zeros for padding)
    rc = (lib or _load()).gdn_oracle_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), n, Hqk, Hv, K, V, _ptr(ssm_state),
        ssm_state.shape[0], _ptr(idx, ctypes.c_int64), _scale(scale, K),
        int(bool(use_qk_l2norm_in_kernel)), _ptr(o), int(nthreads))
    if rc == ORACLE_ERR_SLOT and allow_bad_slots:
        return o
    if rc != ORACLE_OK:
        raise RuntimeError("gdn_oracle_decode failed with code %d" % rc)
    return o


def product(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=True,
            use_qk_l2norm_in_kernel=False, cu_seqlens=None, nthreads=0, lib=None):
    """Gated Delta Product by its recurrence: q [B, T, Hqk, K], k [B, T, n_h, Hqk, K],
    v [B, T, n_h, Hv, V], g [B, T, Hv], beta [B, T, n_h, Hv].  Returns ``(o, final_state)``."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if q.ndim != 4 or k.ndim != 5 or v.ndim != 5:
        raise ValueError("q must be [B, T, Hqk, K], k [B, T, n_h, Hqk, K], v [B, T, n_h, Hv, V]")
    B, T, Hqk, K = q.shape
    n_h = k.shape[2]
    Hv, V = v.shape[3], v.shape[4]
    if (k.shape != (B, T, n_h, Hqk, K) or v.shape[:3] != (B, T, n_h) or g.shape != (B, T, Hv)
            or beta.shape != (B, T, n_h, Hv)):
        raise ValueError("inconsistent shapes")
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = _i64(cu_seqlens)
    N = cu.shape[0] - 1
    init = _f64(initial_state)
    if init is not None and init.shape != (N, Hv, K, V):
        raise ValueError("initial_state must be [N, Hv, K, V]")
    o = np.full((B, T, Hv, V), np.nan)
    fin = np.zeros((N, Hv, K, V), dtype=np.float64) if output_final_state else None
    rc = (lib or _load()).gdn_oracle_product(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B * T, n_h, Hqk, Hv, K, V,
        _ptr(cu, ctypes.c_int64), N, _scale(scale, K), int(bool(use_qk_l2norm_in_kernel)),
        _ptr(init), _ptr(o), _ptr(fin), int(nthreads))
    if rc != ORACLE_OK:
        raise RuntimeError("gdn_oracle_product failed with code %d" % rc)
    return o, fin


def product_decode(q, k, v, g, beta, ssm_state, batch_indices=None, scale=None,
                   use_qk_l2norm_in_kernel=True, nthreads=0, allow_bad_slots=False, lib=None):
    """One Gated Delta Product token per request: q [n, Hqk, K], k [n, n_h, Hqk, K],
    v [n, n_h, Hv, V], g [n, Hv], beta [n, n_h, Hv].  ``ssm_state`` (float64 numpy) is updated
    in place; returns ``o`` [n, Hv, V]; ``-1`` slots give zero rows."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if not (isinstance(ssm_state, np.ndarray) and ssm_state.dtype == np.float64
            and ssm_state.flags.c_contiguous):
        raise TypeError("ssm_state must be a C-contiguous float64 numpy array (updated in place)")
    n, Hqk, K = q.shape
    n_h = k.shape[1]
    Hv, V = v.shape[2], v.shape[3]
    if ssm_state.ndim != 4 or ssm_state.shape[1:] != (Hv, K, V):
        raise ValueError("ssm_state must be [num_slots, Hv, K, V]")
    idx = _i64(batch_indices)
    o = np.full((n, Hv, V), np.nan)
    rc = (lib or _load()).gdn_oracle_product_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), n, n_h, Hqk, Hv, K, V, _ptr(ssm_state),
        ssm_state.shape[0], _ptr(idx, ctypes.c_int64), _scale(scale, K),
        int(bool(use_qk_l2norm_in_kernel)), _ptr(o), int(nthreads))
    if rc == ORACLE_ERR_SLOT and allow_bad_slots:
        return o
    if rc != ORACLE_OK:
        raise RuntimeError("gdn_oracle_product_decode failed with code %d" % rc)
    return o


def backward(q, k, v, g, beta, d_o, d_final_state=None, scale=None, initial_state=None,
             use_qk_l2norm_in_kernel=False, cu_seqlens=None, nthreads=0, lib=None):
    """Gradients of the gated delta rule (layouts of :func:`recurrent`) for the output
    gradient ``d_o`` [B, T, Hv, V] and optional final-state gradient [N, Hv, K, V].
    Returns ``(dq, dk, dv, dg, dbeta, d_initial_state)`` as float64 numpy."""
    q, k, v, g, beta, cu, init, (B, T, Hqk, Hv, K, V, N) = _prep_seq(
        q, k, v, g, beta, cu_seqlens, initial_state)
    do = _f64(d_o)
    dfin = _f64(d_final_state)
    if do.shape != (B, T, Hv, V):
        raise ValueError("d_o must be [B, T, Hv, V]")
    if dfin is not None and dfin.shape != (N, Hv, K, V):
        raise ValueError("d_final_state must be [N, Hv, K, V]")
    dq = np.zeros((B, T, Hqk, K))
    dk = np.zeros((B, T, Hqk, K))
    dv = np.full((B, T, Hv, V), np.nan)
    dg = np.full((B, T, Hv), np.nan)
    db = np.full((B, T, Hv), np.nan)
    dinit = np.zeros((N, Hv, K, V))
    rc = (lib or _load()).gdn_oracle_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), B * T, Hqk, Hv, K, V,
        _ptr(cu, ctypes.c_int64), N, _scale(scale, K), int(bool(use_qk_l2norm_in_kernel)),
        _ptr(init), _ptr(do), _ptr(dfin), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(db),
        _ptr(dinit), int(nthreads))
    if rc != ORACLE_OK:
        raise RuntimeError("gdn_oracle_backward failed with code %d" % rc)
    return dq, dk, dv, dg, db, dinit
