/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
 * smoke() check and the benchmark's CPU-baseline leg may load this library.
 * The CUDA path never includes, links or calls anything here, and nothing here
 * includes anything from the CUDA path.
 *
 * What it computes (the sources print no formula; the method they name is the
 * gated delta rule whose per-head log-decay g and write strength beta the GDN
 * mixer produces -- "Megatron-Core API: core.ssm.gated_delta_net.gdn",
 * GatedDeltaNet._compute_gates -- and whose state update is a delta-rule
 * (Householder-type) write -- "Megatron-Core API: core.ssm.gated_delta_product",
 * GatedDeltaProductMixer class description).  The plain reading used here, per
 * (sequence, value head) with a K x V state S:
 *
 *     S   <- exp(g_t) * S                       (decay first)
 *     r    = S^T k_t                            (read with the decayed state)
 *     u    = beta_t * (v_t - r)                 (delta-rule correction)
 *     S   <- S + k_t u^T                        (rank-1 write)
 *     o_t  = scale * S^T q_t                    (read-out with the updated state)
 *
 * with q_t, k_t optionally L2-normalised first (x / sqrt(sum x^2 + eps),
 * eps = 1e-6), scale defaulting to 1/sqrt(K) (torch_chunk_gated_delta_rule,
 * same page), and value head h reading query/key head h / (Hv / Hqk).
 *
 * Entry points:
 *   gdn_oracle_recurrent  -- the definition above, token by token.
 *   gdn_oracle_chunked    -- the chunkwise (WY / UT-transform) evaluation for
 *                            any chunk size C >= 1, chunks restarting at every
 *                            sequence start (torch_chunk_gated_delta_rule's
 *                            chunk_size argument; the fixed 64-token chunking
 *                            of GatedDeltaProductMixer.ssm_inference_chunk_size).
 *   gdn_oracle_decode     -- one token per request on a slot-indexed state
 *                            cache; slot -1 is padding: no state read or write,
 *                            output exactly zero (GatedDeltaProductMixer.ssm_decode;
 *                            "Add GDN dynamic inference" PR review thread).
 *   gdn_oracle_product, gdn_oracle_product_decode -- the Gated Delta Product
 *                            (several writes per token), near the end of this file.
 *   gdn_oracle_backward   -- the gradients of every input of gdn_oracle_recurrent
 *                            (its reverse-mode adjoint), for training: the chunked
 *                            rule is the training path of the GDN layer
 *                            (GatedDeltaNet, torch_chunk_gated_delta_rule's
 *                            deterministic mode; GatedDeltaProductMixer._gdp_chunk_forward
 *                            serves training too).  Pinned by central finite
 *                            differences and by autograd of an independent
 *                            recurrence in the tests.
 *
 * Layouts (all row-major, fp64):
 *   q, k   [T_total, Hqk, K]     v, o [T_total, Hv, V]     g, beta [T_total, Hv]
 *   states [N, Hv, K, V]         cu_seqlens [N + 1] int64, monotone, starts at 0.
 *
 * Build:  gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (oracle/build.py).
 * FP contraction is off so that x86 and Arm hosts give identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GDN_ORACLE_L2_EPS 1e-6

/* Error codes returned by every entry point. */
#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2
#define ORACLE_ERR_SLOT 3

/* Copy x (length n) to out, L2-normalised when use != 0. */
static void oracle_l2norm(const double* x, int n, int use, double* out) {
  if (!use) {
    memcpy(out, x, (size_t)n * sizeof(double));
    return;
  }
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  const double r = 1.0 / sqrt(ss + GDN_ORACLE_L2_EPS);
  for (int i = 0; i < n; ++i) out[i] = x[i] * r;
}

static int check_common(int Hqk, int Hv, int K, int V, const int64_t* cu, int N) {
  if (Hqk <= 0 || Hv <= 0 || K <= 0 || V <= 0 || N < 0 || !cu) return ORACLE_ERR_ARG;
  if (Hv % Hqk != 0) return ORACLE_ERR_ARG;
  if (cu[0] != 0) return ORACLE_ERR_ARG;
  for (int n = 0; n < N; ++n)
    if (cu[n + 1] < cu[n]) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* OpenMP threads of a call: nthreads > 0 as given, 0 the process default (the count OpenMP
   had before the first call set it), so a one-thread call does not stick to later calls. */
static int g_default_threads = 0;
static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (g_default_threads == 0) g_default_threads = omp_get_max_threads();
  omp_set_num_threads(nthreads > 0 ? nthreads : g_default_threads);
#else
  (void)nthreads;
#endif
}

/* One step of the rule on a K x V state S (in place).  qn, kn are already
 * normalised.  Writes the V-vector o.  Used by the recurrent and decode paths. */
static void oracle_step(double* S, const double* qn, const double* kn, const double* v,
                        double g, double beta, double scale, int K, int V,
                        double* r, double* u, double* o) {
  const double a = exp(g);
  for (int i = 0; i < K * V; ++i) S[i] *= a;
  for (int j = 0; j < V; ++j) r[j] = 0.0;
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) r[j] += S[i * V + j] * kn[i];
  for (int j = 0; j < V; ++j) u[j] = beta * (v[j] - r[j]);
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) S[i * V + j] += kn[i] * u[j];
  for (int j = 0; j < V; ++j) o[j] = 0.0;
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) o[j] += S[i * V + j] * qn[i];
  for (int j = 0; j < V; ++j) o[j] *= scale;
}

/*
 * Token-by-token recurrence over packed sequences.
 * initial_state may be NULL (zeros); final_state may be NULL (not written).
 */
int gdn_oracle_recurrent(const double* q, const double* k, const double* v,
                         const double* g, const double* beta, int T_total, int Hqk,
                         int Hv, int K, int V, const int64_t* cu_seqlens, int N,
                         double scale, int use_qk_l2norm, const double* initial_state,
                         double* o, double* final_state, int nthreads) {
  int err = check_common(Hqk, Hv, K, V, cu_seqlens, N);
  if (err) return err;
  if (cu_seqlens[N] > T_total || !q || !k || !v || !g || !beta || !o) return ORACLE_ERR_ARG;
  const int group = Hv / Hqk;
  int failed = 0;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int n = 0; n < N; ++n) {
    for (int h = 0; h < Hv; ++h) {
      double* S = (double*)malloc(sizeof(double) * ((size_t)K * V + 2 * K + 2 * V));
      if (!S) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      double* qn = S + (size_t)K * V;
      double* kn = qn + K;
      double* r = kn + K;
      double* u = r + V;
      const size_t soff = ((size_t)n * Hv + h) * K * V;
      if (initial_state)
        memcpy(S, initial_state + soff, sizeof(double) * K * V);
      else
        memset(S, 0, sizeof(double) * K * V);
      const int hq = h / group;
      for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
        oracle_l2norm(q + ((size_t)t * Hqk + hq) * K, K, use_qk_l2norm, qn);
        oracle_l2norm(k + ((size_t)t * Hqk + hq) * K, K, use_qk_l2norm, kn);
        oracle_step(S, qn, kn, v + ((size_t)t * Hv + h) * V, g[(size_t)t * Hv + h],
                    beta[(size_t)t * Hv + h], scale, K, V, r, u,
                    o + ((size_t)t * Hv + h) * V);
      }
      if (final_state) memcpy(final_state + soff, S, sizeof(double) * K * V);
      free(S);
    }
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * Forward substitution for a unit lower-triangular system (I + A) X = B,
 * A strictly lower (L x L, row stride L), B and X are L x m (row stride m).
 * Row i: X_i = B_i - sum_{j<i} A_ij X_j.  X may alias B.
 */
static void oracle_unit_lower_solve(const double* A, int L, const double* B, int m, double* X) {
  for (int i = 0; i < L; ++i) {
    double* xi = X + (size_t)i * m;
    if (xi != B + (size_t)i * m) memcpy(xi, B + (size_t)i * m, sizeof(double) * m);
    for (int j = 0; j < i; ++j) {
      const double aij = A[(size_t)i * L + j];
      if (aij == 0.0) continue;
      const double* xj = X + (size_t)j * m;
      for (int c = 0; c < m; ++c) xi[c] -= aij * xj[c];
    }
  }
}

/*
 * Chunkwise evaluation, chunk size C, chunks restarting at every sequence start
 * and the last chunk of a sequence possibly partial.  Per chunk of L tokens with
 * in-chunk cumulative log-decay G_i = sum_{m<=i} g_m and state S at chunk entry:
 *
 *   A_ij = beta_i (k_i . k_j) exp(G_i - G_j)             for j < i, else 0
 *   [W | U] = (I + A)^{-1} [diag(beta exp(G)) K | diag(beta) V]
 *   U'  = U - W S
 *   o_i = scale (exp(G_i) q_i^T S + sum_{j<=i} (q_i . k_j) exp(G_i - G_j) U'_j)
 *   S  <- exp(G_{L-1}) S + sum_j exp(G_{L-1} - G_j) k_j U'_j^T
 *
 * This reaches the recurrent result exactly up to rounding whenever every g is
 * finite (a g of -inf makes G_i - G_j undefined here; the recurrent form handles
 * it).
 */
int gdn_oracle_chunked(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, int T_total, int Hqk, int Hv, int K, int V,
                       const int64_t* cu_seqlens, int N, double scale, int use_qk_l2norm,
                       int chunk_size, const double* initial_state, double* o,
                       double* final_state, int nthreads) {
  int err = check_common(Hqk, Hv, K, V, cu_seqlens, N);
  if (err) return err;
  if (chunk_size < 1 || cu_seqlens[N] > T_total || !q || !k || !v || !g || !beta || !o)
    return ORACLE_ERR_ARG;
  const int group = Hv / Hqk;
  const int C = chunk_size;
  int failed = 0;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int n = 0; n < N; ++n) {
    for (int h = 0; h < Hv; ++h) {
      const size_t per = (size_t)K * V          /* S */
                         + (size_t)C * K * 2    /* Qn, Kn */
                         + (size_t)C * 3        /* G, beta, decay-to-end */
                         + (size_t)C * C        /* A */
                         + (size_t)C * (K + V)  /* RHS -> [W | U] */
                         + (size_t)C * V        /* U' */
                         + (size_t)K * V;       /* scratch */
      double* buf = (double*)malloc(sizeof(double) * per);
      if (!buf) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      double* S = buf;
      double* Qn = S + (size_t)K * V;
      double* Kn = Qn + (size_t)C * K;
      double* G = Kn + (size_t)C * K;
      double* bt = G + C;
      double* dend = bt + C;
      double* A = dend + C;
      double* WU = A + (size_t)C * C;
      double* Up = WU + (size_t)C * (K + V);
      const int m = K + V;
      const size_t soff = ((size_t)n * Hv + h) * K * V;
      if (initial_state)
        memcpy(S, initial_state + soff, sizeof(double) * K * V);
      else
        memset(S, 0, sizeof(double) * K * V);
      const int hq = h / group;
      for (int64_t c0 = cu_seqlens[n]; c0 < cu_seqlens[n + 1]; c0 += C) {
        const int64_t rem = cu_seqlens[n + 1] - c0;
        const int L = rem < C ? (int)rem : C;
        double acc = 0.0;
        for (int i = 0; i < L; ++i) {
          const int64_t t = c0 + i;
          oracle_l2norm(q + ((size_t)t * Hqk + hq) * K, K, use_qk_l2norm, Qn + (size_t)i * K);
          oracle_l2norm(k + ((size_t)t * Hqk + hq) * K, K, use_qk_l2norm, Kn + (size_t)i * K);
          acc += g[(size_t)t * Hv + h];
          G[i] = acc;
          bt[i] = beta[(size_t)t * Hv + h];
        }
        for (int i = 0; i < L; ++i) dend[i] = exp(G[L - 1] - G[i]);
        /* A (strictly lower) */
        for (int i = 0; i < L; ++i) {
          for (int j = 0; j < L; ++j) {
            double val = 0.0;
            if (j < i) {
              double kk = 0.0;
              for (int d = 0; d < K; ++d) kk += Kn[(size_t)i * K + d] * Kn[(size_t)j * K + d];
              val = bt[i] * kk * exp(G[i] - G[j]);
            }
            A[(size_t)i * L + j] = val;
          }
        }
        /* right-hand side [diag(beta exp(G)) K | diag(beta) V], then solve in place */
        for (int i = 0; i < L; ++i) {
          const int64_t t = c0 + i;
          const double sw = bt[i] * exp(G[i]);
          for (int d = 0; d < K; ++d) WU[(size_t)i * m + d] = sw * Kn[(size_t)i * K + d];
          const double* vt = v + ((size_t)t * Hv + h) * V;
          for (int e = 0; e < V; ++e) WU[(size_t)i * m + K + e] = bt[i] * vt[e];
        }
        oracle_unit_lower_solve(A, L, WU, m, WU);
        /* U' = U - W S */
        for (int i = 0; i < L; ++i) {
          for (int e = 0; e < V; ++e) {
            double ws = 0.0;
            for (int d = 0; d < K; ++d) ws += WU[(size_t)i * m + d] * S[(size_t)d * V + e];
            Up[(size_t)i * V + e] = WU[(size_t)i * m + K + e] - ws;
          }
        }
        /* outputs */
        for (int i = 0; i < L; ++i) {
          const int64_t t = c0 + i;
          double* ot = o + ((size_t)t * Hv + h) * V;
          const double gi = exp(G[i]);
          for (int e = 0; e < V; ++e) {
            double qs = 0.0;
            for (int d = 0; d < K; ++d) qs += Qn[(size_t)i * K + d] * S[(size_t)d * V + e];
            ot[e] = gi * qs;
          }
          for (int j = 0; j <= i; ++j) {
            double qk = 0.0;
            for (int d = 0; d < K; ++d) qk += Qn[(size_t)i * K + d] * Kn[(size_t)j * K + d];
            const double w = qk * exp(G[i] - G[j]);
            for (int e = 0; e < V; ++e) ot[e] += w * Up[(size_t)j * V + e];
          }
          for (int e = 0; e < V; ++e) ot[e] *= scale;
        }
        /* state to the next chunk */
        const double gl = exp(G[L - 1]);
        for (size_t x = 0; x < (size_t)K * V; ++x) S[x] *= gl;
        for (int j = 0; j < L; ++j)
          for (int d = 0; d < K; ++d) {
            const double kd = dend[j] * Kn[(size_t)j * K + d];
            for (int e = 0; e < V; ++e) S[(size_t)d * V + e] += kd * Up[(size_t)j * V + e];
          }
      }
      if (final_state) memcpy(final_state + soff, S, sizeof(double) * K * V);
      free(buf);
    }
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * One decode token per request on a slot-indexed state cache, updated in place.
 *   state [num_slots, Hv, K, V]; batch_indices [n] (NULL = identity, i.e. the
 *   cache is already in request order).  Slot -1: output row zero, no state
 *   access.  Any other slot outside [0, num_slots): output row zero, no state
 *   access, and the call returns ORACLE_ERR_SLOT after finishing the others.
 * Requests are applied in order i = 0..n-1 for every head, so a repeated slot
 * sees the earlier request's write (the parallel loop runs over heads only).
 */
int gdn_oracle_decode(const double* q, const double* k, const double* v, const double* g,
                      const double* beta, int n, int Hqk, int Hv, int K, int V,
                      double* state, int num_slots, const int64_t* batch_indices,
                      double scale, int use_qk_l2norm, double* o, int nthreads) {
  if (n < 0 || Hqk <= 0 || Hv <= 0 || K <= 0 || V <= 0 || Hv % Hqk != 0 || num_slots < 0)
    return ORACLE_ERR_ARG;
  if (n > 0 && (!q || !k || !v || !g || !beta || !o || !state)) return ORACLE_ERR_ARG;
  if (!batch_indices && n > num_slots) return ORACLE_ERR_ARG;
  const int group = Hv / Hqk;
  int bad_slot = 0, failed = 0;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < Hv; ++h) {
    double* tmp = (double*)malloc(sizeof(double) * (2 * (size_t)K + 2 * (size_t)V));
    if (!tmp) {
#pragma omp atomic write
      failed = 1;
      continue;
    }
    double* qn = tmp;
    double* kn = qn + K;
    double* r = kn + K;
    double* u = r + V;
    const int hq = h / group;
    for (int i = 0; i < n; ++i) {
      const int64_t s = batch_indices ? batch_indices[i] : i;
      double* oi = o + ((size_t)i * Hv + h) * V;
      if (s < 0 || s >= num_slots) {
        for (int e = 0; e < V; ++e) oi[e] = 0.0;
        if (s != -1) {
#pragma omp atomic write
          bad_slot = 1;
        }
        continue;
      }
      double* S = state + ((size_t)s * Hv + h) * K * V;
      oracle_l2norm(q + ((size_t)i * Hqk + hq) * K, K, use_qk_l2norm, qn);
      oracle_l2norm(k + ((size_t)i * Hqk + hq) * K, K, use_qk_l2norm, kn);
      oracle_step(S, qn, kn, v + ((size_t)i * Hv + h) * V, g[(size_t)i * Hv + h],
                  beta[(size_t)i * Hv + h], scale, K, V, r, u, oi);
    }
    free(tmp);
  }
  if (failed) return ORACLE_ERR_NOMEM;
  return bad_slot ? ORACLE_ERR_SLOT : ORACLE_OK;
}

/* Threads an OpenMP region will use (1 without OpenMP). */
int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
  return g_default_threads ? g_default_threads : omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Gated Delta Product: several delta-rule (Householder-type) writes per token.
 * "Megatron-Core API: core.ssm.gated_delta_product", GatedDeltaProductMixer: each token is
 * projected into the V, K, Q, beta and decay terms of a sequence of Householder updates, as
 * many as num_householder (n_h) sets.  The pages print no formula; the plain reading taken:
 * per token t the decay is applied once, before the first write; write j = 0..n_h-1 uses its
 * own key, value and beta; the single query of the token reads the state after the last
 * write:
 *
 *     S   <- exp(g_t) * S
 *     for j = 0 .. n_h - 1:   r = S^T k_tj;  u = beta_tj (v_tj - r);  S <- S + k_tj u^T
 *     o_t  = scale * S^T q_t
 *
 * Layouts (row-major, fp64):
 *   q [T_total, Hqk, K]   k [T_total, n_h, Hqk, K]   v [T_total, n_h, Hv, V]
 *   g [T_total, Hv]       beta [T_total, n_h, Hv]    o [T_total, Hv, V]
 * states, cu_seqlens, the L2 norm, scale and the head map as for gdn_oracle_recurrent; with
 * n_h = 1 this is gdn_oracle_recurrent.
 */

/* The writes of one token on S (decay already applied).  kb, vb, bb point at the token's
 * first key / value / beta of this head; consecutive writes are ks, vs, bs apart. */
static void oracle_product_writes(double* S, const double* kb, size_t ks, const double* vb,
                                  size_t vs, const double* bb, size_t bs, int n_h, int K, int V,
                                  int use_qk_l2norm, double* kn, double* r) {
  for (int j = 0; j < n_h; ++j) {
    oracle_l2norm(kb + (size_t)j * ks, K, use_qk_l2norm, kn);
    const double* vj = vb + (size_t)j * vs;
    const double bj = bb[(size_t)j * bs];
    for (int c = 0; c < V; ++c) r[c] = 0.0;
    for (int i = 0; i < K; ++i)
      for (int c = 0; c < V; ++c) r[c] += S[i * V + c] * kn[i];
    for (int c = 0; c < V; ++c) r[c] = bj * (vj[c] - r[c]);   /* r becomes u */
    for (int i = 0; i < K; ++i)
      for (int c = 0; c < V; ++c) S[i * V + c] += kn[i] * r[c];
  }
}

/* o = scale * S^T qn */
static void oracle_readout(const double* S, const double* qn, double scale, int K, int V,
                           double* o) {
  for (int c = 0; c < V; ++c) o[c] = 0.0;
  for (int i = 0; i < K; ++i)
    for (int c = 0; c < V; ++c) o[c] += S[i * V + c] * qn[i];
  for (int c = 0; c < V; ++c) o[c] *= scale;
}

int gdn_oracle_product(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, int T_total, int n_h, int Hqk, int Hv, int K, int V,
                       const int64_t* cu_seqlens, int N, double scale, int use_qk_l2norm,
                       const double* initial_state, double* o, double* final_state,
                       int nthreads) {
  int err = check_common(Hqk, Hv, K, V, cu_seqlens, N);
  if (err) return err;
  if (n_h < 1 || cu_seqlens[N] > T_total || !q || !k || !v || !g || !beta || !o)
    return ORACLE_ERR_ARG;
  const int group = Hv / Hqk;
  int failed = 0;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int n = 0; n < N; ++n) {
    for (int h = 0; h < Hv; ++h) {
      double* S = (double*)malloc(sizeof(double) * ((size_t)K * V + 2 * K + V));
      if (!S) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      double* qn = S + (size_t)K * V;
      double* kn = qn + K;
      double* r = kn + K;
      const size_t soff = ((size_t)n * Hv + h) * K * V;
      const int hq = h / group;   /* query / key head of value head h */
      if (initial_state)
        memcpy(S, initial_state + soff, sizeof(double) * K * V);
      else
        memset(S, 0, sizeof(double) * K * V);
      for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
        const double a = exp(g[(size_t)t * Hv + h]);
        for (size_t x = 0; x < (size_t)K * V; ++x) S[x] *= a;
        oracle_product_writes(S, k + (((size_t)t * n_h) * Hqk + hq) * K, (size_t)Hqk * K,
                              v + (((size_t)t * n_h) * Hv + h) * V, (size_t)Hv * V,
                              beta + ((size_t)t * n_h) * Hv + h, (size_t)Hv, n_h, K, V,
                              use_qk_l2norm, kn, r);
        oracle_l2norm(q + ((size_t)t * Hqk + hq) * K, K, use_qk_l2norm, qn);
        oracle_readout(S, qn, scale, K, V, o + ((size_t)t * Hv + h) * V);
      }
      if (final_state) memcpy(final_state + soff, S, sizeof(double) * K * V);
      free(S);
    }
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * One token per request of the Gated Delta Product on a slot-indexed cache (the decode step
 * of GatedDeltaProductMixer.ssm_decode): q [n, Hqk, K], k [n, n_h, Hqk, K],
 * v [n, n_h, Hv, V], g [n, Hv], beta [n, n_h, Hv], state [num_slots, Hv, K, V] updated in
 * place, batch_indices [n] (NULL: request i uses slot i; -1: padding, zero output, no state
 * access), o [n, Hv, V].
 */
int gdn_oracle_product_decode(const double* q, const double* k, const double* v,
                              const double* g, const double* beta, int n, int n_h, int Hqk,
                              int Hv, int K, int V, double* state, int num_slots,
                              const int64_t* batch_indices, double scale, int use_qk_l2norm,
                              double* o, int nthreads) {
  if (n < 0 || n_h < 1 || Hqk <= 0 || Hv <= 0 || K <= 0 || V <= 0 || Hv % Hqk) return ORACLE_ERR_ARG;
  if (K > 1024 || V > 1024) return ORACLE_ERR_ARG;
  if (n > 0 && (!q || !k || !v || !g || !beta || !o || !state)) return ORACLE_ERR_ARG;
  const int group = Hv / Hqk;
  int bad = 0;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int i = 0; i < n; ++i) {
    for (int h = 0; h < Hv; ++h) {
      double* oi = o + ((size_t)i * Hv + h) * V;
      const int64_t s = batch_indices ? batch_indices[i] : i;
      if (s < 0 || s >= num_slots) {
        for (int c = 0; c < V; ++c) oi[c] = 0.0;
        if (s != -1) {
#pragma omp atomic write
          bad = 1;
        }
        continue;
      }
      double buf[3 * 1024];
      double *qn = buf, *kn = buf + K, *r = buf + 2 * K;
      double* S = state + ((size_t)s * Hv + h) * K * V;
      const int hq = h / group;
      const double a = exp(g[(size_t)i * Hv + h]);
      for (size_t x = 0; x < (size_t)K * V; ++x) S[x] *= a;
      oracle_product_writes(S, k + (((size_t)i * n_h) * Hqk + hq) * K, (size_t)Hqk * K,
                            v + (((size_t)i * n_h) * Hv + h) * V, (size_t)Hv * V,
                            beta + ((size_t)i * n_h) * Hv + h, (size_t)Hv, n_h, K, V,
                            use_qk_l2norm, kn, r);
      oracle_l2norm(q + ((size_t)i * Hqk + hq) * K, K, use_qk_l2norm, qn);
      oracle_readout(S, qn, scale, K, V, oi);
    }
  }
  return bad ? ORACLE_ERR_SLOT : ORACLE_OK;
}

/*
 * Backward of the gated delta rule (the reverse-mode adjoint of gdn_oracle_recurrent).  For a
 * loss with gradients d_o [T_total, Hv, V] on the outputs and d_final [N, Hv, K, V] on the
 * final states (NULL: zero), returns the gradients of every input:
 *   dq, dk [T_total, Hqk, K] (summed over the value heads sharing a query/key head),
 *   dv [T_total, Hv, V], dg, dbeta [T_total, Hv], d_initial [N, Hv, K, V] (may be NULL).
 *
 * With S_{t-1} the state before token t, a = exp(g_t), hat-q / hat-k the (optionally)
 * normalised vectors, r = a S_{t-1}^T k, u = beta (v - r), S_t = a S_{t-1} + k u^T and
 * o_t = scale S_t^T q, walking t backwards with dS the gradient of S_t:
 *   dS   += scale q do^T                    dq   = scale (a S_{t-1} do + (u . do) k)
 *   du    = dS^T k                          dk   = dS u
 *   dbeta = du . (v - r)                    dv   = beta du          dr = -beta du
 *   dk   += a S_{t-1} dr                    da   = <dS, S_{t-1}> + (S_{t-1}^T k) . dr
 *   dg    = a da                            dS  <- a (dS + k dr^T)     (the gradient of S_{t-1})
 * then the L2 norm's Jacobian x -> x / sqrt(|x|^2 + eps) maps d(hat-x) to dx.  The states are
 * recomputed forward first (stored per token).
 */
static void oracle_norm_backward(const double* x, const double* dxh, int n, int use, double* dx) {
  if (!use) {
    memcpy(dx, dxh, (size_t)n * sizeof(double));
    return;
  }
  double ss = 0.0, xd = 0.0;
  for (int i = 0; i < n; ++i) { ss += x[i] * x[i]; xd += x[i] * dxh[i]; }
  const double rho = 1.0 / sqrt(ss + GDN_ORACLE_L2_EPS);
  for (int i = 0; i < n; ++i) dx[i] = rho * dxh[i] - rho * rho * rho * xd * x[i];
}

int gdn_oracle_backward(const double* q, const double* k, const double* v, const double* g,
                        const double* beta, int T_total, int Hqk, int Hv, int K, int V,
                        const int64_t* cu_seqlens, int N, double scale, int use_qk_l2norm,
                        const double* initial_state, const double* d_o, const double* d_final,
                        double* dq, double* dk, double* dv, double* dg, double* dbeta,
                        double* d_initial, int nthreads) {
  int err = check_common(Hqk, Hv, K, V, cu_seqlens, N);
  if (err) return err;
  if (cu_seqlens[N] > T_total || !q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv ||
      !dg || !dbeta)
    return ORACLE_ERR_ARG;
  const int group = Hv / Hqk;
  int failed = 0;
  memset(dq, 0, sizeof(double) * (size_t)T_total * Hqk * K);
  memset(dk, 0, sizeof(double) * (size_t)T_total * Hqk * K);
  set_threads(nthreads);
  /* one task per (sequence, query/key head): its value heads add into the same dq / dk rows */
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int n = 0; n < N; ++n) {
    for (int hq = 0; hq < Hqk; ++hq) {
      const int64_t t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - cu_seqlens[n];
      const size_t KV = (size_t)K * V;
      double* states = (double*)malloc(sizeof(double) * (KV * ((size_t)L + 2) + 6 * (size_t)K + 4 * (size_t)V));
      if (!states) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      double* dS = states + KV * (size_t)(L + 1);   /* states[t] = S before token t0 + t */
      double* qn = dS + KV;
      double* kn = qn + K;
      double* dqh = kn + K;
      double* dkh = dqh + K;
      double* tmpk = dkh + K;
      double* tmpk2 = tmpk + K;
      double* r = tmpk2 + K;
      double* u = r + V;
      double* du = u + V;
      double* dr = du + V;
      for (int h = hq * group; h < (hq + 1) * group; ++h) {
        const size_t soff = ((size_t)n * Hv + h) * KV;
        if (initial_state)
          memcpy(states, initial_state + soff, sizeof(double) * KV);
        else
          memset(states, 0, sizeof(double) * KV);
        /* forward: states[t + 1] = S after token t */
        for (int64_t t = 0; t < L; ++t) {
          const int64_t tt = t0 + t;
          const double* Sp = states + KV * (size_t)t;
          double* Sn = states + KV * (size_t)(t + 1);
          oracle_l2norm(k + ((size_t)tt * Hqk + hq) * K, K, use_qk_l2norm, kn);
          const double a = exp(g[(size_t)tt * Hv + h]);
          const double bt = beta[(size_t)tt * Hv + h];
          const double* vt = v + ((size_t)tt * Hv + h) * V;
          for (int c = 0; c < V; ++c) r[c] = 0.0;
          for (int i = 0; i < K; ++i)
            for (int c = 0; c < V; ++c) r[c] += a * Sp[i * V + c] * kn[i];
          for (int c = 0; c < V; ++c) u[c] = bt * (vt[c] - r[c]);
          for (int i = 0; i < K; ++i)
            for (int c = 0; c < V; ++c) Sn[i * V + c] = a * Sp[i * V + c] + kn[i] * u[c];
        }
        if (d_final)
          memcpy(dS, d_final + soff, sizeof(double) * KV);
        else
          memset(dS, 0, sizeof(double) * KV);
        for (int64_t t = L - 1; t >= 0; --t) {
          const int64_t tt = t0 + t;
          const double* Sp = states + KV * (size_t)t;
          const double* qraw = q + ((size_t)tt * Hqk + hq) * K;
          const double* kraw = k + ((size_t)tt * Hqk + hq) * K;
          oracle_l2norm(qraw, K, use_qk_l2norm, qn);
          oracle_l2norm(kraw, K, use_qk_l2norm, kn);
          const double a = exp(g[(size_t)tt * Hv + h]);
          const double bt = beta[(size_t)tt * Hv + h];
          const double* vt = v + ((size_t)tt * Hv + h) * V;
          const double* dot = d_o + ((size_t)tt * Hv + h) * V;
          /* recompute S_{t-1}^T k (kept apart from the decay: r = a S_{t-1}^T k) and u */
          for (int c = 0; c < V; ++c) r[c] = 0.0;
          for (int i = 0; i < K; ++i)
            for (int c = 0; c < V; ++c) r[c] += Sp[i * V + c] * kn[i];
          for (int c = 0; c < V; ++c) u[c] = bt * (vt[c] - a * r[c]);
          /* read-out */
          for (int i = 0; i < K; ++i)
            for (int c = 0; c < V; ++c) dS[i * V + c] += scale * qn[i] * dot[c];
          double udo = 0.0;
          for (int c = 0; c < V; ++c) udo += u[c] * dot[c];
          for (int i = 0; i < K; ++i) {
            double s = 0.0;
            for (int c = 0; c < V; ++c) s += Sp[i * V + c] * dot[c];
            dqh[i] = scale * (a * s + udo * kn[i]);
          }
          /* rank-1 write and the delta-rule read */
          for (int c = 0; c < V; ++c) {
            double s = 0.0;
            for (int i = 0; i < K; ++i) s += dS[i * V + c] * kn[i];
            du[c] = s;
          }
          double db = 0.0;
          for (int c = 0; c < V; ++c) {
            db += du[c] * (vt[c] - a * r[c]);
            dv[((size_t)tt * Hv + h) * V + c] = bt * du[c];
            dr[c] = -bt * du[c];
          }
          dbeta[(size_t)tt * Hv + h] = db;
          double da = 0.0;
          for (int i = 0; i < K; ++i) {
            double s1 = 0.0, s2 = 0.0;
            for (int c = 0; c < V; ++c) {
              s1 += dS[i * V + c] * u[c];
              s2 += Sp[i * V + c] * dr[c];
              da += dS[i * V + c] * Sp[i * V + c];
            }
            dkh[i] = s1 + a * s2;
          }
          for (int c = 0; c < V; ++c) da += r[c] * dr[c];
          dg[(size_t)tt * Hv + h] = a * da;
          for (int i = 0; i < K; ++i)
            for (int c = 0; c < V; ++c) dS[i * V + c] = a * (dS[i * V + c] + kn[i] * dr[c]);
          oracle_norm_backward(qraw, dqh, K, use_qk_l2norm, tmpk);
          oracle_norm_backward(kraw, dkh, K, use_qk_l2norm, tmpk2);
          for (int i = 0; i < K; ++i) {
            dq[((size_t)tt * Hqk + hq) * K + i] += tmpk[i];
            dk[((size_t)tt * Hqk + hq) * K + i] += tmpk2[i];
          }
        }
        if (d_initial) memcpy(d_initial + soff, dS, sizeof(double) * KV);
      }
      free(states);
    }
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}
