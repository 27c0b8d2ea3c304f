// gdn_gates_bwd.cu -- the backward of the chunked rule through the fused gates.
//
// The GDN mixer derives "the per-head log-decay g and the write strength beta" from its gate
// features a, b and the per-head parameters A_log, dt_bias ("Megatron-Core API:
// core.ssm.gated_delta_net.gdn", GatedDeltaNet._compute_gates):
//     g = -exp(A_log[h]) softplus(a + dt_bias[h]),     beta = sigmoid(b).
// The backward materialises g and beta (fp32, the expressions the fused forward evaluates),
// runs the chunked backward on them for dg and dbeta, and applies the chain rule:
//     da = dg (-exp(A_log) sigmoid(a + dt_bias)),      db = dbeta beta (1 - beta),
//     dA_log[h] = sum over tokens of dg g,             ddt_bias[h] = sum over tokens of da.
// The two sums are deterministic: each CTA reduces a fixed token range in a fixed order into
// a partial per head, and one CTA adds the partials in block order (fp64).
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPartials = 1024;

__global__ void __launch_bounds__(kThreads) gates_materialise_kernel(GateArgs ga, long long n_elem,
                                                                     int Hv, float* g, float* beta) {
  for (long long i = blockIdx.x * (long long)kThreads + threadIdx.x; i < n_elem;
       i += (long long)gridDim.x * kThreads) {
    const int h = (int)(i % Hv);
    float gv, bv;
    fused_gates(ga, (size_t)i, h, &gv, &bv);
    g[i] = gv;
    beta[i] = bv;
  }
}

// CTA j: tokens [j tpb, (j + 1) tpb) of the [T_total, Hv] arrays; thread (r, h) = (tid / Hv,
// tid % Hv) takes tokens r, r + R, ... of the range (R = kThreads / Hv), so every access is
// coalesced and every sum runs in a fixed order.
__global__ void __launch_bounds__(kThreads) gates_bwd_kernel(GateArgs ga, const float* dg,
                                                             const float* dbeta, long long T_total,
                                                             int Hv, long long tpb, float* da,
                                                             float* db, float* partial) {
  __shared__ float red[2][kThreads];
  const int tid = threadIdx.x;
  const int R = kThreads / Hv;
  const int r = tid / Hv, h = tid % Hv;
  const long long t0 = blockIdx.x * tpb, t1 = min(T_total, t0 + tpb);
  float sA = 0.f, sD = 0.f;
  if (r < R) {
    const float eA = expf(ga.A_log[h]);
    const float bias = ga.dt_bias[h];
    for (long long t = t0 + r; t < t1; t += R) {
      const size_t i = (size_t)t * Hv + h;
      const float x = load_elem(ga.a, i, ga.ab_dtype) + bias;
      const float g = -eA * softplus_f(x);
      const float dav = dg[i] * (-eA * sigmoid_f(x));
      const float be = sigmoid_f(load_elem(ga.b, i, ga.ab_dtype));
      da[i] = dav;
      db[i] = dbeta[i] * be * (1.f - be);
      sA = fmaf(dg[i], g, sA);
      sD += dav;
    }
  }
  red[0][tid] = sA;
  red[1][tid] = sD;
  __syncthreads();
  if (tid < Hv) {
    float a0 = 0.f, a1 = 0.f;
    for (int rr = 0; rr < R; ++rr) {
      a0 += red[0][rr * Hv + tid];
      a1 += red[1][rr * Hv + tid];
    }
    partial[((size_t)blockIdx.x * Hv + tid) * 2 + 0] = a0;
    partial[((size_t)blockIdx.x * Hv + tid) * 2 + 1] = a1;
  }
}

__global__ void __launch_bounds__(kThreads) gates_param_kernel(const float* partial, int nblocks, int Hv,
                                                               float* dA_log, float* ddt_bias) {
  for (int h = threadIdx.x; h < Hv; h += kThreads) {
    double s0 = 0.0, s1 = 0.0;
    for (int j = 0; j < nblocks; ++j) {
      s0 += partial[((size_t)j * Hv + h) * 2 + 0];
      s1 += partial[((size_t)j * Hv + h) * 2 + 1];
    }
    dA_log[h] = (float)s0;
    ddt_bias[h] = (float)s1;
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t gates_bwd_extra_bytes(long long T_total, int Hv) {
  const size_t elems = (size_t)T_total * Hv;
  return 4 * align256(elems * sizeof(float)) + align256((size_t)kMaxPartials * Hv * 2 * sizeof(float));
}

cudaError_t launch_gates_materialise(const GateArgs& ga, long long T_total, int Hv, float* g,
                                     float* beta, cudaStream_t stream) {
  const long long n = T_total * Hv;
  if (n <= 0) return cudaSuccess;
  const long long blocks = std::min<long long>((n + kThreads - 1) / kThreads, 4096);
  gates_materialise_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(ga, n, Hv, g, beta);
  return cudaGetLastError();
}

cudaError_t launch_gates_bwd(const GateArgs& ga, const float* dg, const float* dbeta,
                             long long T_total, int Hv, float* da, float* db, float* dA_log,
                             float* ddt_bias, float* partial, cudaStream_t stream) {
  if (Hv > kThreads) return cudaErrorInvalidValue;
  int nblocks = 1;
  long long tpb = T_total > 0 ? T_total : 1;
  if (T_total > 0) {
    nblocks = (int)std::min<long long>(kMaxPartials, (T_total + 63) / 64);
    tpb = (T_total + nblocks - 1) / nblocks;
    nblocks = (int)((T_total + tpb - 1) / tpb);
    gates_bwd_kernel<<<nblocks, kThreads, 0, stream>>>(ga, dg, dbeta, T_total, Hv, tpb, da, db,
                                                        partial);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  } else {
    nblocks = 0;
  }
  gates_param_kernel<<<1, kThreads, 0, stream>>>(partial, nblocks, Hv, dA_log, ddt_bias);
  return cudaGetLastError();
}

}  // namespace gdn
