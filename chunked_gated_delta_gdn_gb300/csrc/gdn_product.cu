// gdn_product.cu -- the Gated Delta Product on top of the chunk kernels.
//
// The product ("Megatron-Core API: core.ssm.gated_delta_product", GatedDeltaProductMixer:
// each token drives a sequence of Householder-type delta-rule writes) applies, per token t,
// the decay exp(g_t) once, then n_h writes with their own key, value and beta, then reads
// the state with the token's single query.  With the writes laid out [T, n_h, ...] this is
// exactly the gated delta rule over the T * n_h writes in order, provided the decay of each
// token sits on its first write (g' = g_t there, 0 on the others) and the query on its last
// (q' = q_t there, 0 on the others; the zero queries' outputs are discarded).  k, v and beta
// already have that layout, so only q', g', the scaled cu_seqlens and the output gather
// need work; these kernels do it, and the chunk kernels run on the write sequence.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// q' [T * n_h, Hqk * K] in 16-byte units: the token's query on its last write, zeros before.
__global__ void expand_q_kernel(const uint4* __restrict__ q, uint4* __restrict__ qe,
                                long long units_total, int units_per_row, int n_h) {
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units_total;
       u += (long long)gridDim.x * blockDim.x) {
    const long long row = u / units_per_row;
    const int col = (int)(u - row * units_per_row);
    const long long t = row / n_h;
    const int j = (int)(row - t * n_h);
    qe[u] = (j == n_h - 1) ? q[t * units_per_row + col] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// g' [T * n_h, Hv]: the token's log-decay on its first write, zeros after.
__global__ void expand_g_kernel(const float* __restrict__ g, float* __restrict__ ge,
                                long long total, int Hv, int n_h) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / Hv;
    const int h = (int)(e - row * Hv);
    const long long t = row / n_h;
    const int j = (int)(row - t * n_h);
    ge[e] = (j == 0) ? g[t * Hv + h] : 0.f;
  }
}

__global__ void scale_cu_kernel(const int32_t* __restrict__ cu, int32_t* __restrict__ cue,
                                int count, int n_h) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) cue[i] = cu[i] * n_h;
}

// o [T, Hv * V] in 16-byte units from row t * n_h + n_h - 1 of o' [T * n_h, Hv * V].
__global__ void gather_o_kernel(const uint4* __restrict__ oe, uint4* __restrict__ o,
                                long long units_total, int units_per_row, int n_h) {
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units_total;
       u += (long long)gridDim.x * blockDim.x) {
    const long long t = u / units_per_row;
    const int col = (int)(u - t * units_per_row);
    o[u] = oe[(t * n_h + n_h - 1) * units_per_row + col];
  }
}

unsigned grid_for(long long work) {
  const long long b = (work + kThreads - 1) / kThreads;
  return (unsigned)(b < 1 ? 1 : (b > 152LL * 16 ? 152LL * 16 : b));   // grid-stride beyond this
}

}  // namespace

cudaError_t launch_product_expand(const void* q, const float* g, void* q_exp, float* g_exp,
                                  const int32_t* cu, int32_t* cu_exp, long long T_total, int n_h,
                                  int Hqk, int Hv, int K, int io_dtype, int num_seqs,
                                  cudaStream_t stream) {
  if (T_total > 0) {
    const int upr = (int)(((long long)Hqk * K * (io_dtype == GDN_BF16 ? 2 : 4)) / 16);
    const long long units = T_total * n_h * upr;
    expand_q_kernel<<<grid_for(units), kThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(q), reinterpret_cast<uint4*>(q_exp), units, upr, n_h);
    const long long ge = T_total * n_h * Hv;
    expand_g_kernel<<<grid_for(ge), kThreads, 0, stream>>>(g, g_exp, ge, Hv, n_h);
  }
  if (cu)
    scale_cu_kernel<<<(num_seqs + 1 + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
        cu, cu_exp, num_seqs + 1, n_h);
  return cudaGetLastError();
}

cudaError_t launch_product_gather(const void* o_exp, void* o, long long T_total, int n_h, int Hv,
                                  int V, int io_dtype, cudaStream_t stream) {
  if (T_total <= 0) return cudaSuccess;
  const int upr = (int)(((long long)Hv * V * (io_dtype == GDN_BF16 ? 2 : 4)) / 16);
  const long long units = T_total * upr;
  gather_o_kernel<<<grid_for(units), kThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(o_exp), reinterpret_cast<uint4*>(o), units, upr, n_h);
  return cudaGetLastError();
}

}  // namespace gdn
