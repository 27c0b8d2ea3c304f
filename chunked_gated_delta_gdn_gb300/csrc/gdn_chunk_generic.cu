// gdn_chunk_generic.cu -- chunkwise gated delta rule on the fp32 CUDA cores.
//
// Serves every shape and dtype gdn_chunk_fwd accepts (in particular fp32 I/O,
// whose 1e-4 error budget rules out bf16 / tf32 tensor-core operands).  Four
// launches on the caller's stream, all graph-capturable:
//
//   1. chunk table  -- from cu_seqlens on the device: chunk_off[n] = number of
//                      64-token chunks before sequence n (no host sync; the
//                      later grids are sized by the upper bound T/64 + N).
//   2. prep         -- per (chunk, value head): in-chunk cumulative log-decay G,
//                      q/k L2 norm, A = strict_lower(diag(beta) K K^T * exp(G_i - G_j)),
//                      and the UT-transform solve (I + A) [W | U] =
//                      [diag(beta exp(G)) K | diag(beta) V] by forward substitution.
//   3. state        -- per (sequence, value head, 32-column tile of V), serial
//                      over chunks: records the entry state, U' = U - W S,
//                      S <- exp(G_last) S + (diag(exp(G_last - G)) K)^T U'.
//   4. output       -- per (chunk, value head, 32-column tile):
//                      o = scale (diag(exp G) Q S + (Q K^T * exp(G_i - G_j) * [j <= i]) U').
//
// The chunk length 64 is the inference kernels' fixed chunking
// ("Megatron-Core API: core.ssm.gated_delta_product", ssm_inference_chunk_size);
// the argument set is torch_chunk_gated_delta_rule's ("Megatron-Core API:
// core.ssm.gated_delta_net.gdn").  Intermediates live in the caller's workspace.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int kVT = 32;  // V columns per CTA in the state / output kernels

struct WsLayout {
  int32_t* chunk_off;  // [N + 2]: chunk offsets, then a validity flag
  float* W;            // [NC][Hv][C][K]
  float* U;            // [NC][Hv][C][V]   (U, then U')
  float* G;            // [NC][Hv][C]
  float* S;            // [NC][Hv][K][V]   state at chunk entry
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline WsLayout ws_layout(void* base, long long NC, int N, int Hv, int K,
                                              int V, size_t* total) {
  WsLayout w;
  char* p = reinterpret_cast<char*>(base);
  size_t off = 0;
  w.chunk_off = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + sizeof(int32_t) * (size_t)(N + 2));
  w.W = reinterpret_cast<float*>(p + off);
  off = align256(off + sizeof(float) * (size_t)NC * Hv * C * K);
  w.U = reinterpret_cast<float*>(p + off);
  off = align256(off + sizeof(float) * (size_t)NC * Hv * C * V);
  w.G = reinterpret_cast<float*>(p + off);
  off = align256(off + sizeof(float) * (size_t)NC * Hv * C);
  w.S = reinterpret_cast<float*>(p + off);
  off = align256(off + sizeof(float) * (size_t)NC * Hv * K * V);
  if (total) *total = off;
  return w;
}

// Token range of sequence n (cu_seqlens on the device, or uniform rows of T).
__device__ __forceinline__ void seq_bounds(const ChunkArgs& a, int n, int* bos, int* eos) {
  if (a.cu_seqlens) {
    *bos = a.cu_seqlens[n];
    *eos = a.cu_seqlens[n + 1];
  } else {
    *bos = n * a.T;
    *eos = (n + 1) * a.T;
  }
}

// Slot of sequence n when a slot cache is used: -1 padding / invalid, else slot.
__device__ __forceinline__ int seq_slot(const ChunkArgs& a, int n) {
  if (!a.state_indices) return n;
  const int s = a.state_indices[n];
  return (s >= 0 && s < a.num_slots) ? s : -1;
}

// ---------------------------------------------------------------- 1. chunk table
// cu_seqlens must start at 0, never decrease and end at or before the token
// count; otherwise every sequence is treated as empty (nothing is computed or
// written), GDN_DEV_BAD_CU_SEQLENS is reported, and chunk_off[N + 1] = 0 tells
// the later kernels to skip.  This bounds the chunk count by T/64 + N, the size
// the workspace was laid out for.
__global__ void chunk_table_kernel(const ChunkArgs a, int32_t* chunk_off) {
  __shared__ int32_t carry;
  __shared__ int bad;
  __shared__ int32_t scan[1024];
  const int N = a.num_seqs;
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  if (threadIdx.x == 0) { carry = 0; bad = 0; }
  __syncthreads();
  if (a.cu_seqlens) {
    for (int n = threadIdx.x; n <= N; n += blockDim.x) {
      const int x = a.cu_seqlens[n];
      const bool ok = (n == 0) ? (x == 0) : (x >= a.cu_seqlens[n - 1] && x <= T_total);
      if (!ok) bad = 1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && bad) report(a.dev_status, GDN_DEV_BAD_CU_SEQLENS);
  for (int base = 0; base < N; base += blockDim.x) {
    const int n = base + threadIdx.x;
    int cnt = 0;
    if (n < N) {
      int bos, eos;
      seq_bounds(a, n, &bos, &eos);
      if (!bad) cnt = (eos - bos + C - 1) / C;
      if (a.state_indices) {
        const int s = a.state_indices[n];
        if (s < -1 || s >= a.num_slots) report(a.dev_status, GDN_DEV_BAD_SLOT);
      }
    }
    scan[threadIdx.x] = cnt;
    __syncthreads();
    for (int d = 1; d < (int)blockDim.x; d <<= 1) {  // inclusive Hillis-Steele scan
      const int x = threadIdx.x >= d ? scan[threadIdx.x - d] : 0;
      __syncthreads();
      scan[threadIdx.x] += x;
      __syncthreads();
    }
    if (n < N) chunk_off[n + 1] = carry + scan[threadIdx.x];
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry += scan[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    chunk_off[0] = 0;
    chunk_off[N + 1] = bad ? 0 : 1;
  }
}

// Chunk c -> (sequence n, first token, length); false when c is past the end.
__device__ __forceinline__ bool locate_chunk(const ChunkArgs& a, const int32_t* chunk_off, int c,
                                             int* n_out, int* t0, int* L) {
  const int N = a.num_seqs;
  if (c >= chunk_off[N]) return false;
  int lo = 0, hi = N - 1;  // largest n with chunk_off[n] <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
  }
  int bos, eos;
  seq_bounds(a, lo, &bos, &eos);
  *n_out = lo;
  *t0 = bos + (c - chunk_off[lo]) * C;
  *L = min(C, eos - *t0);
  return true;
}

// Load rows [t0, t0 + L) of a [T, H, D] tensor (head hd) into dst[C][D] fp32,
// L2-normalised per row when asked; rows >= L are zero.  Needs a __syncthreads
// after return before the tile is read.
__device__ void load_rows(const void* src, int dtype, int t0, int L, int H, int hd, int D,
                          bool l2, float* dst) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < C; r += kThreads / 32) {
    float* d = dst + r * D;
    if (r >= L) {
      for (int e = lane; e < D; e += 32) d[e] = 0.f;
      continue;
    }
    const size_t base = ((size_t)(t0 + r) * H + hd) * D;
    float ss = 0.f;
    for (int e = lane; e < D; e += 32) {
      const float x = load_elem(src, base + e, dtype);
      d[e] = x;
      ss += x * x;
    }
    if (l2) {
      ss = warp_sum(ss);
      const float rn = 1.0f / sqrtf(ss + kL2Eps);
      for (int e = lane; e < D; e += 32) d[e] *= rn;
    }
  }
}

// g and beta of element i = token * Hv + h: given, or computed from the raw gate
// features (fused gates).
__device__ __forceinline__ void gate_values(const ChunkArgs& a, size_t i, int h, float* g,
                                            float* beta) {
  if (a.gates.mode == kGatesFused) {
    fused_gates(a.gates, i, h, g, beta);
  } else {
    *g = a.g[i];
    *beta = load_elem(a.beta, i, a.beta_dtype);
  }
}

// In-chunk inclusive cumsum of g (rows >= L get the last valid value) and beta
// (zero for rows >= L).  Done by warp 0.
__device__ void load_gates(const ChunkArgs& a, int t0, int L, int h, float* G, float* bt) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
  if (lane < L) gate_values(a, (size_t)(t0 + lane) * a.Hv + h, h, &g0, &b0);
  if (lane + 32 < L) gate_values(a, (size_t)(t0 + lane + 32) * a.Hv + h, h, &g1, &b1);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float x0 = __shfl_up_sync(0xffffffffu, g0, o);
    const float x1 = __shfl_up_sync(0xffffffffu, g1, o);
    if (lane >= o) { g0 += x0; g1 += x1; }
  }
  g1 += __shfl_sync(0xffffffffu, g0, 31);
  G[lane] = g0;
  G[lane + 32] = g1;
  bt[lane] = b0;
  bt[lane + 32] = b1;
}

// ---------------------------------------------------------------- 2. prep
// smem: Kn[C][K], X[C][K + V], A[C][C], G[C], bt[C]
__global__ void __launch_bounds__(kThreads) chunk_prep_kernel(const ChunkArgs a, WsLayout ws) {
  extern __shared__ float smem[];
  const int K = a.K, V = a.V, M = K + V;
  float* Kn = smem;
  float* X = Kn + C * K;
  float* A = X + C * M;
  float* G = A + C * C;
  float* bt = G + C;
  const int c = blockIdx.x, h = blockIdx.y;
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  if (a.state_indices && seq_slot(a, n) < 0) return;
  const int hq = h / (a.Hv / a.Hqk);
  load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Kn);
  load_gates(a, t0, L, h, G, bt);
  __syncthreads();
  // A (strictly lower) and the right-hand side [diag(beta exp G) Kn | diag(beta) V].
  for (int e = threadIdx.x; e < C * C; e += kThreads) {
    const int i = e / C, j = e - i * C;
    float val = 0.f;
    if (j < i) {
      float kk = 0.f;
      for (int d = 0; d < K; ++d) kk += Kn[i * K + d] * Kn[j * K + d];
      val = bt[i] * kk * expf(G[i] - G[j]);
    }
    A[e] = val;
  }
  for (int e = threadIdx.x; e < C * M; e += kThreads) {
    const int i = e / M, col = e - i * M;
    float x = 0.f;
    if (i < L) {
      x = col < K ? bt[i] * expf(G[i]) * Kn[i * K + col]
                  : bt[i] * load_elem(a.v, ((size_t)(t0 + i) * a.Hv + h) * V + (col - K), a.io_dtype);
    }
    X[e] = x;
  }
  __syncthreads();
  // Forward substitution, one column of [W | U] per thread (columns are
  // independent, so no barrier is needed inside the sweep).
  const size_t ch = (size_t)c * a.Hv + h;
  for (int col = threadIdx.x; col < M; col += kThreads) {
    for (int i = 1; i < L; ++i) {
      float acc = X[i * M + col];
      for (int j = 0; j < i; ++j) acc -= A[i * C + j] * X[j * M + col];
      X[i * M + col] = acc;
    }
    if (col < K) {
      float* Wd = ws.W + ch * C * K;
      for (int i = 0; i < C; ++i) Wd[i * K + col] = X[i * M + col];
    } else {
      float* Ud = ws.U + ch * C * V;
      for (int i = 0; i < C; ++i) Ud[i * V + (col - K)] = X[i * M + col];
    }
  }
  if (threadIdx.x < C) ws.G[ch * C + threadIdx.x] = G[threadIdx.x];
}

// ---------------------------------------------------------------- 3. state
// Per (sequence, head, 32-column tile).  smem: S[K][32], W[C][K], U[C][32], Kn[C][K], G[C]
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(const ChunkArgs a, WsLayout ws) {
  extern __shared__ float smem[];
  const int K = a.K, V = a.V;
  float* S = smem;
  float* W = S + K * kVT;
  float* U = W + C * K;
  float* Kn = U + C * kVT;
  float* G = Kn + C * K;
  const int n = blockIdx.x, h = blockIdx.y, c0 = blockIdx.z * kVT;
  const int vt = min(kVT, V - c0);
  const int slot = seq_slot(a, n);
  if (a.state_indices && slot < 0) return;
  if (!ws.chunk_off[a.num_seqs + 1]) return;   // invalid cu_seqlens: nothing to do
  int bos, eos;
  seq_bounds(a, n, &bos, &eos);
  const int hq = h / (a.Hv / a.Hqk);
  const size_t st_off = ((size_t)slot * a.Hv + h) * K * V;
  for (int e = threadIdx.x; e < K * kVT; e += kThreads) {
    const int d = e / kVT, cc = e - d * kVT;
    S[e] = (a.initial_state && cc < vt) ? a.initial_state[st_off + (size_t)d * V + c0 + cc] : 0.f;
  }
  const int first = ws.chunk_off[n];
  for (int t0 = bos, ci = first; t0 < eos; t0 += C, ++ci) {
    const int L = min(C, eos - t0);
    const size_t ch = (size_t)ci * a.Hv + h;
    __syncthreads();
    float* Srec = ws.S + ch * K * V;
    for (int e = threadIdx.x; e < K * kVT; e += kThreads) {
      const int d = e / kVT, cc = e - d * kVT;
      if (cc < vt) Srec[(size_t)d * V + c0 + cc] = S[e];
    }
    const float* Wg = ws.W + ch * C * K;
    for (int e = threadIdx.x; e < C * K; e += kThreads) W[e] = Wg[e];
    float* Ug = ws.U + ch * C * V;
    for (int e = threadIdx.x; e < C * kVT; e += kThreads) {
      const int i = e / kVT, cc = e - i * kVT;
      U[e] = cc < vt ? Ug[(size_t)i * V + c0 + cc] : 0.f;
    }
    if (threadIdx.x < C) G[threadIdx.x] = ws.G[ch * C + threadIdx.x];
    load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Kn);
    __syncthreads();
    // U' = U - W S   (rows >= L of W and U are zero, so U' is zero there)
    for (int e = threadIdx.x; e < C * kVT; e += kThreads) {
      const int i = e / kVT, cc = e - i * kVT;
      float acc = U[e];
      for (int d = 0; d < K; ++d) acc -= W[i * K + d] * S[d * kVT + cc];
      U[e] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < C * kVT; e += kThreads) {
      const int i = e / kVT, cc = e - i * kVT;
      if (cc < vt) Ug[(size_t)i * V + c0 + cc] = U[e];
    }
    // S <- exp(G_last) S + sum_t exp(G_last - G_t) Kn_t U'_t
    const float gl = G[L - 1];
    const float dl = expf(gl);
    for (int e = threadIdx.x; e < K * kVT; e += kThreads) {
      const int d = e / kVT, cc = e - d * kVT;
      float acc = dl * S[e];
      for (int t = 0; t < L; ++t) acc += expf(gl - G[t]) * Kn[t * K + d] * U[t * kVT + cc];
      S[e] = acc;
    }
  }
  __syncthreads();
  if (a.final_state) {
    for (int e = threadIdx.x; e < K * kVT; e += kThreads) {
      const int d = e / kVT, cc = e - d * kVT;
      if (cc < vt) a.final_state[st_off + (size_t)d * V + c0 + cc] = S[e];
    }
  }
}

// ---------------------------------------------------------------- 4. output
// Per (chunk, head, 32-column tile).  smem: Qn[C][K], Kn[C][K], S[K][32], U[C][32], P[C][C], G[C]
__global__ void __launch_bounds__(kThreads) chunk_output_kernel(const ChunkArgs a, WsLayout ws) {
  extern __shared__ float smem[];
  const int K = a.K, V = a.V;
  float* Qn = smem;
  float* Kn = Qn + C * K;
  float* S = Kn + C * K;
  float* U = S + K * kVT;
  float* P = U + C * kVT;
  float* G = P + C * C;
  const int c = blockIdx.x, h = blockIdx.y, c0 = blockIdx.z * kVT;
  const int vt = min(kVT, V - c0);
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  if (a.state_indices && seq_slot(a, n) < 0) {  // padding sequence: zero rows
    for (int e = threadIdx.x; e < L * vt; e += kThreads) {
      const int i = e / vt, cc = e - i * vt;
      store_elem(a.o, ((size_t)(t0 + i) * a.Hv + h) * V + c0 + cc, 0.f, a.io_dtype);
    }
    return;
  }
  const int hq = h / (a.Hv / a.Hqk);
  const size_t ch = (size_t)c * a.Hv + h;
  load_rows(a.q, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Qn);
  load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Kn);
  const float* Sg = ws.S + ch * K * V;
  for (int e = threadIdx.x; e < K * kVT; e += kThreads) {
    const int d = e / kVT, cc = e - d * kVT;
    S[e] = cc < vt ? Sg[(size_t)d * V + c0 + cc] : 0.f;
  }
  const float* Ug = ws.U + ch * C * V;
  for (int e = threadIdx.x; e < C * kVT; e += kThreads) {
    const int i = e / kVT, cc = e - i * kVT;
    U[e] = cc < vt ? Ug[(size_t)i * V + c0 + cc] : 0.f;
  }
  if (threadIdx.x < C) G[threadIdx.x] = ws.G[ch * C + threadIdx.x];
  __syncthreads();
  for (int e = threadIdx.x; e < C * C; e += kThreads) {
    const int i = e / C, j = e - i * C;
    float val = 0.f;
    if (j <= i && i < L) {
      float qk = 0.f;
      for (int d = 0; d < K; ++d) qk += Qn[i * K + d] * Kn[j * K + d];
      val = qk * expf(G[i] - G[j]);
    }
    P[e] = val;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < L * kVT; e += kThreads) {
    const int i = e / kVT, cc = e - i * kVT;
    if (cc >= vt) continue;
    float qs = 0.f;
    for (int d = 0; d < K; ++d) qs += Qn[i * K + d] * S[d * kVT + cc];
    float acc = expf(G[i]) * qs;
    for (int j = 0; j <= i; ++j) acc += P[i * C + j] * U[j * kVT + cc];
    store_elem(a.o, ((size_t)(t0 + i) * a.Hv + h) * V + c0 + cc, a.scale * acc, a.io_dtype);
  }
}

size_t prep_smem(int K, int V) { return sizeof(float) * ((size_t)C * K + (size_t)C * (K + V) + C * C + 2 * C); }
size_t state_smem(int K) { return sizeof(float) * ((size_t)K * kVT + (size_t)C * K + C * kVT + (size_t)C * K + C); }
size_t output_smem(int K) { return sizeof(float) * (2 * (size_t)C * K + (size_t)K * kVT + C * kVT + C * C + C); }

}  // namespace

size_t chunk_generic_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V) {
  size_t total = 0;
  ws_layout(nullptr, max_chunks(T_total, num_seqs), num_seqs, Hv, K, V, &total);
  return total;
}

cudaError_t launch_chunk_generic(const ChunkArgs& a) {
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  const long long NC = max_chunks(T_total, a.num_seqs);
  WsLayout ws = ws_layout(a.workspace, NC, a.num_seqs, a.Hv, a.K, a.V, nullptr);
  cudaError_t err;
  const size_t sp = prep_smem(a.K, a.V), ss = state_smem(a.K), so = output_smem(a.K);
  if ((err = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp))) return err;
  if ((err = cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss))) return err;
  if ((err = cudaFuncSetAttribute(chunk_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)so))) return err;
  chunk_table_kernel<<<1, 1024, 0, a.stream>>>(a, ws.chunk_off);
  if ((err = cudaGetLastError())) return err;
  if (NC > 0 && a.num_seqs > 0) {
    chunk_prep_kernel<<<dim3((unsigned)NC, a.Hv), kThreads, sp, a.stream>>>(a, ws);
    if ((err = cudaGetLastError())) return err;
  }
  const unsigned vtiles = (unsigned)((a.V + kVT - 1) / kVT);
  if (a.num_seqs > 0) {
    chunk_state_kernel<<<dim3(a.num_seqs, a.Hv, vtiles), kThreads, ss, a.stream>>>(a, ws);
    if ((err = cudaGetLastError())) return err;
  }
  if (NC > 0 && a.num_seqs > 0) {
    chunk_output_kernel<<<dim3((unsigned)NC, a.Hv, vtiles), kThreads, so, a.stream>>>(a, ws);
    if ((err = cudaGetLastError())) return err;
  }
  return cudaSuccess;
}

}  // namespace gdn
