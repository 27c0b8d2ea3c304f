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
#include "gdn_chunk_util.cuh"

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

// acc[r][s] = sum_d X[ti + 16 r][d] Y[tj + 16 s][d] over d < K, for the 64 x 64 products of the
// chunk (rows of X and Y at stride ld in shared memory).  Thread t takes ti = t / 16 and
// tj = t % 16: its rows and columns are 16 apart, so with an odd ld a warp's reads of Y fall in
// 16 different banks and those of X are broadcasts; each read feeds four FMAs.
__device__ __forceinline__ void gram64(const float* X, const float* Y, int ld, int K, float (&acc)[4][4]) {
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
  for (int d = 0; d < K; ++d) {
    float x[4], y[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] = X[(ti + 16 * r) * ld + d];
#pragma unroll
    for (int q = 0; q < 4; ++q) y[q] = Y[(tj + 16 * q) * ld + d];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(x[r], y[q], acc[r][q]);
  }
}

// ---------------------------------------------------------------- 2. prep
// smem: Kn[C][K + 1] (rows padded by one float: the K K^T product reads 32 rows at one column
// per warp, which then fall in 32 different banks), A[C][C], G[C], bt[C], be[C] = beta exp(G).
// Thread t owns column t of [W | U] (K + V <= 256 columns): it builds the column of the
// right-hand side [diag(beta exp G) Kn | diag(beta) V] in registers and solves (I + A) x = rhs
// there by a right-looking substitution, four columns of A at a time (each float4 of A is a
// broadcast read that feeds four FMAs); rows past the chunk end are zero in A and in the
// right-hand side, so every column runs all 64 rows.
__global__ void __launch_bounds__(kThreads, 2) chunk_prep_kernel(const ChunkArgs a, WsLayout ws) {
  extern __shared__ float smem[];
  const int K = a.K, V = a.V, M = K + V, ldk = K + 1;
  float* Kn = smem;
  float* A = Kn + C * ldk;   // 16-byte aligned: C (K + 1) floats before it
  float* G = A + C * C;
  float* bt = G + C;
  float* be = bt + C;
  const int c = blockIdx.x, h = blockIdx.y;
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  if (a.state_indices && seq_slot(a, n) < 0) return;
  const int hq = h / (a.Hv / a.Hqk);
  const int col = threadIdx.x;
  // this column's V entries, issued before the K K^T product
  float x[C];
#pragma unroll
  for (int i = 0; i < C; ++i)
    x[i] = (col >= K && col < M && i < L)
               ? load_elem(a.v, ((size_t)(t0 + i) * a.Hv + h) * V + (col - K), a.io_dtype) : 0.f;
  load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Kn, ldk);
  load_gates(a, t0, L, h, G, bt);
  __syncthreads();
  if (threadIdx.x < C) be[threadIdx.x] = bt[threadIdx.x] * expf(G[threadIdx.x]);
  // A (strictly lower)
  {
    float acc[4][4];
    gram64(Kn, Kn, ldk, K, acc);
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = ti + 16 * r, j = tj + 16 * q;
        A[i * C + j] = j < i ? bt[i] * acc[r][q] * expf(G[i] - G[j]) : 0.f;
      }
  }
  __syncthreads();
  if (col < M) {
    // the right-hand side (rows >= L of be and bt are zero)
    if (col < K) {
#pragma unroll
      for (int i = 0; i < C; ++i) x[i] = be[i] * Kn[i * ldk + col];
    } else {
#pragma unroll
      for (int i = 0; i < C; ++i) x[i] *= bt[i];
    }
#pragma unroll
    for (int g = 0; g < C / 4; ++g) {
      const int m0 = 4 * g;
      // the diagonal block: rows m0 + 1 .. m0 + 3 by the columns before them
#pragma unroll
      for (int r = 1; r < 4; ++r) {
        const float4 av = *reinterpret_cast<const float4*>(A + (m0 + r) * C + m0);
        const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int e = 0; e < r; ++e) x[m0 + r] = fmaf(-aa[e], x[m0 + e], x[m0 + r]);
      }
      // the rows below the block by its four columns
#pragma unroll
      for (int i = m0 + 4; i < C; ++i) {
        const float4 av = *reinterpret_cast<const float4*>(A + i * C + m0);
        x[i] = fmaf(-av.x, x[m0], x[i]);
        x[i] = fmaf(-av.y, x[m0 + 1], x[i]);
        x[i] = fmaf(-av.z, x[m0 + 2], x[i]);
        x[i] = fmaf(-av.w, x[m0 + 3], x[i]);
      }
    }
    const size_t ch = (size_t)c * a.Hv + h;
    if (col < K) {
      float* Wd = ws.W + ch * C * K;
#pragma unroll
      for (int i = 0; i < C; ++i) Wd[i * K + col] = x[i];
    } else {
      float* Ud = ws.U + ch * C * V;
#pragma unroll
      for (int i = 0; i < C; ++i) Ud[i * V + (col - K)] = x[i];
    }
  }
  if (threadIdx.x < C) ws.G[((size_t)c * a.Hv + h) * C + threadIdx.x] = G[threadIdx.x];
}

// ---------------------------------------------------------------- 3. state
// Per (sequence, head, 32-column tile).  smem: S[K][32], W[C][K + 1] (rows padded by one float),
// U[C][32], Kn[C][K], G[C], then dl[C] = exp(G_last - G_t) of the chunk.  Both products are
// register-blocked: thread t takes rows t / 8 + 32 r and the four columns 4 (t % 8) .. + 3 (read
// as one float4 of S or U').
template <int RK>   // rows of the state update a thread takes: K <= 32 RK
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(const ChunkArgs a, WsLayout ws) {
  extern __shared__ float smem[];
  const int K = a.K, V = a.V, ldw = K + 1;
  float* S = smem;
  float* W = S + K * kVT;
  float* U = W + C * ldw;
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
  // The next chunk's W, U tile, G and raw k rows are loaded into registers while the current
  // chunk computes (k rows: warp w takes rows w + 8 u, lane l the elements l + 32 m).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w_row_step = kThreads / K, w_col_step = kThreads - w_row_step * K;
  float wr[32], ur[8], kr[8][4], gr = 0.f;
  auto fetch = [&](size_t chn, int t0n, int Ln) {
    const float* Wg = ws.W + chn * C * K;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = threadIdx.x + kThreads * j;
      wr[j] = e < C * K ? Wg[e] : 0.f;
    }
    const float* Ug = ws.U + chn * C * V;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = threadIdx.x + kThreads * j, i = e / kVT, cc = e - i * kVT;
      ur[j] = cc < vt ? Ug[(size_t)i * V + c0 + cc] : 0.f;
    }
    if (threadIdx.x < C) gr = ws.G[chn * C + threadIdx.x];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = warp + 8 * u;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = lane + 32 * m;
        kr[u][m] = (r < Ln && e < K) ? load_elem(a.k, ((size_t)(t0n + r) * a.Hqk + hq) * K + e, a.io_dtype) : 0.f;
      }
    }
  };
  if (bos < eos) fetch((size_t)first * a.Hv + h, bos, min(C, eos - bos));
  for (int t0 = bos, ci = first; t0 < eos; t0 += C, ++ci) {
    const int L = min(C, eos - t0);
    const size_t ch = (size_t)ci * a.Hv + h;
    __syncthreads();
    float* Srec = ws.S + ch * K * V;
    float* Ug = ws.U + ch * C * V;
    for (int e = threadIdx.x; e < K * kVT; e += kThreads) {
      const int d = e / kVT, cc = e - d * kVT;
      if (cc < vt) Srec[(size_t)d * V + c0 + cc] = S[e];
    }
    // this chunk's operands from the registers into shared memory (k rows normalised); element
    // e = t + 256 j of W sits at row e / K, column e % K, stepped without a division per element
    {
      int wrow = threadIdx.x / K, wcol = threadIdx.x - wrow * K;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (threadIdx.x + kThreads * j < C * K) W[wrow * ldw + wcol] = wr[j];
        wrow += w_row_step;
        wcol += w_col_step;
        if (wcol >= K) { wcol -= K; ++wrow; }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) U[threadIdx.x + kThreads * j] = ur[j];
    if (threadIdx.x < C) G[threadIdx.x] = gr;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = warp + 8 * u;
      float rn = 1.f;
      if (a.use_qk_l2norm && r < L) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(kr[u][m], kr[u][m], ss);
        rn = 1.0f / sqrtf(warp_sum(ss) + kL2Eps);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = lane + 32 * m;
        if (e < K) Kn[r * K + e] = kr[u][m] * rn;
      }
    }
    if (t0 + C < eos) fetch(ch + a.Hv, t0 + C, min(C, eos - t0 - C));   // the next chunk's, in flight
    __syncthreads();
    // U' = U - W S   (rows >= L of W and U are zero, so U' is zero there)
    const int ti = threadIdx.x >> 3, c4 = 4 * (threadIdx.x & 7);
    {
      float acc[2][4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float4 u = *reinterpret_cast<const float4*>(U + (ti + 32 * r) * kVT + c4);
        acc[r][0] = u.x; acc[r][1] = u.y; acc[r][2] = u.z; acc[r][3] = u.w;
      }
      for (int d = 0; d < K; ++d) {
        const float4 sv = *reinterpret_cast<const float4*>(S + d * kVT + c4);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float w = W[(ti + 32 * r) * ldw + d];
          acc[r][0] = fmaf(-w, sv.x, acc[r][0]); acc[r][1] = fmaf(-w, sv.y, acc[r][1]);
          acc[r][2] = fmaf(-w, sv.z, acc[r][2]); acc[r][3] = fmaf(-w, sv.w, acc[r][3]);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        *reinterpret_cast<float4*>(U + (ti + 32 * r) * kVT + c4) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < C * kVT; e += kThreads) {
      const int i = e / kVT, cc = e - i * kVT;
      if (cc < vt) Ug[(size_t)i * V + c0 + cc] = U[e];
    }
    // S <- exp(G_last) S + sum_t exp(G_last - G_t) Kn_t U'_t
    const float gl = G[L - 1];
    const float dl = expf(gl);
    float* dlt = G + C;
    if (threadIdx.x < C) dlt[threadIdx.x] = threadIdx.x < L ? expf(gl - G[threadIdx.x]) : 0.f;
    __syncthreads();
    {   // rows d = ti + 32 r < K
      float acc[RK][4];
#pragma unroll
      for (int r = 0; r < RK; ++r) {
        const int d = ti + 32 * r;
        float4 sv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (d < K) sv = *reinterpret_cast<const float4*>(S + d * kVT + c4);
        acc[r][0] = dl * sv.x; acc[r][1] = dl * sv.y; acc[r][2] = dl * sv.z; acc[r][3] = dl * sv.w;
      }
      for (int t = 0; t < L; ++t) {
        const float4 uv = *reinterpret_cast<const float4*>(U + t * kVT + c4);
        const float wt = dlt[t];
#pragma unroll
        for (int r = 0; r < RK; ++r) {
          const int d = ti + 32 * r;
          const float kw = d < K ? wt * Kn[t * K + d] : 0.f;
          acc[r][0] = fmaf(kw, uv.x, acc[r][0]); acc[r][1] = fmaf(kw, uv.y, acc[r][1]);
          acc[r][2] = fmaf(kw, uv.z, acc[r][2]); acc[r][3] = fmaf(kw, uv.w, acc[r][3]);
        }
      }
#pragma unroll
      for (int r = 0; r < RK; ++r) {
        const int d = ti + 32 * r;
        if (d < K)
          *reinterpret_cast<float4*>(S + d * kVT + c4) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      }
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
// Per (chunk, head, TW-column tile; TW = 64 when V <= 64, so that P and the q, k rows are formed
// once per chunk and head, else 32).  smem: Qn[C][K + 1], Kn[C][K + 1] (rows padded as in the
// prep), S[K][TW], U[C][TW], P[C][C + 1], G[C].  P by gram64; the output register-blocked: thread
// t takes the four columns 4 (t % (TW / 4)) .. + 3 of rows t / (TW / 4) + (1024 / TW) r.
template <int TW>
__global__ void __launch_bounds__(kThreads) chunk_output_kernel(const ChunkArgs a, WsLayout ws) {
  constexpr int CG = TW / 4, RS = kThreads / CG, RR = C / RS;
  extern __shared__ float smem[];
  const int K = a.K, V = a.V, ldk = K + 1, ldp = C + 1;
  float* Qn = smem;
  float* Kn = Qn + C * ldk;
  float* S = Kn + C * ldk;
  float* U = S + K * TW;
  float* P = U + C * TW;
  float* G = P + C * ldp;
  const int c = blockIdx.x, h = blockIdx.y, c0 = blockIdx.z * TW;
  const int vt = min(TW, V - c0);
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
  load_rows(a.q, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Qn, ldk);
  load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, a.use_qk_l2norm != 0, Kn, ldk);
  const float* Sg = ws.S + ch * K * V;
  for (int e = threadIdx.x; e < K * TW; e += kThreads) {
    const int d = e / TW, cc = e - d * TW;
    S[e] = cc < vt ? Sg[(size_t)d * V + c0 + cc] : 0.f;
  }
  const float* Ug = ws.U + ch * C * V;
  for (int e = threadIdx.x; e < C * TW; e += kThreads) {
    const int i = e / TW, cc = e - i * TW;
    U[e] = cc < vt ? Ug[(size_t)i * V + c0 + cc] : 0.f;
  }
  if (threadIdx.x < C) G[threadIdx.x] = ws.G[ch * C + threadIdx.x];
  __syncthreads();
  {
    float acc[4][4];
    gram64(Qn, Kn, ldk, K, acc);
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = ti + 16 * r, j = tj + 16 * q;
        P[i * ldp + j] = (j <= i && i < L) ? acc[r][q] * expf(G[i] - G[j]) : 0.f;
      }
  }
  __syncthreads();
  const int ti = threadIdx.x / CG, c4 = 4 * (threadIdx.x % CG);
  float qs[RR][4], acc[RR][4];
#pragma unroll
  for (int r = 0; r < RR; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) { qs[r][q] = 0.f; acc[r][q] = 0.f; }
  for (int d = 0; d < K; ++d) {
    const float4 sv = *reinterpret_cast<const float4*>(S + d * TW + c4);
#pragma unroll
    for (int r = 0; r < RR; ++r) {
      const float x = Qn[(ti + RS * r) * ldk + d];
      qs[r][0] = fmaf(x, sv.x, qs[r][0]); qs[r][1] = fmaf(x, sv.y, qs[r][1]);
      qs[r][2] = fmaf(x, sv.z, qs[r][2]); qs[r][3] = fmaf(x, sv.w, qs[r][3]);
    }
  }
  for (int j = 0; j < L; ++j) {   // P is zero above the diagonal and past the chunk end
    const float4 uv = *reinterpret_cast<const float4*>(U + j * TW + c4);
#pragma unroll
    for (int r = 0; r < RR; ++r) {
      const float pv = P[(ti + RS * r) * ldp + j];
      acc[r][0] = fmaf(pv, uv.x, acc[r][0]); acc[r][1] = fmaf(pv, uv.y, acc[r][1]);
      acc[r][2] = fmaf(pv, uv.z, acc[r][2]); acc[r][3] = fmaf(pv, uv.w, acc[r][3]);
    }
  }
#pragma unroll
  for (int r = 0; r < RR; ++r) {
    const int i = ti + RS * r;
    if (i >= L) continue;
    const float eg = expf(G[i]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c4 + q < vt)
        store_elem(a.o, ((size_t)(t0 + i) * a.Hv + h) * V + c0 + c4 + q, a.scale * fmaf(eg, qs[r][q], acc[r][q]),
                   a.io_dtype);
  }
}

// The state pass for K <= 64 (two rows of the update a thread) or up to 128 (four).
cudaError_t launch_state_kernel(const ChunkArgs& a, const WsLayout& ws, size_t ss) {
  const unsigned vtiles = (unsigned)((a.V + kVT - 1) / kVT);
  const dim3 grid(a.num_seqs, a.Hv, vtiles);
  cudaError_t err;
  if (a.K <= 64) {
    if ((err = cudaFuncSetAttribute(chunk_state_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss))) return err;
    chunk_state_kernel<2><<<grid, kThreads, ss, a.stream>>>(a, ws);
  } else {
    if ((err = cudaFuncSetAttribute(chunk_state_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss))) return err;
    chunk_state_kernel<4><<<grid, kThreads, ss, a.stream>>>(a, ws);
  }
  return cudaGetLastError();
}

size_t prep_smem(int K, int V) { (void)V; return sizeof(float) * ((size_t)C * (K + 1) + C * C + 3 * C); }
size_t state_smem(int K) { return sizeof(float) * ((size_t)K * kVT + (size_t)C * (K + 1) + C * kVT + (size_t)C * K + 2 * C); }
size_t output_smem(int K, int TW) { return sizeof(float) * (2 * (size_t)C * (K + 1) + (size_t)K * TW + C * TW + (size_t)C * (C + 1) + C); }

// The output pass: one CTA per (chunk, head, 64 columns) when V <= 64, else per 32 columns.
cudaError_t launch_output_kernel(const ChunkArgs& a, const WsLayout& ws, long long NC) {
  const int TW = a.V <= 64 ? 64 : kVT;
  const size_t so = output_smem(a.K, TW);
  const dim3 grid((unsigned)NC, a.Hv, (unsigned)((a.V + TW - 1) / TW));
  cudaError_t err;
  if (TW == 64) {
    if ((err = cudaFuncSetAttribute(chunk_output_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)so))) return err;
    chunk_output_kernel<64><<<grid, kThreads, so, a.stream>>>(a, ws);
  } else {
    if ((err = cudaFuncSetAttribute(chunk_output_kernel<kVT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)so))) return err;
    chunk_output_kernel<kVT><<<grid, kThreads, so, a.stream>>>(a, ws);
  }
  return cudaGetLastError();
}

}  // namespace

size_t chunk_generic_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V) {
  size_t total = 0;
  ws_layout(nullptr, max_chunks(T_total, num_seqs), num_seqs, Hv, K, V, &total);
  return total;
}

cudaError_t launch_chunk_prep(const ChunkArgs& a, int32_t* chunk_off, float* W, float* U,
                              float* G) {
  WsLayout ws;
  ws.chunk_off = chunk_off;
  ws.W = W;
  ws.U = U;
  ws.G = G;
  ws.S = nullptr;
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  const long long NC = max_chunks(T_total, a.num_seqs);
  const size_t sp = prep_smem(a.K, a.V);
  cudaError_t err;
  if ((err = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp))) return err;
  if (NC <= 0 || a.num_seqs <= 0) return cudaSuccess;
  chunk_prep_kernel<<<dim3((unsigned)NC, a.Hv), kThreads, sp, a.stream>>>(a, ws);
  return cudaGetLastError();
}

cudaError_t launch_chunk_states(const ChunkArgs& a, int32_t* chunk_off, float* W, float* U,
                                float* G, float* S) {
  WsLayout ws;
  ws.chunk_off = chunk_off;
  ws.W = W;
  ws.U = U;
  ws.G = G;
  ws.S = S;
  if (a.num_seqs <= 0) return cudaSuccess;
  return launch_state_kernel(a, ws, state_smem(a.K));
}

cudaError_t launch_chunk_generic(const ChunkArgs& a) {
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  const long long NC = max_chunks(T_total, a.num_seqs);
  WsLayout ws = ws_layout(a.workspace, NC, a.num_seqs, a.Hv, a.K, a.V, nullptr);
  cudaError_t err;
  const size_t sp = prep_smem(a.K, a.V), ss = state_smem(a.K);
  if ((err = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp))) return err;
  chunk_table_kernel<<<1, 1024, 0, a.stream>>>(a, ws.chunk_off);
  if ((err = cudaGetLastError())) return err;
  if (NC > 0 && a.num_seqs > 0) {
    chunk_prep_kernel<<<dim3((unsigned)NC, a.Hv), kThreads, sp, a.stream>>>(a, ws);
    if ((err = cudaGetLastError())) return err;
  }
  if (a.num_seqs > 0 && (err = launch_state_kernel(a, ws, ss))) return err;
  if (NC > 0 && a.num_seqs > 0 && (err = launch_output_kernel(a, ws, NC))) return err;
  return cudaSuccess;
}

}  // namespace gdn
