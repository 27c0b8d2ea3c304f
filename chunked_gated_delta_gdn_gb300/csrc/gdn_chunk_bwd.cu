// gdn_chunk_bwd.cu -- backward of the chunkwise gated delta rule on the fp32 CUDA cores.
//
// For a loss with gradient dO on the outputs and dS_fin on the final states, computes
// dq, dk, dv, dg, dbeta and the initial-state gradient.  Training runs the chunked rule
// ("Megatron-Core API: core.ssm.gated_delta_net.gdn", torch_chunk_gated_delta_rule, the
// deterministic mode; "Megatron-Core API: core.ssm.gated_delta_product",
// _gdp_chunk_forward serves training too); the sources give no backward, so this is the
// exact adjoint of the forward evaluation.  Within a chunk of L <= 64 tokens (in-chunk
// cumulative log-decay G, gamma_i = exp(G_i), lambda_i = exp(G_{L-1} - G_i),
// Gamma_ij = exp(G_i - G_j), normalised Q, K, entry state S0):
//   A  = strict_lower(diag(beta) K K^T * Gamma),   T = (I + A)^{-1}
//   X  = diag(beta) (V - diag(gamma) K S0),          U' = T X
//   P  = (Q K^T * Gamma) on and below the diagonal
//   O  = scale (diag(gamma) Q S0 + P U'),   S_end = gamma_L S0 + K^T diag(lambda) U'
// and, with dS the gradient of S_end:
//   dU' = scale P^T dO + diag(lambda) K dS,   dX = T^T dU',   dV = diag(beta) dX
//   dS0 = gamma_L dS + scale Q^T diag(gamma) dO - K^T diag(gamma beta) dX
//   F   = scale (dO U'^T) * Gamma on and below the diagonal
//   dA  = -(dX U'^T) strictly below the diagonal,   E = diag(beta) dA * Gamma
//   dQ  = scale diag(gamma) dO S0^T + F K
//   dK  = F^T Q + diag(lambda) U' dS^T - diag(gamma beta) dX S0^T + (E + E^T) K
//   dbeta_i = dX_i . (V_i - gamma_i S0^T k_i) + sum_j dA_ij (K K^T * Gamma)_ij
//   dG_i = scale gamma_i q_i . S0 dO_i - beta_i gamma_i k_i . S0 dX_i - lambda_i k_i . dS u'_i
//          + rowsum_i(Z) - colsum_i(Z),   Z = F * (Q K^T) + E * (K K^T),
//          plus gamma_L <S0, dS> + sum_j lambda_j k_j . dS u'_j at i = L - 1,
//   dg  = the reverse in-chunk cumulative sum of dG;
// the L2 norm's Jacobian then maps dQ, dK (summed over the value heads of a query/key
// head, in a fixed order) to dq, dk.
//
// Six launches on the caller's stream, no host sync and no atomics (the result is
// bitwise reproducible run to run):
//   1. chunk table  from cu_seqlens, on the device
//   2. states       the forward recompute of the entry state S0 of every chunk and of U':
//                   bf16 with K = V = 128, the tensor-core forward kernel in record mode;
//                   otherwise (after 3) the fp32 state pass per (sequence, value head,
//                   32 columns) on W, U from the prep kernel
//   3. prep         per (chunk, value head): T, dUp = scale P^T dO, G, and for the fp32
//                   state pass W = T diag(beta gamma) K, U = T diag(beta) V
//   4. reverse      per (sequence, value head, 32 columns), chunks last to first:
//                   records dS (the gradient of each chunk's exit state) and dX
//   5. grad         per (chunk, value head): dv, dbeta, dg, and dQ, dK per value head
//   6. qk           per token: the group sum and the L2-norm Jacobian -> dq, dk;
//                   zero gradients for tokens outside every sequence
#include "gdn_chunk_util.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;
constexpr int KP = GDN_MAX_HEAD_DIM;  // tiles are padded to the largest head dim
constexpr int LD = KP + 1;            // row stride of [C][KP] tiles (odd: column reads hit distinct banks)
constexpr int LDC = C + 1;            // row stride of [C][C] tiles
constexpr int VT = 32;                // V columns per V tile
constexpr int LDT = VT + 1;           // row stride of [C][VT] tiles

struct BwdWs {
  int32_t* chunk_off;  // [N + 2]
  float* W;            // [NC][Hv][C][K]
  float* U;            // [NC][Hv][C][V]  U, then U'
  float* G;            // [NC][Hv][C]
  float* S;            // [NC][Hv][K][V]  state at chunk entry
  float* T;            // [NC][Hv][C][C]
  float* dUp;          // [NC][Hv][C][V]  scale P^T dO
  float* dS;           // [NC][Hv][K][V]  gradient of the chunk's exit state
  float* dX;           // [NC][Hv][C][V]
  float* Z;            // [NC][Hv][K][V]  scale Q^T diag(gamma) dO
  float* dQ;           // [T_total][Hv][K] per value head, before the norm
  float* dK;           // [T_total][Hv][K]
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline BwdWs bwd_layout(void* base, long long NC, int N, int Hv, int K, int V,
                                            long long T_total, size_t* total) {
  BwdWs w;
  char* p = reinterpret_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = p + off;
    off = align256(off + bytes);
    return r;
  };
  const size_t f = sizeof(float), ch = (size_t)NC * Hv;
  w.chunk_off = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)(N + 2)));
  w.W = reinterpret_cast<float*>(take(f * ch * C * K));
  w.U = reinterpret_cast<float*>(take(f * ch * C * V));
  w.G = reinterpret_cast<float*>(take(f * ch * C));
  w.S = reinterpret_cast<float*>(take(f * ch * K * V));
  w.T = reinterpret_cast<float*>(take(f * ch * C * C));
  w.dUp = reinterpret_cast<float*>(take(f * ch * C * V));
  w.dS = reinterpret_cast<float*>(take(f * ch * K * V));
  w.dX = reinterpret_cast<float*>(take(f * ch * C * V));
  w.Z = reinterpret_cast<float*>(take(f * ch * K * V));
  w.dQ = reinterpret_cast<float*>(take(f * (size_t)T_total * Hv * K));
  w.dK = reinterpret_cast<float*>(take(f * (size_t)T_total * Hv * K));
  if (total) *total = off;
  return w;
}

// acc[r][c] += sum_{k0 <= k < k1} A(r, k) B(k, c) over shared-memory operands with
// A(r, k) = a[r * AR + k * AK] and B(k, c) = b[k * BK + c * BC].  The callers give each
// warp its own rows (A reads are broadcasts) and each lane its own columns (B reads
// are consecutive or odd-strided, so conflict-free).
template <int TM, int TN, int AR, int AK, int BK, int BC>
__device__ __forceinline__ void fma_tile(float (&acc)[TM][TN], const float* a, const float* b,
                                         int k0, int k1) {
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    float x[TM], y[TN];
#pragma unroll
    for (int r = 0; r < TM; ++r) x[r] = a[r * AR + k * AK];
#pragma unroll
    for (int c = 0; c < TN; ++c) y[c] = b[k * BK + c * BC];
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
      for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(x[r], y[c], acc[r][c]);
  }
}

template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN]) {
#pragma unroll
  for (int r = 0; r < TM; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[r][c] = 0.f;
}

// Columns [D, KP) of a [C][LD] tile set to zero.
__device__ __forceinline__ void zero_cols(float* dst, int D) {
  const int w = KP - D;
  if (w <= 0) return;
  for (int e = threadIdx.x; e < C * w; e += blockDim.x) dst[(e / w) * LD + D + e % w] = 0.f;
}

// Columns [c0, c0 + width) of rows [t0, t0 + L) of a [T, H, D] tensor (head hd) into
// dst[C][ld], each row times rs[r] when rs is given; rows >= L and columns >= D zero.
// Warps [w0, w0 + nw) of the block take part.
__device__ void load_tile(const void* src, int dtype, int t0, int L, int H, int hd, int D, int c0,
                          int width, const float* rs, float* dst, int ld, int w0, int nw) {
  const int warp = (int)(threadIdx.x >> 5) - w0, lane = threadIdx.x & 31;
  if (warp < 0 || warp >= nw) return;
  for (int r = warp; r < C; r += nw) {
    const float s = rs ? rs[r] : 1.f;
    for (int e = lane; e < width; e += 32) {
      float x = 0.f;
      if (r < L && c0 + e < D) x = s * load_elem(src, ((size_t)(t0 + r) * H + hd) * D + c0 + e, dtype);
      dst[r * ld + e] = x;
    }
  }
}

// Rows [i0, i0 + TM) and columns lane + 32 c (< D) of a [C][D] fp32 block in global memory.
template <int TM, int TN>
__device__ __forceinline__ void store_rows(float* dst, int D, const float (&acc)[TM][TN], int i0,
                                           int lane, float s) {
#pragma unroll
  for (int r = 0; r < TM; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c) {
      const int col = lane + 32 * c;
      if (col < D) dst[(size_t)(i0 + r) * D + col] = s * acc[r][c];
    }
}

// ---------------------------------------------------------------- 3. prep
// Per (chunk, value head), 16 warps: A and P, T = (I + A)^{-1}, dUp = scale P^T dO and
// Z = scale Q^T diag(gamma) dO (the part of the state-gradient step that does not depend on
// the state gradient, taken out of the serial reverse pass), and for the fp32 state pass
// W = T diag(beta gamma) K, U = T diag(beta) V.
constexpr int kPrepThreads = 512;
constexpr int DLD = KP + 4;  // row stride of [C][KP] tiles read as float4 (16-byte aligned rows)
constexpr size_t kPrepSmem = sizeof(float) * (2 * C * LD + C * DLD + 3 * C * LDC + 3 * C);

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const ChunkArgs a, const BwdArgs b,
                                                                BwdWs ws, int need_wu) {
  extern __shared__ float smem[];
  float* Kn = smem;           // [C][LD] normalised k (then diag(beta gamma) k)
  float* Qn = Kn + C * LD;    // [C][LD] normalised q
  float* dO = Qn + C * LD;    // [C][DLD] dO (then diag(beta) v)
  float* A = dO + C * DLD;    // [C][LDC]
  float* P = A + C * LDC;     // [C][LDC]
  float* Tm = P + C * LDC;    // [C][LDC]
  float* G = Tm + C * LDC;    // [C]
  float* bt = G + C;          // [C]
  float* gm = bt + C;         // [C] gamma
  const int c = blockIdx.x, h = blockIdx.y;
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  const int K = a.K, V = a.V, hq = h / (a.Hv / a.Hqk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool l2 = a.use_qk_l2norm != 0;
  load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, l2, Kn, LD);
  load_rows(a.q, a.io_dtype, t0, L, a.Hqk, hq, K, l2, Qn, LD);
  zero_cols(Kn, K);
  zero_cols(Qn, K);
  load_tile(b.d_o, a.io_dtype, t0, L, a.Hv, h, V, 0, KP, nullptr, dO, DLD, 0, kPrepThreads / 32);
  load_gates(a, t0, L, h, G, bt);
  __syncthreads();
  if (tid < C) gm[tid] = expf(G[tid]);
  {  // A = strict_lower(diag(beta) K K^T * Gamma), P = (Q K^T * Gamma) on and below the diagonal
    const int i0 = 4 * warp;
    float kk[4][2], qk[4][2];
    zero(kk);
    zero(qk);
    fma_tile<4, 2, LD, 1, 1, 32 * LD>(kk, Kn + i0 * LD, Kn + lane * LD, 0, K);
    fma_tile<4, 2, LD, 1, 1, 32 * LD>(qk, Qn + i0 * LD, Kn + lane * LD, 0, K);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int i = i0 + r, j = lane + 32 * m;
        const float gij = j <= i ? expf(G[i] - G[j]) : 0.f;
        A[i * LDC + j] = j < i ? bt[i] * kk[r][m] * gij : 0.f;
        P[i * LDC + j] = qk[r][m] * gij;
      }
  }
  __syncthreads();
  const size_t ch = (size_t)c * a.Hv + h;
  const int ty = tid >> 4, tx = tid & 15;  // 32 row groups x 16 groups of 8 columns
  {  // Z = scale Q^T diag(gamma) dO: rows d = ty + 32 r, columns 8 tx .. 8 tx + 7
    float z[4][8];
    zero(z);
    for (int i = 0; i < L; ++i) {
      const float g = gm[i];
      float x[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) x[r] = g * Qn[i * LD + ty + 32 * r];
      const float4 y0 = ld4(dO + i * DLD + 8 * tx), y1 = ld4(dO + i * DLD + 8 * tx + 4);
      const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 8; ++q) z[r][q] = fmaf(x[r], y[q], z[r][q]);
    }
    float* Zg = ws.Z + ch * K * V;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = ty + 32 * r;
      if (d >= K) continue;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int col = 8 * tx + 4 * hlf;
        if (col < V)
          st4(Zg + (size_t)d * V + col,
              make_float4(a.scale * z[r][4 * hlf], a.scale * z[r][4 * hlf + 1],
                          a.scale * z[r][4 * hlf + 2], a.scale * z[r][4 * hlf + 3]));
      }
    }
  }
  if (tid < C) {
    // T = (I + A)^{-1}, one column per thread by forward substitution (four partial sums)
    const int j = tid;
    for (int i = 0; i < C; ++i) {
      float t = i == j ? 1.f : 0.f;
      if (i > j) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int m = j;
        for (; m + 3 < i; m += 4) {
          s0 = fmaf(A[i * LDC + m], Tm[m * LDC + j], s0);
          s1 = fmaf(A[i * LDC + m + 1], Tm[(m + 1) * LDC + j], s1);
          s2 = fmaf(A[i * LDC + m + 2], Tm[(m + 2) * LDC + j], s2);
          s3 = fmaf(A[i * LDC + m + 3], Tm[(m + 3) * LDC + j], s3);
        }
        for (; m < i; ++m) s0 = fmaf(A[i * LDC + m], Tm[m * LDC + j], s0);
        t = -((s0 + s1) + (s2 + s3));
      }
      Tm[i * LDC + j] = t;
    }
  }
  __syncthreads();
  {  // dUp = scale P^T dO: rows i = ty, ty + 32, columns 8 tx .. 8 tx + 7 (P[m][i] = 0 for m < i)
    float u[2][8];
    zero(u);
    for (int m = ty; m < C; ++m) {
      const float x0 = P[m * LDC + ty], x1 = P[m * LDC + ty + 32];
      const float4 y0 = ld4(dO + m * DLD + 8 * tx), y1 = ld4(dO + m * DLD + 8 * tx + 4);
      const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        u[0][q] = fmaf(x0, y[q], u[0][q]);
        u[1][q] = fmaf(x1, y[q], u[1][q]);
      }
    }
    float* Ug = ws.dUp + ch * C * V;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = ty + 32 * r;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int col = 8 * tx + 4 * hlf;
        if (col < V)
          st4(Ug + (size_t)i * V + col,
              make_float4(a.scale * u[r][4 * hlf], a.scale * u[r][4 * hlf + 1],
                          a.scale * u[r][4 * hlf + 2], a.scale * u[r][4 * hlf + 3]));
      }
    }
  }
  for (int e = tid; e < C * C; e += kPrepThreads) {
    const int i = e / C, j = e - i * C;
    ws.T[ch * C * C + e] = Tm[i * LDC + j];
  }
  if (tid < C) ws.G[ch * C + tid] = G[tid];
  if (need_wu) {  // the inputs of the fp32 forward state pass
    __syncthreads();
    for (int e = tid; e < C * KP; e += kPrepThreads) {
      const int r = e / KP, d = e - r * KP;
      Kn[r * LD + d] *= bt[r] * gm[r];
    }
    load_tile(a.v, a.io_dtype, t0, L, a.Hv, h, V, 0, KP, bt, dO, DLD, 0, kPrepThreads / 32);
    __syncthreads();
    const int i0 = 4 * warp;
    float acc[4][4];
    zero(acc);  // W = T diag(beta gamma) K  (T lower triangular: columns m <= i)
    fma_tile<4, 4, LDC, 1, LD, 32>(acc, Tm + i0 * LDC, Kn + lane, 0, i0 + 4);
    store_rows(ws.W + ch * C * K, K, acc, i0, lane, 1.f);
    zero(acc);  // U = T diag(beta) V
    fma_tile<4, 4, LDC, 1, DLD, 32>(acc, Tm + i0 * LDC, dO + lane, 0, i0 + 4);
    store_rows(ws.U + ch * C * V, V, acc, i0, lane, 1.f);
  }
}

// ---------------------------------------------------------------- 4. reverse
// Per (32 columns of V, value head, sequence), chunks last to first, 8 warps, two CTAs per SM.
// The state gradient dS of the 32 columns lives in registers (a 4 x 4 block per thread) and,
// for the next chunk's K dS, in shared memory.  Per chunk:
//   Y = K dS,  dU' = dUp + diag(lambda) Y,  dX = T^T dU',
//   dS <- gamma_L dS + Z - K^T diag(gamma beta) dX     (Z from the prep kernel)
constexpr int kRevThreads = 256;
constexpr int KLD = KP + 4;   // [C][KLD]: k rows, float4 reads
constexpr int TLD = C + 2;    // [KP][TLD]: k transposed, float2 reads
constexpr size_t kRevSmem = sizeof(float) * (C * KLD + KP * TLD + KP * VT + 2 * C * VT + 2 * C);

__global__ void __launch_bounds__(kRevThreads, 2) bwd_reverse_kernel(const ChunkArgs a,
                                                                     const BwdArgs b, BwdWs ws) {
  extern __shared__ float smem[];
  float* Kn = smem;             // [C][KLD]
  float* Kt = Kn + C * KLD;     // [KP][TLD]
  float* dSs = Kt + KP * TLD;   // [KP][VT]
  float* X1 = dSs + KP * VT;    // [C][VT] dUp, then dU'
  float* X2 = X1 + C * VT;      // [C][VT] -diag(gamma beta) dX
  float* G = X2 + C * VT;       // [C]
  float* bt = G + C;            // [C]
  // blocks: (32-column slice, value head, sequence), the slice fastest so that the slices of
  // one head run side by side and share its k, T, dUp and Z reads in L2
  const int nvt = (a.V + VT - 1) / VT;
  const int c0 = (int)(blockIdx.x % nvt) * VT, h = (int)((blockIdx.x / nvt) % a.Hv);
  const int n = (int)(blockIdx.x / nvt / a.Hv);
  const int K = a.K, V = a.V, hq = h / (a.Hv / a.Hqk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tx = tid & 7, ty = tid >> 3;   // columns 4 tx .. 4 tx + 3; rows 4 ty.. or 2 ty..
  const int col = c0 + 4 * tx;             // V % 4 == 0: a column group is all in or all out
  const bool colok = col < V;
  const size_t st_off = ((size_t)n * a.Hv + h) * K * V;
  if (!ws.chunk_off[a.num_seqs + 1]) {  // invalid cu_seqlens: zero gradient
    if (b.d_initial && colok) {
      for (int r = 0; r < 4; ++r)
        if (4 * ty + r < K) st4(b.d_initial + st_off + (size_t)(4 * ty + r) * V + col, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    return;
  }
  int bos, eos;
  seq_bounds(a, n, &bos, &eos);
  const bool l2 = a.use_qk_l2norm != 0;
  float s[4][4];   // dS rows 4 ty + r, columns col .. col + 3
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int d = 4 * ty + r;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b.d_final && colok && d < K) x = ld4(b.d_final + st_off + (size_t)d * V + col);
    s[r][0] = x.x; s[r][1] = x.y; s[r][2] = x.z; s[r][3] = x.w;
    st4(dSs + d * VT + 4 * tx, x);
  }
  const int first = ws.chunk_off[n];
  const int nch = (eos - bos + C - 1) / C;
  for (int qc = nch - 1; qc >= 0; --qc) {
    const int t0 = bos + qc * C, L = min(C, eos - t0);
    const size_t ch = (size_t)(first + qc) * a.Hv + h;
    __syncthreads();  // the previous chunk is done with every tile
    if (colok) {      // record dS, the gradient of this chunk's exit state
      float* dSg = ws.dS + ch * K * V;
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (4 * ty + r < K)
          st4(dSg + (size_t)(4 * ty + r) * V + col, make_float4(s[r][0], s[r][1], s[r][2], s[r][3]));
    }
    // normalised k rows into Kn and Kt (warp w: rows w, w + 8, ...)
    for (int r = warp; r < C; r += kRevThreads / 32) {
      float x[4];
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int d = lane + 32 * m;
        x[m] = (r < L && d < K) ? load_elem(a.k, ((size_t)(t0 + r) * a.Hqk + hq) * K + d, a.io_dtype) : 0.f;
        ss = fmaf(x[m], x[m], ss);
      }
      if (l2) {
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss + kL2Eps);
#pragma unroll
        for (int m = 0; m < 4; ++m) x[m] *= rn;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        Kn[r * KLD + lane + 32 * m] = x[m];
        Kt[(lane + 32 * m) * TLD + r] = x[m];
      }
    }
    load_gates(a, t0, L, h, G, bt);
    const float* dUg = ws.dUp + ch * C * V;
    for (int e = tid; e < C * (VT / 4); e += kRevThreads) {
      const int i = e / (VT / 4), q = e - i * (VT / 4);
      const int cc = c0 + 4 * q;
      st4(X1 + i * VT + 4 * q, cc < V ? ld4(dUg + (size_t)i * V + cc) : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    float z[4][4];   // Z rows 4 ty + r, columns col ..
    {
      const float* Zg = ws.Z + ch * K * V;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = 4 * ty + r;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (colok && d < K) x = ld4(Zg + (size_t)d * V + col);
        z[r][0] = x.x; z[r][1] = x.y; z[r][2] = x.z; z[r][3] = x.w;
      }
    }
    __syncthreads();
    const float gL = G[L - 1];
    {  // Y = K dS for rows 2 ty, 2 ty + 1; dU' = dUp + lambda Y
      float y[2][4];
      zero(y);
#pragma unroll 4
      for (int d = 0; d < K; ++d) {
        const float2 xa = *reinterpret_cast<const float2*>(Kt + d * TLD + 2 * ty);
        const float4 xb = ld4(dSs + d * VT + 4 * tx);
        const float bb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          y[0][q] = fmaf(xa.x, bb[q], y[0][q]);
          y[1][q] = fmaf(xa.y, bb[q], y[1][q]);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = 2 * ty + r;
        const float lam = expf(gL - G[i]);
        float4 u = ld4(X1 + i * VT + 4 * tx);
        u.x = fmaf(lam, y[r][0], u.x);
        u.y = fmaf(lam, y[r][1], u.y);
        u.z = fmaf(lam, y[r][2], u.z);
        u.w = fmaf(lam, y[r][3], u.w);
        st4(X1 + i * VT + 4 * tx, u);
      }
    }
    __syncthreads();
    {  // dX = T^T dU' for rows 2 ty, 2 ty + 1 (T[j][i] = 0 for j < i)
      float x[2][4];
      zero(x);
      const float* Tg = ws.T + ch * C * C;
      for (int j = 2 * ty; j < C; ++j) {
        const float2 ta = __ldg(reinterpret_cast<const float2*>(Tg + j * C + 2 * ty));
        const float4 xb = ld4(X1 + j * VT + 4 * tx);
        const float bb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          x[0][q] = fmaf(ta.x, bb[q], x[0][q]);
          x[1][q] = fmaf(ta.y, bb[q], x[1][q]);
        }
      }
      float* dXg = ws.dX + ch * C * V;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = 2 * ty + r;
        if (colok) st4(dXg + (size_t)i * V + col, make_float4(x[r][0], x[r][1], x[r][2], x[r][3]));
        const float w = -expf(G[i]) * bt[i];
        st4(X2 + i * VT + 4 * tx, make_float4(w * x[r][0], w * x[r][1], w * x[r][2], w * x[r][3]));
      }
    }
    __syncthreads();
    {  // dS <- gamma_L dS + Z - K^T diag(gamma beta) dX
      const float dl = expf(gL);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) s[r][q] = fmaf(dl, s[r][q], z[r][q]);
#pragma unroll 4
      for (int i = 0; i < L; ++i) {
        const float4 xa = ld4(Kn + i * KLD + 4 * ty);
        const float4 xb = ld4(X2 + i * VT + 4 * tx);
        const float aa[4] = {xa.x, xa.y, xa.z, xa.w}, bb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) s[r][q] = fmaf(aa[r], bb[q], s[r][q]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
        st4(dSs + (4 * ty + r) * VT + 4 * tx, make_float4(s[r][0], s[r][1], s[r][2], s[r][3]));
    }
  }
  if (b.d_initial && colok) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (4 * ty + r < K)
        st4(b.d_initial + st_off + (size_t)(4 * ty + r) * V + col,
            make_float4(s[r][0], s[r][1], s[r][2], s[r][3]));
  }
}

// ---------------------------------------------------------------- 5. grad
constexpr int kGradThreads = 512;
constexpr int kGradWarps = kGradThreads / 32;
constexpr size_t kGradSmem = sizeof(float) * (2 * VT * LD + 4 * C * LDT + 2 * C * LD +
                                              2 * C * LDC + kGradWarps * C + 9 * C + kGradWarps);

__global__ void __launch_bounds__(kGradThreads) bwd_grad_kernel(const ChunkArgs a, const BwdArgs b,
                                                                BwdWs ws) {
  extern __shared__ float smem[];
  float* S0T = smem;            // [VT][LD]  S0 tile, transposed
  float* dST = S0T + VT * LD;   // [VT][LD]  dS tile, transposed
  float* dOs = dST + VT * LD;   // [C][LDT]
  float* dXs = dOs + C * LDT;   // [C][LDT]
  float* Us = dXs + C * LDT;    // [C][LDT]
  float* Vs = Us + C * LDT;     // [C][LDT]
  float* Qn = Vs + C * LDT;     // [C][LD]
  float* Kn = Qn + C * LD;      // [C][LD]
  float* Fs = Kn + C * LD;      // [C][LDC]
  float* Es = Fs + C * LDC;     // [C][LDC]
  float* colp = Es + C * LDC;   // [warps][C]  per-warp column sums of Z
  float* G = colp + kGradWarps * C;
  float* bt = G + C;
  float* gm = bt + C;           // gamma
  float* lm = gm + C;           // lambda
  float* dGr = lm + C;          // dG without the column sums
  float* om = dGr + C;          // omega_i = lambda_i k_i . dS u'_i
  float* dbr = om + C;          // dbeta
  float* cs = dbr + C;          // column sums of Z
  float* xg = cs + C;           // dG, then dg
  float* red = xg + C;          // [warps] partial <S0, dS>
  const int c = blockIdx.x, h = blockIdx.y;
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  const int K = a.K, V = a.V, hq = h / (a.Hv / a.Hqk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool l2 = a.use_qk_l2norm != 0;
  const size_t ch = (size_t)c * a.Hv + h;
  const int i0 = 4 * warp;  // 16 warps x 4 rows
  load_gates(a, t0, L, h, G, bt);
  float H1[4][4], H2[4][4], H3[4][4], OU[4][2], XU[4][2];
  zero(H1);
  zero(H2);
  zero(H3);
  zero(OU);
  zero(XU);
  float xv[4] = {0.f, 0.f, 0.f, 0.f}, sd = 0.f;
  // Phase A: the products that reduce over V, one 32-column tile at a time
  for (int c0 = 0; c0 < V; c0 += VT) {
    __syncthreads();
    const float* Sg = ws.S + ch * K * V;
    const float* dSg = ws.dS + ch * K * V;
    for (int e = threadIdx.x; e < KP * VT; e += kGradThreads) {
      const int d = e / VT, cc = e - d * VT;
      float s0 = 0.f, ds = 0.f;
      if (d < K && c0 + cc < V) {
        s0 = Sg[(size_t)d * V + c0 + cc];
        ds = dSg[(size_t)d * V + c0 + cc];
      }
      S0T[cc * LD + d] = s0;
      dST[cc * LD + d] = ds;
      sd = fmaf(s0, ds, sd);
    }
    const float* Ug = ws.U + ch * C * V;
    const float* dXg = ws.dX + ch * C * V;
    for (int e = threadIdx.x; e < C * VT; e += kGradThreads) {
      const int i = e / VT, cc = e - i * VT;
      const bool ok = i < L && c0 + cc < V;
      const size_t tv = ((size_t)(t0 + i) * a.Hv + h) * V + c0 + cc;
      const float dx = ok ? dXg[(size_t)i * V + c0 + cc] : 0.f;
      dOs[i * LDT + cc] = ok ? load_elem(b.d_o, tv, a.io_dtype) : 0.f;
      dXs[i * LDT + cc] = dx;
      Us[i * LDT + cc] = ok ? Ug[(size_t)i * V + c0 + cc] : 0.f;
      Vs[i * LDT + cc] = ok ? load_elem(a.v, tv, a.io_dtype) : 0.f;
      if (ok) store_elem(b.dv, tv, bt[i] * dx, a.io_dtype);
    }
    __syncthreads();
    fma_tile<4, 4, LDT, 1, LD, 32>(H1, dOs + i0 * LDT, S0T + lane, 0, VT);
    fma_tile<4, 4, LDT, 1, LD, 32>(H2, dXs + i0 * LDT, S0T + lane, 0, VT);
    fma_tile<4, 4, LDT, 1, LD, 32>(H3, Us + i0 * LDT, dST + lane, 0, VT);
    fma_tile<4, 2, LDT, 1, 1, 32 * LDT>(OU, dOs + i0 * LDT, Us + lane * LDT, 0, VT);
    fma_tile<4, 2, LDT, 1, 1, 32 * LDT>(XU, dXs + i0 * LDT, Us + lane * LDT, 0, VT);
#pragma unroll
    for (int r = 0; r < 4; ++r) xv[r] = fmaf(dXs[(i0 + r) * LDT + lane], Vs[(i0 + r) * LDT + lane], xv[r]);
  }
  // Phase B: Q K^T, K K^T and the [C][C] adjoints F, E
  load_rows(a.q, a.io_dtype, t0, L, a.Hqk, hq, K, l2, Qn, LD);
  load_rows(a.k, a.io_dtype, t0, L, a.Hqk, hq, K, l2, Kn, LD);
  zero_cols(Qn, K);
  zero_cols(Kn, K);
  sd = warp_sum(sd);
  if (lane == 0) red[warp] = sd;
  if (threadIdx.x < C) {
    gm[threadIdx.x] = expf(G[threadIdx.x]);
    lm[threadIdx.x] = expf(G[L - 1] - G[threadIdx.x]);
  }
  __syncthreads();
  float rz[4], dba[4];
  {
    float QK[4][2], KK[4][2];
    zero(QK);
    zero(KK);
    fma_tile<4, 2, LD, 1, 1, 32 * LD>(QK, Qn + i0 * LD, Kn + lane * LD, 0, K);
    fma_tile<4, 2, LD, 1, 1, 32 * LD>(KK, Kn + i0 * LD, Kn + lane * LD, 0, K);
    float cz[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r;
      rz[r] = 0.f;
      dba[r] = 0.f;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int j = lane + 32 * m;
        const float gij = j <= i ? expf(G[i] - G[j]) : 0.f;
        const float f = a.scale * OU[r][m] * gij;
        const float dA = j < i ? -XU[r][m] : 0.f;
        const float e = bt[i] * gij * dA;
        const float z = f * QK[r][m] + e * KK[r][m];
        rz[r] += z;
        cz[m] += z;
        dba[r] = fmaf(dA * gij, KK[r][m], dba[r]);
        Fs[i * LDC + j] = f;
        Es[i * LDC + j] = e;
      }
    }
    colp[warp * C + lane] = cz[0];
    colp[warp * C + lane + 32] = cz[1];
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    rz[r] = warp_sum(rz[r]);
    dba[r] = warp_sum(dba[r]);
    xv[r] = warp_sum(xv[r]);
  }
  // row dots with the V-reduced products (q_i . S0 dO_i, k_i . S0 dX_i, k_i . dS u'_i)
  float qh1[4], kh2[4], kh3[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float qv = Qn[(i0 + r) * LD + lane + 32 * m], kv = Kn[(i0 + r) * LD + lane + 32 * m];
      x1 = fmaf(qv, H1[r][m], x1);
      x2 = fmaf(kv, H2[r][m], x2);
      x3 = fmaf(kv, H3[r][m], x3);
    }
    qh1[r] = warp_sum(x1);
    kh2[r] = warp_sum(x2);
    kh3[r] = warp_sum(x3);
  }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r;
      const float omega = lm[i] * kh3[r];
      om[i] = i < L ? omega : 0.f;
      dGr[i] = a.scale * gm[i] * qh1[r] - bt[i] * gm[i] * kh2[r] - omega + rz[r];
      dbr[i] = xv[r] - gm[i] * kh2[r] + dba[r];
    }
  }
  __syncthreads();
  // Phase C: dQ, dK per value head
  {
    float dQ[4][4], dK[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int i = i0 + r;
        dQ[r][m] = a.scale * gm[i] * H1[r][m];
        dK[r][m] = lm[i] * H3[r][m] - gm[i] * bt[i] * H2[r][m];
      }
    fma_tile<4, 4, LDC, 1, LD, 32>(dQ, Fs + i0 * LDC, Kn + lane, 0, i0 + 4);  // F K       (j <= i)
    fma_tile<4, 4, 1, LDC, LD, 32>(dK, Fs + i0, Qn + lane, i0, C);            // F^T Q     (j >= i)
    fma_tile<4, 4, LDC, 1, LD, 32>(dK, Es + i0 * LDC, Kn + lane, 0, i0 + 4);  // E K       (j < i)
    fma_tile<4, 4, 1, LDC, LD, 32>(dK, Es + i0, Kn + lane, i0, C);            // E^T K     (j > i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r;
      if (i >= L) continue;
      float* dq = ws.dQ + ((size_t)(t0 + i) * a.Hv + h) * K;
      float* dk = ws.dK + ((size_t)(t0 + i) * a.Hv + h) * K;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int d = lane + 32 * m;
        if (d < K) {
          dq[d] = dQ[r][m];
          dk[d] = dK[r][m];
        }
      }
    }
  }
  // dG: column sums in a fixed order, the exit-state terms on the last row, then the
  // reverse in-chunk cumulative sum
  if (threadIdx.x < C) {
    float s = 0.f;
    for (int w = 0; w < kGradWarps; ++w) s += colp[w * C + threadIdx.x];
    cs[threadIdx.x] = s;
  }
  __syncthreads();
  if (warp == 0) {
    float sdt = 0.f;
    for (int w = 0; w < kGradWarps; ++w) sdt += red[w];
    const float omsum = warp_sum(om[lane] + om[lane + 32]);
    float x0 = lane < L ? dGr[lane] - cs[lane] : 0.f;
    float x1 = lane + 32 < L ? dGr[lane + 32] - cs[lane + 32] : 0.f;
    const float extra = gm[L - 1] * sdt + omsum;
    if (lane == L - 1) x0 += extra;
    if (lane + 32 == L - 1) x1 += extra;
    // suffix sums: dg_i = sum_{j >= i} dG_j
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_down_sync(0xffffffffu, x0, o);
      const float y1 = __shfl_down_sync(0xffffffffu, x1, o);
      if (lane + o < 32) { x0 += y0; x1 += y1; }
    }
    x0 += __shfl_sync(0xffffffffu, x1, 0);
    const size_t base = (size_t)t0 * a.Hv + h;
    if (lane < L) {
      b.dg[base + (size_t)lane * a.Hv] = x0;
      b.dbeta[base + (size_t)lane * a.Hv] = dbr[lane];
    }
    if (lane + 32 < L) {
      b.dg[base + (size_t)(lane + 32) * a.Hv] = x1;
      b.dbeta[base + (size_t)(lane + 32) * a.Hv] = dbr[lane + 32];
    }
  }
}

// ---------------------------------------------------------------- 6. qk
constexpr int kQkThreads = 128;

__global__ void __launch_bounds__(kQkThreads) bwd_qk_kernel(const ChunkArgs a, const BwdArgs b,
                                                            BwdWs ws, int T_total) {
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.num_seqs, K = a.K, V = a.V;
  int covered = 0;
  if (ws.chunk_off[N + 1]) covered = a.cu_seqlens ? a.cu_seqlens[N] : N * a.T;
  const bool in = t < covered;
  const int grp = a.Hv / a.Hqk;
  const bool l2 = a.use_qk_l2norm != 0;
  for (int hq = warp; hq < a.Hqk; hq += kQkThreads / 32) {
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const void* x_src = which ? a.k : a.q;
      const float* dsrc = which ? ws.dK : ws.dQ;
      void* dst = which ? b.dk : b.dq;
      float dx[4], x[4];
      float ss = 0.f, xd = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int d = lane + 32 * m;
        dx[m] = 0.f;
        x[m] = 0.f;
        if (in && d < K) {
          for (int hh = hq * grp; hh < (hq + 1) * grp; ++hh)
            dx[m] += dsrc[((size_t)t * a.Hv + hh) * K + d];
          x[m] = load_elem(x_src, ((size_t)t * a.Hqk + hq) * K + d, a.io_dtype);
        }
        ss = fmaf(x[m], x[m], ss);
        xd = fmaf(x[m], dx[m], xd);
      }
      if (l2) {
        ss = warp_sum(ss);
        xd = warp_sum(xd);
        const float rho = 1.0f / sqrtf(ss + kL2Eps);
        const float c3 = rho * rho * rho * xd;
#pragma unroll
        for (int m = 0; m < 4; ++m) dx[m] = rho * dx[m] - c3 * x[m];
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int d = lane + 32 * m;
        if (d < K) store_elem(dst, ((size_t)t * a.Hqk + hq) * K + d, dx[m], a.io_dtype);
      }
    }
  }
  if (!in) {  // tokens outside every sequence: zero gradients
    for (int e = threadIdx.x; e < a.Hv * V; e += kQkThreads)
      store_elem(b.dv, (size_t)t * a.Hv * V + e, 0.f, a.io_dtype);
    for (int e = threadIdx.x; e < a.Hv; e += kQkThreads) {
      b.dg[(size_t)t * a.Hv + e] = 0.f;
      b.dbeta[(size_t)t * a.Hv + e] = 0.f;
    }
  }
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V) {
  size_t total = 0;
  bwd_layout(nullptr, max_chunks(T_total, num_seqs), num_seqs, Hv, K, V, T_total, &total);
  return total;
}

cudaError_t launch_chunk_bwd(const ChunkArgs& a_in, const BwdArgs& b) {
  ChunkArgs a = a_in;
  a.final_state = nullptr;  // the forward state pass records entry states only
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  const long long NC = max_chunks(T_total, a.num_seqs);
  BwdWs ws = bwd_layout(a.workspace, NC, a.num_seqs, a.Hv, a.K, a.V, T_total, nullptr);
  cudaError_t err;
  if ((err = cudaFuncSetAttribute(bwd_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem))) return err;
  if ((err = cudaFuncSetAttribute(bwd_reverse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRevSmem))) return err;
  if ((err = cudaFuncSetAttribute(bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmem))) return err;
  chunk_table_kernel<<<1, 1024, 0, a.stream>>>(a, ws.chunk_off);
  if ((err = cudaGetLastError())) return err;
  // Forward recompute of the state entering every chunk and of U'.  bf16 with K = V = 128:
  // the tensor-core kernel in record mode (its output goes to scratch that the dQ buffer
  // reuses later); otherwise the fp32 state pass on W, U from the prep kernel.
  const bool tc = chunk_tc_supported(a.K, a.V, a.io_dtype, a.beta_dtype) &&
                  a.gates.mode == kGatesGiven;
  if (tc && T_total > 0) {
    ChunkArgs f = a;
    f.o = ws.dQ;   // [T_total][Hv][V] bf16 fits in [T_total][Hv][K] fp32
    f.rec_states = ws.S;
    f.rec_u = ws.U;
    f.rec_chunk_off = ws.chunk_off;
    if ((err = launch_chunk_tc(f))) return err;
  }
  if (NC > 0) {
    bwd_prep_kernel<<<dim3((unsigned)NC, a.Hv), kPrepThreads, kPrepSmem, a.stream>>>(a, b, ws,
                                                                                      tc ? 0 : 1);
    if ((err = cudaGetLastError())) return err;
  }
  if (!tc && (err = launch_chunk_states(a, ws.chunk_off, ws.W, ws.U, ws.G, ws.S))) return err;
  const unsigned vtiles = (unsigned)((a.V + VT - 1) / VT);
  if (a.num_seqs > 0) {
    const long long blocks = (long long)vtiles * a.Hv * a.num_seqs;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    bwd_reverse_kernel<<<(unsigned)blocks, kRevThreads, kRevSmem, a.stream>>>(a, b, ws);
    if ((err = cudaGetLastError())) return err;
  }
  if (NC > 0) {
    bwd_grad_kernel<<<dim3((unsigned)NC, a.Hv), kGradThreads, kGradSmem, a.stream>>>(a, b, ws);
    if ((err = cudaGetLastError())) return err;
  }
  if (T_total > 0) {
    bwd_qk_kernel<<<T_total, kQkThreads, 0, a.stream>>>(a, b, ws, T_total);
    if ((err = cudaGetLastError())) return err;
  }
  return cudaSuccess;
}

}  // namespace gdn
