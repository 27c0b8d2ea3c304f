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
// Launches on the caller's stream, no host sync and no atomics (the result is
// bitwise reproducible run to run).  Two paths: bf16 with K = V = 128 runs every product on
// the tcgen05 tensor cores (bf16 operands, fp32 accumulators), everything else in fp32 on the
// CUDA cores.
//   1. chunk table  from cu_seqlens, on the device
//   2. states       the forward recompute of the state entering every chunk and of U':
//                   tensor cores: the forward kernel in record mode (bf16 operand tiles, and
//                   for the reverse pass T^T, P and its per-token vectors);
//                   CUDA cores: the prep and state passes of the fp32 chunk path
//   3. prep         CUDA cores only, per (chunk, value head): T = (I + A)^{-1},
//                   dUp = scale P^T dO, Z = scale Q^T diag(gamma) dO
//   4. reverse      chunks last to first, recording dS (the gradient of each chunk's exit
//                   state) and dX, writing dv and the row dots dX_i . v_i; tensor cores: one
//                   CTA per (sequence, value head), dS^T in TMEM; CUDA cores: per (sequence,
//                   value head, 32 columns)
//   5. grad         dbeta, dg; tensor cores: per (chunk, query/key head), the group's value
//                   heads summed in TMEM and the L2-norm Jacobian applied -> dq, dk; CUDA
//                   cores: per (chunk, value head), dQ, dK per value head
//   6. qk           CUDA cores: per (token, query/key head), the group sum and the L2-norm
//                   Jacobian -> dq, dk; zero gradients for tokens outside every sequence
//                   (tensor cores: only that zeroing)
#include <string.h>

#include "gdn_chunk_util.cuh"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;
constexpr int KP = GDN_MAX_HEAD_DIM;  // tiles are padded to the largest head dim
constexpr int LD = KP + 1;            // row stride of [C][KP] tiles (odd: column reads hit distinct banks)
constexpr int LDC = C + 1;            // row stride of [C][C] tiles
constexpr int VT = 32;                // V columns per V tile

// Scratch of the backward.  The fp32 path keeps fp32 tiles in every slot; the tensor-core path
// (bf16, K = V = 128) keeps bf16 operand tiles in the S, dS, U, dX slots (half the fp32 size:
// the per-(chunk, head) strides sS, sdS, sU, sdX are in floats), T^T and P together in the T
// slot, the reverse pass's per-token vectors in the G slot, and has no W, dUp, Z or per-token dQ,
// dK.
struct BwdWs {
  int32_t* chunk_off;  // [N + 2]
  float* W;            // [NC][Hv][C][K]          (fp32 path)
  float* U;            // [NC][Hv][C][V]  U, then U'
  float* G;            // [NC][Hv][C] (fp32 path); [NC][Hv][kRvFloats] (tensor-core path)
  float* S;            // [NC][Hv][K][V]  state at chunk entry
  float* T;            // [NC][Hv][C][C]
  float* dUp;          // [NC][Hv][C][V]  scale P^T dO   (fp32 path)
  float* dS;           // [NC][Hv][K][V]  gradient of the chunk's exit state
  float* dX;           // [NC][Hv][C][V]
  float* Z;            // [NC][Hv][K][V]  scale Q^T diag(gamma) dO   (fp32 path)
  float* XV;           // [NC][Hv][4][C]  partial row dots dX_i . v_i per 32-column slice
  float* dQ;           // [T_total][Hv][K] per value head, before the norm   (fp32 path)
  float* dK;           // [T_total][Hv][K]                                   (fp32 path)
  size_t sS, sdS, sU, sdX;   // slot strides (floats) per (chunk, head) of S, dS, U, dX
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Stage timestamps of the tensor-core reverse and grad passes (a diagnostic build,
// -DGDN_CHUNK_STAMPS): thread 0 records clock64 at the stage boundaries of iterations 32 .. 95
// in the first eight CTAs of the reverse pass, and the grad pass's issuing thread (256) those of
// the first two value heads (slots 0 .. 12) and the epilogue (slots 13 .. 15 of head 0) in CTAs
// 4000 .. 4007
// (gdn_bwd_stamps_read copies them out).  Without the define the stamps compile to nothing.
#ifdef GDN_CHUNK_STAMPS
__device__ unsigned long long g_rev_stamps[8][64][16];
__device__ unsigned long long g_grad_stamps[8][2][16];
#define GDN_RSTAMP(p)                                                               \
  do {                                                                              \
    if (tid == 0 && blockIdx.x < 8 && it >= 32 && it < 96)                          \
      g_rev_stamps[blockIdx.x][it - 32][p] = clock64();                             \
  } while (0)
#define GDN_GSTAMP(hd, p)                                                           \
  do {                                                                              \
    if (tid == 256 && blockIdx.x >= 4000 && blockIdx.x < 4008 && (hd) < 2)          \
      g_grad_stamps[blockIdx.x - 4000][hd][p] = clock64();                          \
  } while (0)
#else
#define GDN_RSTAMP(p) \
  do {                \
  } while (0)
#define GDN_GSTAMP(hd, p) \
  do {                    \
  } while (0)
#endif

__host__ __device__ inline BwdWs bwd_layout(void* base, long long NC, int N, int Hv, int K, int V,
                                            long long T_total, bool tc, size_t* total) {
  BwdWs w;
  char* p = reinterpret_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = p + off;
    off = align256(off + bytes);
    return r;
  };
  const size_t f = sizeof(float), ch = (size_t)NC * Hv;
  const size_t tile = tc ? 2 : 1;   // bf16 tiles take half an fp32 slot
  w.sS = w.sdS = (size_t)K * V / tile;
  w.sU = w.sdX = (size_t)C * V / tile;
  w.chunk_off = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)(N + 2)));
  w.W = tc ? nullptr : reinterpret_cast<float*>(take(f * ch * C * K));
  w.U = reinterpret_cast<float*>(take(f * ch * w.sU));
  w.G = reinterpret_cast<float*>(take(f * ch * (tc ? kRvFloats : C)));
  w.S = reinterpret_cast<float*>(take(f * ch * w.sS));
  w.T = reinterpret_cast<float*>(take(f * ch * C * C));
  w.dUp = tc ? nullptr : reinterpret_cast<float*>(take(f * ch * C * V));
  w.dS = reinterpret_cast<float*>(take(f * ch * w.sdS));
  w.dX = reinterpret_cast<float*>(take(f * ch * w.sdX));
  w.Z = tc ? nullptr : reinterpret_cast<float*>(take(f * ch * K * V));
  w.XV = reinterpret_cast<float*>(take(f * ch * 4 * C));
  w.dQ = tc ? nullptr : reinterpret_cast<float*>(take(f * (size_t)T_total * Hv * K));
  w.dK = tc ? nullptr : reinterpret_cast<float*>(take(f * (size_t)T_total * Hv * K));
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
// Per (chunk, value head), 16 warps, two CTAs per SM: A and P, T = (I + A)^{-1} (in place of
// A), dUp = scale P^T dO and Z = scale Q^T diag(gamma) dO -- the part of the state-gradient
// step that does not depend on the state gradient, taken out of the serial reverse pass.
// dO is taken in two halves of 64 columns.
constexpr int kPrepThreads = 512;
constexpr int HW = KP / 2;        // dO columns per half
constexpr int HLD = HW + 4;       // row stride of the dO half (float4 reads)
constexpr size_t kPrepSmem = sizeof(float) * (2 * C * LD + C * HLD + C * LDC + 3 * C);
constexpr int kBarT = 1;          // named barrier of the two warps that build T

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }


__device__ __forceinline__ void load4(const void* p, size_t i, int dtype, float (&x)[4]) {
  if (dtype == GDN_BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p) + i);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const float4 v = ld4(reinterpret_cast<const float*>(p) + i);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
}

__device__ __forceinline__ void store4(void* p, size_t i, int dtype, const float (&x)[4]) {
  if (dtype == GDN_BF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p) + i) = u;
  } else {
    st4(reinterpret_cast<float*>(p) + i, make_float4(x[0], x[1], x[2], x[3]));
  }
}


__global__ void __launch_bounds__(kPrepThreads, 2) bwd_prep_kernel(const ChunkArgs a,
                                                                   const BwdArgs b, BwdWs ws) {
  extern __shared__ float smem[];
  float* Kn = smem;           // [C][LD] normalised k
  float* P = smem;            // [C][LDC] P, over Kn once A and P are formed
  float* Qn = Kn + C * LD;    // [C][LD] normalised q
  float* Dh = Qn + C * LD;    // [C][HLD] one half of dO's columns
  float* At = Dh + C * HLD;   // [C][LDC] A, then T in place
  float* G = At + C * LDC;    // [C]
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
  load_tile(b.d_o, a.io_dtype, t0, L, a.Hv, h, V, 0, HW, nullptr, Dh, HLD, 0, kPrepThreads / 32);
  load_gates(a, t0, L, h, G, bt);
  __syncthreads();
  if (tid < C) gm[tid] = expf(G[tid]);
  {  // A = strict_lower(diag(beta) K K^T * Gamma), P = (Q K^T * Gamma) on and below the
     // diagonal; warps whose rows all lie below 32 skip the upper column half
    const int i0 = 4 * warp;
    float kk[4][2], qk[4][2];
    zero(kk);
    zero(qk);
    if (i0 + 3 < 32) {
      float k1[4][1], q1[4][1];
      zero(k1);
      zero(q1);
      fma_tile<4, 1, LD, 1, 1, 0>(k1, Kn + i0 * LD, Kn + lane * LD, 0, K);
      fma_tile<4, 1, LD, 1, 1, 0>(q1, Qn + i0 * LD, Kn + lane * LD, 0, K);
#pragma unroll
      for (int r = 0; r < 4; ++r) { kk[r][0] = k1[r][0]; qk[r][0] = q1[r][0]; }
    } else {
      fma_tile<4, 2, LD, 1, 1, 32 * LD>(kk, Kn + i0 * LD, Kn + lane * LD, 0, K);
      fma_tile<4, 2, LD, 1, 1, 32 * LD>(qk, Qn + i0 * LD, Kn + lane * LD, 0, K);
    }
    __syncthreads();  // every read of Kn is done: P may overwrite it
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int i = i0 + r, j = lane + 32 * m;
        const float gij = j <= i ? expf(G[i] - G[j]) : 0.f;
        At[i * LDC + j] = j < i ? bt[i] * kk[r][m] * gij : 0.f;
        P[i * LDC + j] = qk[r][m] * gij;
      }
  }
  __syncthreads();
  if (tid < C) {
    // T = (I + A)^{-1} in place, row by row, one column per thread: row i of T needs row i of
    // A and rows < i of T (own column); after the row's reads a barrier, then the row is written
    const int j = tid;
    for (int i = 0; i < C; ++i) {
      float t = i == j ? 1.f : 0.f;
      if (i > j) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int m = j;
        for (; m + 3 < i; m += 4) {
          s0 = fmaf(At[i * LDC + m], At[m * LDC + j], s0);
          s1 = fmaf(At[i * LDC + m + 1], At[(m + 1) * LDC + j], s1);
          s2 = fmaf(At[i * LDC + m + 2], At[(m + 2) * LDC + j], s2);
          s3 = fmaf(At[i * LDC + m + 3], At[(m + 3) * LDC + j], s3);
        }
        for (; m < i; ++m) s0 = fmaf(At[i * LDC + m], At[m * LDC + j], s0);
        t = -((s0 + s1) + (s2 + s3));
      }
      asm volatile("bar.sync %0, %1;" ::"n"(kBarT), "n"(C) : "memory");
      At[i * LDC + j] = t;
    }
  }
  const size_t ch = (size_t)c * a.Hv + h;
  const int ty = tid >> 4, tx = tid & 15;   // Z: 32 row groups x 16 groups of 4 columns
  for (int half = 0; half < 2; ++half) {
    if (half == 1) {
      __syncthreads();   // every read of the first half is done
      load_tile(b.d_o, a.io_dtype, t0, L, a.Hv, h, V, HW, HW, nullptr, Dh, HLD, 0,
                kPrepThreads / 32);
      __syncthreads();
    }
    const int cbase = half * HW;
    {  // Z = scale Q^T diag(gamma) dO: rows d = ty + 32 r, columns cbase + 4 tx .. + 3
      float z[4][4];
      zero(z);
      for (int i = 0; i < L; ++i) {
        const float g = gm[i];
        const float4 y4 = ld4(Dh + i * HLD + 4 * tx);
        const float y[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float x = g * Qn[i * LD + ty + 32 * r];
#pragma unroll
          for (int q = 0; q < 4; ++q) z[r][q] = fmaf(x, y[q], z[r][q]);
        }
      }
      const int col = cbase + 4 * tx;
      float* Zg = ws.Z + ch * K * V;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = ty + 32 * r;
        if (d < K && col < V)
          st4(Zg + (size_t)d * V + col, make_float4(a.scale * z[r][0], a.scale * z[r][1],
                                                    a.scale * z[r][2], a.scale * z[r][3]));
      }
    }
    if (half == 0) __syncthreads();   // T (and P) complete before dUp's first use of P
    {  // dUp = scale P^T dO: rows i = ty, ty + 32, columns cbase + 4 tx .. + 3 (P[m][i] = 0, m < i)
      float u[2][4];
      zero(u);
      for (int m = ty; m < C; ++m) {
        const float x0 = P[m * LDC + ty], x1 = P[m * LDC + ty + 32];
        const float4 y4 = ld4(Dh + m * HLD + 4 * tx);
        const float y[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          u[0][q] = fmaf(x0, y[q], u[0][q]);
          u[1][q] = fmaf(x1, y[q], u[1][q]);
        }
      }
      const int col = cbase + 4 * tx;
      float* Ug = ws.dUp + ch * C * V;
      if (col < V) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
          st4(Ug + (size_t)(ty + 32 * r) * V + col,
              make_float4(a.scale * u[r][0], a.scale * u[r][1], a.scale * u[r][2], a.scale * u[r][3]));
      }
    }
    if (cbase + HW >= V) break;   // V <= 64: one half holds every column
  }
  for (int e = tid; e < C * C; e += kPrepThreads) {
    const int i = e / C, j = e - i * C;
    ws.T[ch * C * C + e] = At[i * LDC + j];
  }
  if (tid < C) ws.G[ch * C + tid] = G[tid];
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

// The pass also writes dv = diag(beta) dX and the per-slice partial row dots dX_i . v_i.
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
    // normalised k rows into Kn and Kt (warp w: rows w + 8 s; every load issued first)
    {
      float x[C / (kRevThreads / 32)][4];
#pragma unroll
      for (int s8 = 0; s8 < C / (kRevThreads / 32); ++s8) {
        const int r = warp + (kRevThreads / 32) * s8;
#pragma unroll
        for (int m = 0; m < 4; ++m) {   // lane takes features lane + 32 m
          const int d = lane + 32 * m;
          x[s8][m] = (r < L && d < K) ? load_elem(a.k, ((size_t)(t0 + r) * a.Hqk + hq) * K + d, a.io_dtype) : 0.f;
        }
      }
#pragma unroll
      for (int s8 = 0; s8 < C / (kRevThreads / 32); ++s8) {
        const int r = warp + (kRevThreads / 32) * s8;
        if (l2) {
          float ss = 0.f;
#pragma unroll
          for (int m = 0; m < 4; ++m) ss = fmaf(x[s8][m], x[s8][m], ss);
          const float rn = 1.0f / sqrtf(warp_sum(ss) + kL2Eps);
#pragma unroll
          for (int m = 0; m < 4; ++m) x[s8][m] *= rn;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int d = lane + 32 * m;
          Kn[r * KLD + d] = x[s8][m];
          Kt[d * TLD + r] = x[s8][m];
        }
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
        float xv = 0.f;
        if (colok) {
          st4(dXg + (size_t)i * V + col, make_float4(x[r][0], x[r][1], x[r][2], x[r][3]));
          if (i < L) {   // dv = beta dX; partial dX . v over this thread's four columns
            const size_t tv = ((size_t)(t0 + i) * a.Hv + h) * V + col;
            const float bi = bt[i];
            const float dv4[4] = {bi * x[r][0], bi * x[r][1], bi * x[r][2], bi * x[r][3]};
            store4(b.dv, tv, a.io_dtype, dv4);
            float v4[4];
            load4(a.v, tv, a.io_dtype, v4);
            xv = x[r][0] * v4[0] + x[r][1] * v4[1] + x[r][2] * v4[2] + x[r][3] * v4[3];
          }
        }
        // the eight threads of a row (tx = lane % 8) add their partials in a fixed order
        xv += __shfl_xor_sync(0xffffffffu, xv, 1);
        xv += __shfl_xor_sync(0xffffffffu, xv, 2);
        xv += __shfl_xor_sync(0xffffffffu, xv, 4);
        if (tx == 0) ws.XV[(ch * 4 + (size_t)(c0 / VT)) * C + i] = xv;
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
// Per (chunk, value head), 16 warps.  Every product runs on 4 x 4 (or 4 x 2) register blocks
// with lanes arranged 4 x 8 inside the warp and both operands read as float4 (float2) rows
// of shared-memory tiles stored with the reduction index outermost, so that each k step costs
// one broadcast-like and one contiguous wavefront per operand.
//   [C][KP] outputs (H layout): warp w -> rows 16 (w / 4) + 4 ly, columns 32 (w % 4) + 4 lx
//   [C][C]  outputs (S layout): warp w -> rows 16 (w / 4) + 4 ly, columns 16 (w % 4) + 2 lx
// with ly = lane / 8, lx = lane % 8.  Shared memory: region R1 holds the V tiles of phase A
// (S0, dS transposed, and dO, dX, U' transposed), then q, k transposed (phase B), then
// F, F^T, E, E^T (phase C); region R2 holds the normalised q, k rows for the whole CTA.
// Phase A: H1 = dO S0^T, H2 = dX S0^T, H3 = U' dS^T, dO U'^T, dX U'^T (reduce over V);
// phase B: Q K^T, K K^T, then F, E and the row / column sums of Z (reduce over K);
// phase C: dQ += F K, dK += F^T Q + (E + E^T) K (reduce over the chunk's tokens).
constexpr int kGradThreads = 512;
constexpr int kGradWarps = kGradThreads / 32;
constexpr int RLD = C + 4;  // row stride of tiles indexed by token (float4 along tokens)
constexpr int kR1A = 2 * VT * KLD + 3 * VT * RLD;
constexpr int kR1B = 2 * KP * RLD;
constexpr int kR1C = 4 * C * RLD;
constexpr int kR1 = kR1A > kR1B ? (kR1A > kR1C ? kR1A : kR1C) : (kR1B > kR1C ? kR1B : kR1C);
constexpr int kR2 = 2 * C * KLD;
constexpr int kGradVec = 16 * C + kGradWarps;   // G, beta, gamma, lambda; 3 x [4][C]; red
constexpr size_t kGradSmem = sizeof(float) * (kR1 + kR2 + kGradVec);

__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }

__global__ void __launch_bounds__(kGradThreads) bwd_grad_kernel(const ChunkArgs a, const BwdArgs b,
                                                                BwdWs ws) {
  extern __shared__ float smem[];
  float* R1 = smem;
  float* Qn = R1 + kR1;          // [C][KLD] normalised q rows
  float* Kn = Qn + C * KLD;      // [C][KLD] normalised k rows
  float* G = Kn + C * KLD;       // [C]
  float* bt = G + C;             // [C]
  float* gm = bt + C;            // [C] gamma
  float* lm = gm + C;            // [C] lambda
  float* rowp = lm + C;          // [4][C] row partial sums of Z (per column group of warps)
  float* colp = rowp + 4 * C;    // [4][C] column partial sums of Z (per row group of warps)
  float* dbp = colp + 4 * C;     // [4][C] partial sum_j dA_ij (K K^T * Gamma)_ij
  float* red = dbp + 4 * C;      // [warps] partial <S0, dS>
  // phase A views of R1
  float* S0T = R1;               // [VT][KLD]
  float* dST = S0T + VT * KLD;   // [VT][KLD]
  float* dOT = dST + VT * KLD;   // [VT][RLD]
  float* dXT = dOT + VT * RLD;   // [VT][RLD]
  float* UT = dXT + VT * RLD;    // [VT][RLD]
  // phase B / C views
  float* QT = R1;                // [KP][RLD]
  float* KT = QT + KP * RLD;     // [KP][RLD]
  float* Fs = R1;                // [C][RLD] F[i][j]
  float* FT = Fs + C * RLD;      // [C][RLD] F[j][i]
  float* Es = FT + C * RLD;      // [C][RLD] E[i][j]
  float* ET = Es + C * RLD;      // [C][RLD] E[j][i]

  const int c = blockIdx.x, h = blockIdx.y;
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  const int K = a.K, V = a.V, hq = h / (a.Hv / a.Hqk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ly = lane >> 3, lx = lane & 7;
  const int rS = 16 * (warp >> 2) + 4 * ly;     // first row of this thread (both layouts)
  const int cH = 32 * (warp & 3) + 4 * lx;      // first column, H layout
  const int cS = 16 * (warp & 3) + 2 * lx;      // first column, S layout
  const bool l2 = a.use_qk_l2norm != 0;
  const size_t ch = (size_t)c * a.Hv + h;

  // normalised q, k rows (warp w: rows 4 w .. 4 w + 3); every load issued before the norms
  load_gates(a, t0, L, h, G, bt);
  {
    float x[2][4][4];
#pragma unroll
    for (int which = 0; which < 2; ++which)
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int r = 4 * warp + r4, d = lane + 32 * m;
          x[which][r4][m] = (r < L && d < K)
                                ? load_elem(which ? a.k : a.q, ((size_t)(t0 + r) * a.Hqk + hq) * K + d,
                                            a.io_dtype)
                                : 0.f;
        }
#pragma unroll
    for (int which = 0; which < 2; ++which)
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(x[which][r4][m], x[which][r4][m], ss);
        const float rn = l2 ? 1.0f / sqrtf(warp_sum(ss) + kL2Eps) : 1.f;
        float* dst = (which ? Kn : Qn) + (4 * warp + r4) * KLD + lane;
#pragma unroll
        for (int m = 0; m < 4; ++m) dst[32 * m] = x[which][r4][m] * rn;
      }
  }
  __syncthreads();
  if (tid < C) {
    gm[tid] = expf(G[tid]);
    lm[tid] = expf(G[L - 1] - G[tid]);
  }

  // ---- phase A: products reducing over V, 32 columns at a time
  float H1[4][4], H2[4][4], H3[4][4], OU[4][2], XU[4][2];
  zero(H1);
  zero(H2);
  zero(H3);
  zero(OU);
  zero(XU);
  float sd = 0.f;
  const float* Sg = ws.S + ch * K * V;
  const float* dSg = ws.dS + ch * K * V;
  const float* Ug = ws.U + ch * C * V;
  const float* dXg = ws.dX + ch * C * V;
  for (int c0 = 0; c0 < V; c0 += VT) {
    __syncthreads();
    {  // S0, dS tiles transposed: thread -> row d = tid % 128, columns 8 (tid / 128) + 0..7
      const int d = tid & 127, cg = tid >> 7;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int cc = 8 * cg + 4 * hlf;
        float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), ds = s0;
        if (d < K && c0 + cc < V) {
          s0 = ld4(Sg + (size_t)d * V + c0 + cc);
          ds = ld4(dSg + (size_t)d * V + c0 + cc);
        }
        S0T[(cc + 0) * KLD + d] = s0.x; S0T[(cc + 1) * KLD + d] = s0.y;
        S0T[(cc + 2) * KLD + d] = s0.z; S0T[(cc + 3) * KLD + d] = s0.w;
        dST[(cc + 0) * KLD + d] = ds.x; dST[(cc + 1) * KLD + d] = ds.y;
        dST[(cc + 2) * KLD + d] = ds.z; dST[(cc + 3) * KLD + d] = ds.w;
        sd = fmaf(s0.x, ds.x, fmaf(s0.y, ds.y, fmaf(s0.z, ds.z, fmaf(s0.w, ds.w, sd))));
      }
    }
    {  // dO, dX, U', v tiles transposed: thread -> token i = tid % 64, columns 4 (tid / 64) + 0..3
      const int i = tid & 63, cg = tid >> 6;
      const int cc = 4 * cg;
      const bool ok = i < L && c0 + cc < V;
      const size_t tv = ((size_t)(t0 + i) * a.Hv + h) * V + c0 + cc;
      float o4[4] = {0.f, 0.f, 0.f, 0.f};
      float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f), u4 = x4;
      if (ok) {
        x4 = ld4(dXg + (size_t)i * V + c0 + cc);
        u4 = ld4(Ug + (size_t)i * V + c0 + cc);
#pragma unroll
        for (int q = 0; q < 4; ++q) o4[q] = load_elem(b.d_o, tv + q, a.io_dtype);
      }
      const float x[4] = {x4.x, x4.y, x4.z, x4.w}, u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dOT[(cc + q) * RLD + i] = o4[q];
        dXT[(cc + q) * RLD + i] = x[q];
        UT[(cc + q) * RLD + i] = u[q];
      }
    }
    __syncthreads();
#pragma unroll 2
    for (int k = 0; k < VT; ++k) {
      const float4 ao = ld4(dOT + k * RLD + rS), ax = ld4(dXT + k * RLD + rS);
      const float4 au = ld4(UT + k * RLD + rS);
      const float4 bs = ld4(S0T + k * KLD + cH), bd = ld4(dST + k * KLD + cH);
      const float2 bu = ld2(UT + k * RLD + cS);
      const float AO[4] = {ao.x, ao.y, ao.z, ao.w}, AX[4] = {ax.x, ax.y, ax.z, ax.w};
      const float AU[4] = {au.x, au.y, au.z, au.w};
      const float BS[4] = {bs.x, bs.y, bs.z, bs.w}, BD[4] = {bd.x, bd.y, bd.z, bd.w};
      const float BU[2] = {bu.x, bu.y};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          H1[r][q] = fmaf(AO[r], BS[q], H1[r][q]);
          H2[r][q] = fmaf(AX[r], BS[q], H2[r][q]);
          H3[r][q] = fmaf(AU[r], BD[q], H3[r][q]);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          OU[r][q] = fmaf(AO[r], BU[q], OU[r][q]);
          XU[r][q] = fmaf(AX[r], BU[q], XU[r][q]);
        }
      }
    }
  }
  // row dots of the V-reduced products with the normalised rows: q_i . S0 dO_i,
  // k_i . S0 dX_i, k_i . dS u'_i (H layout: partial over 4 columns, then over lx and the
  // four warps sharing the rows)
  float qh1[4], kh2[4], kh3[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float4 qv = ld4(Qn + (rS + r) * KLD + cH), kv = ld4(Kn + (rS + r) * KLD + cH);
    const float Q4[4] = {qv.x, qv.y, qv.z, qv.w}, K4[4] = {kv.x, kv.y, kv.z, kv.w};
    float x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x1 = fmaf(Q4[q], H1[r][q], x1);
      x2 = fmaf(K4[q], H2[r][q], x2);
      x3 = fmaf(K4[q], H3[r][q], x3);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      x1 += __shfl_xor_sync(0xffffffffu, x1, o);
      x2 += __shfl_xor_sync(0xffffffffu, x2, o);
      x3 += __shfl_xor_sync(0xffffffffu, x3, o);
    }
    qh1[r] = x1;
    kh2[r] = x2;
    kh3[r] = x3;
  }
  // dQ, dK accumulators (H layout) start from the V-reduced terms
  float dQ[4][4], dK[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = rS + r;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dQ[r][q] = a.scale * gm[i] * H1[r][q];
      dK[r][q] = lm[i] * H3[r][q] - gm[i] * bt[i] * H2[r][q];
    }
  }
  sd = warp_sum(sd);
  if (lane == 0) red[warp] = sd;
  // partial row dots to shared memory, in the rowp / colp / dbp space (free until phase B)
  float* rd1 = colp;   // [4][C]
  float* rd2 = dbp;    // [4][C]
  float* rd3 = rowp;   // [4][C]
  if (lx == 0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      rd1[(warp & 3) * C + rS + r] = qh1[r];
      rd2[(warp & 3) * C + rS + r] = kh2[r];
      rd3[(warp & 3) * C + rS + r] = kh3[r];
    }
  }
  __syncthreads();   // phase A tiles are dead; rd* written
  // the row dots summed in a fixed order, one token per thread (threads < C)
  float qh1_i = 0.f, kh2_i = 0.f, kh3_i = 0.f;
  if (tid < C) {
    qh1_i = rd1[tid] + rd1[C + tid] + rd1[2 * C + tid] + rd1[3 * C + tid];
    kh2_i = rd2[tid] + rd2[C + tid] + rd2[2 * C + tid] + rd2[3 * C + tid];
    kh3_i = rd3[tid] + rd3[C + tid] + rd3[2 * C + tid] + rd3[3 * C + tid];
  }
  // ---- phase B: q, k transposed into R1; Q K^T, K K^T in the S layout
  {
    const int i = tid & 63, dg = tid >> 6;   // token i, features 16 dg .. 16 dg + 15
#pragma unroll 4
    for (int e = 0; e < 16; ++e) {
      const int d = 16 * dg + e;
      QT[d * RLD + i] = Qn[i * KLD + d];
      KT[d * RLD + i] = Kn[i * KLD + d];
    }
  }
  __syncthreads();
  float QK[4][2], KK[4][2];
  zero(QK);
  zero(KK);
#pragma unroll 4
  for (int d = 0; d < K; ++d) {
    const float4 aq = ld4(QT + d * RLD + rS), ak = ld4(KT + d * RLD + rS);
    const float2 bk = ld2(KT + d * RLD + cS);
    const float AQ[4] = {aq.x, aq.y, aq.z, aq.w}, AK[4] = {ak.x, ak.y, ak.z, ak.w};
    const float BK[2] = {bk.x, bk.y};
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        QK[r][q] = fmaf(AQ[r], BK[q], QK[r][q]);
        KK[r][q] = fmaf(AK[r], BK[q], KK[r][q]);
      }
  }
  float F[4][2], E[4][2], rz[4], dba[4], cz[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = rS + r;
    rz[r] = 0.f;
    dba[r] = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = cS + q;
      const float gij = j <= i ? expf(G[i] - G[j]) : 0.f;
      const float f = a.scale * OU[r][q] * gij;
      const float dA = j < i ? -XU[r][q] : 0.f;
      const float e = bt[i] * gij * dA;
      const float z = f * QK[r][q] + e * KK[r][q];
      F[r][q] = f;
      E[r][q] = e;
      rz[r] += z;
      cz[q] += z;
      dba[r] = fmaf(dA * gij, KK[r][q], dba[r]);
    }
  }
  // reduce: rows over lx (xor 1, 2, 4), columns over ly (xor 8, 16)
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      rz[r] += __shfl_xor_sync(0xffffffffu, rz[r], o);
      dba[r] += __shfl_xor_sync(0xffffffffu, dba[r], o);
    }
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) cz[q] += __shfl_xor_sync(0xffffffffu, cz[q], o);
  __syncthreads();   // Q^T, K^T reads done (F, E overwrite them); rd* reads done
  if (lx == 0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      rowp[(warp & 3) * C + rS + r] = rz[r];
      dbp[(warp & 3) * C + rS + r] = dba[r];
    }
  }
  if (ly == 0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) colp[(warp >> 2) * C + cS + q] = cz[q];
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int j = cS + q;
    st4(FT + j * RLD + rS, make_float4(F[0][q], F[1][q], F[2][q], F[3][q]));
    st4(ET + j * RLD + rS, make_float4(E[0][q], E[1][q], E[2][q], E[3][q]));
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    *reinterpret_cast<float2*>(Fs + (rS + r) * RLD + cS) = make_float2(F[r][0], F[r][1]);
    *reinterpret_cast<float2*>(Es + (rS + r) * RLD + cS) = make_float2(E[r][0], E[r][1]);
  }
  __syncthreads();
  // ---- phase C: dQ += F K;  dK += F^T Q + (E + E^T) K   (H layout)
#pragma unroll 2
  for (int j = 0; j < C; ++j) {
    const float4 f1 = ld4(FT + j * RLD + rS);   // F[i][j]
    const float4 f2 = ld4(Fs + j * RLD + rS);   // F[j][i]
    const float4 e1 = ld4(ET + j * RLD + rS);   // E[i][j]
    const float4 e2 = ld4(Es + j * RLD + rS);   // E[j][i]
    const float4 bk = ld4(Kn + j * KLD + cH), bq = ld4(Qn + j * KLD + cH);
    const float A1[4] = {f1.x, f1.y, f1.z, f1.w}, A2[4] = {f2.x, f2.y, f2.z, f2.w};
    const float A3[4] = {e1.x + e2.x, e1.y + e2.y, e1.z + e2.z, e1.w + e2.w};
    const float BK[4] = {bk.x, bk.y, bk.z, bk.w}, BQ[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dQ[r][q] = fmaf(A1[r], BK[q], dQ[r][q]);
        dK[r][q] = fmaf(A2[r], BQ[q], fmaf(A3[r], BK[q], dK[r][q]));
      }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = rS + r;
    if (i >= L || cH >= K) continue;
    st4(ws.dQ + ((size_t)(t0 + i) * a.Hv + h) * K + cH, make_float4(dQ[r][0], dQ[r][1], dQ[r][2], dQ[r][3]));
    st4(ws.dK + ((size_t)(t0 + i) * a.Hv + h) * K + cH, make_float4(dK[r][0], dK[r][1], dK[r][2], dK[r][3]));
  }
  // ---- dG, dbeta per token (threads < C hold the row dots), then dg by a suffix sum
  float* dGv = Fs;    // [C] (phase C reads of F / E are done after the barrier)
  float* omv = Fs + C;
  __syncthreads();
  if (tid < C) {
    const int i = tid;
    float rsum = 0.f, csum = 0.f, db = 0.f, x = 0.f;
    for (int g = 0; g < 4; ++g) {
      rsum += rowp[g * C + i];
      csum += colp[g * C + i];
      db += dbp[g * C + i];
    }
    for (int g = 0; g < (V + VT - 1) / VT; ++g) x += ws.XV[(ch * 4 + g) * C + i];
    const float omega = i < L ? lm[i] * kh3_i : 0.f;
    omv[i] = omega;
    dGv[i] = i < L ? a.scale * gm[i] * qh1_i - bt[i] * gm[i] * kh2_i - omega + rsum - csum : 0.f;
    if (i < L) b.dbeta[((size_t)(t0 + i)) * a.Hv + h] = x - gm[i] * kh2_i + db;
  }
  __syncthreads();
  if (warp == 0) {
    float sdt = 0.f;
    for (int w = 0; w < kGradWarps; ++w) sdt += red[w];
    const float omsum = warp_sum(omv[lane] + omv[lane + 32]);
    float x0 = dGv[lane], x1 = dGv[lane + 32];
    const float extra = gm[L - 1] * sdt + omsum;
    if (lane == L - 1) x0 += extra;
    if (lane + 32 == L - 1) x1 += extra;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {   // suffix sums: dg_i = sum_{j >= i} dG_j
      const float y0 = __shfl_down_sync(0xffffffffu, x0, o);
      const float y1 = __shfl_down_sync(0xffffffffu, x1, o);
      if (lane + o < 32) { x0 += y0; x1 += y1; }
    }
    x0 += __shfl_sync(0xffffffffu, x1, 0);
    const size_t base = (size_t)t0 * a.Hv + h;
    if (lane < L) b.dg[base + (size_t)lane * a.Hv] = x0;
    if (lane + 32 < L) b.dg[base + (size_t)(lane + 32) * a.Hv] = x1;
  }
}

// ---------------------------------------------------------------- 5b. grad on the tensor cores
// bf16 I/O with K = V = 128: the same quantities as bwd_grad_kernel, with every product a
// tcgen05.mma (bf16 operands in 128-byte-swizzled shared memory, fp32 accumulators in TMEM;
// S0, dS, U', dX and the normalised q, k rounded to bf16 as the forward's tensor-core path
// rounds its operands).  One CTA (8 warps) per (chunk, query/key head), which takes the value
// heads of the group in order; TMEM columns:
//   R1 [0, 256)   [Q; K] [S0 | dS]        M=128 N=256 K=128  -> q_i . S0 dO_i, k_i . S0 dX_i,
//                                                               k_i . dS u'_i (row dots)
//   R2 [256, 320) [dO; dX] U'^T           M=128 N=64  K=128  -> F, dA (and E)
//   R3 [320, 384) [Q; K] K^T              M=128 N=64  K=128  -> Q K^T, K K^T (once: the same
//                                                               for every head of the group)
//   R4 [384, 512) [dQ; dK] += [scale gamma dO | 0 ; -gamma beta dX | lambda U'] [S0 | dS]^T
//                           + [F; E] K + [0; F^T] Q + [0; E^T] K          (K = 256, 64, 64, 64;
//                             the first A operand built as bf16 in R1's columns once the row dots
//                             have read them)
// R4 accumulates over the group's value heads, which gives the group sum of the gradients of
// the normalised q, k rows; the epilogue applies the L2 norm's Jacobian
// dq = r (dq^ - q^ (q^ . dq^)) and writes dq, dk as bf16.  F^T and E^T are MN-major A operands
// whose first 64-row block is a zero tile and whose second is F (resp. E) as stored row-major,
// so no transposed copy is built.
namespace tcg {

// Store 16 consecutive 32-bit columns of this thread's lane and wait for the store.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
using namespace sm100;
constexpr int kWorkThreads = 256;          // warps 0-7: two per TMEM lane quarter
constexpr int kThreads = kWorkThreads + 32;   // and warp 8, which issues the copies and the MMAs
constexpr int kIssuer = kWorkThreads;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t OFF_QK = 0;          // [q; k] rows, 2 k-halves x 128 rows x 128 B
constexpr uint32_t OFF_S0 = 32768;      // S0 rows d, 2 c-halves x 128 rows
constexpr uint32_t OFF_DS = 65536;      // dS rows d (right after S0: [S0 | dS] is one operand)
constexpr uint32_t OFF_OX = 98304;      // [dO; dX] rows
constexpr uint32_t OFF_U = 131072;      // U' rows j, 2 c-halves x 64 rows
constexpr uint32_t OFF_ZERO = 147456;   // 64 rows x 128 B of zeros
constexpr uint32_t OFF_FE = 155648;     // [F; E] rows, K = 64 tokens: 128 rows x 128 B
constexpr uint32_t OFF_VEC = 172032;    // fp32 per-token vectors and scratch, 28 x 64
constexpr uint32_t OFF_BAR = OFF_VEC + 28 * 64 * 4;
constexpr uint32_t SMEM = OFF_BAR + 64 + 1024;
static_assert(SMEM <= 232448, "shared memory budget");
constexpr uint32_t T_R1 = 0, T_R2 = 256, T_R3 = 320, T_R4 = 384, T_COLS = 512;
constexpr int kTmaThread = 160;   // issues the q, k loads and the TMA stores
constexpr int kTmemWarp = 4;      // allocates and frees the tensor memory

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
constexpr float kLog2eG = 1.4426950408889634f;
// 2^x on the special-function unit (the arguments are <= 0 where the value is kept).
__device__ __forceinline__ float ex2g(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// The 8 bf16 of a 16-byte chunk scaled by s.
__device__ __forceinline__ uint4 scaled8(uint4 v, float s) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[q]));
    w[q] = pack2(s * f.x, s * f.y);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// Scale the 8 bf16 of the 16-byte chunk at p by s.
__device__ __forceinline__ void scale8(uint8_t* p, float s) {
  *reinterpret_cast<uint4*>(p) = scaled8(*reinterpret_cast<const uint4*>(p), s);
}
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t lbo) {
  return sdesc_sw128(addr, lbo, 1024);
}

// The operand tiles of value head h (chunk unit ch, first token t0), issued by thread 0: part A,
// the rows [dO; dX] (dO by TMA, dX by bulk copy) and U' (bulk), on `bar_a`; part B, S0 and dS
// (bulk), on `bar_b`.  Part A's space is free once R4's operand has been built in TMEM, part B's
// once R4 has run.
__device__ __forceinline__ void issue_loads_a(uint8_t* sm, const BwdWs& ws, const CUtensorMap* tmO,
                                              uint64_t* bar_a, size_t ch, int h, int t0) {
  const uint8_t* ug = reinterpret_cast<const uint8_t*>(ws.U + ch * ws.sU);
  const uint8_t* xg = reinterpret_cast<const uint8_t*>(ws.dX + ch * ws.sdX);
  mbar_arrive_expect_tx(bar_a, 16384 + 16384 + 2 * 8192);
  bulk_load(sm + OFF_U, ug, 16384, bar_a);
  bulk_load(sm + OFF_OX + 8192, xg, 8192, bar_a);   // dX: rows 64-127 of [dO; dX]
  bulk_load(sm + OFF_OX + 16384 + 8192, xg + 8192, 8192, bar_a);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)   // 64 features x 64 tokens a box, zero past the last token
    tma_load_3d(sm + OFF_OX + hh * 16384, tmO, bar_a, 64 * hh, h, t0);
}
__device__ __forceinline__ void issue_loads_b(uint8_t* sm, const BwdWs& ws, uint64_t* bar_b, size_t ch) {
  mbar_arrive_expect_tx(bar_b, 2 * 32768);
  bulk_load(sm + OFF_S0, reinterpret_cast<const uint8_t*>(ws.S + ch * ws.sS), 32768, bar_b);
  bulk_load(sm + OFF_DS, reinterpret_cast<const uint8_t*>(ws.dS + ch * ws.sdS), 32768, bar_b);
}

__global__ void __launch_bounds__(kThreads, 1) bwd_grad_tc_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmDQ,
    const __grid_constant__ CUtensorMap tmDK, const ChunkArgs a, const BwdArgs b, BwdWs ws) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  float* vec = reinterpret_cast<float*>(sm + OFF_VEC);
  float* G = vec;              float* bt = vec + 64;    float* gm = vec + 128;  float* lm = vec + 192;
  float* qh1 = vec + 256;      float* kh2 = vec + 320;  float* kh3 = vec + 384;
  float* xvr = vec + 640;      float* red = vec + 704;
  float* dGv = vec + 768;      float* om = vec + 832;   float* g2 = vec + 896;
  float* rnv = vec + 1024;     // [128] the rows' L2-norm reciprocals (zero past the chunk end)
  float* colp = vec + 1152;    // [4 row quarters][64] column sums of Z; then [2][128] row dots
  float* dbp = vec + 1408;     // [2][64] partial dbeta terms
  float* rowp = vec + 1536;    // [2 column halves][128 rows] partial row sums of Z
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_a = reinterpret_cast<uint64_t*>(sm + OFF_BAR + 8);     // a head's dO, dX, U'
  uint64_t* bar_b = reinterpret_cast<uint64_t*>(sm + OFF_BAR + 16);    // a head's S0, dS
  uint64_t* bar_qk = reinterpret_cast<uint64_t*>(sm + OFF_BAR + 24);   // the group's q, k
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 32);
  // one CTA per (chunk, query/key head), heads fastest: the CTAs running together read the
  // same tokens (adjacent rows)
  const int Hqk = a.Hqk, Hv = a.Hv, grp = Hv / Hqk;
  const int hq = (int)(blockIdx.x % (unsigned)Hqk), c = (int)(blockIdx.x / (unsigned)Hqk);
  int n, t0, L;
  if (!locate_chunk(a, ws.chunk_off, c, &n, &t0, &L)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool l2 = a.use_qk_l2norm != 0;
  const uint32_t loff = (uint32_t)(32 * (warp & 3)) << 16;
  const int row = 32 * (warp & 3) + lane;   // this thread's TMEM lane
  if (tid == kIssuer) {
    mbar_init(bar, 1);
    mbar_init(bar_a, 1);
    mbar_init(bar_b, 1);
    mbar_init(bar_qk, 1);
    fence_mbar_init();
  }
  __syncthreads();   // the barriers are initialised before any copy is issued
  if (tid == kIssuer) {    // the first value head's tiles
    issue_loads_a(sm, ws, &tmO, bar_a, (size_t)c * Hv + hq * grp, hq * grp, t0);
    issue_loads_b(sm, ws, bar_b, (size_t)c * Hv + hq * grp);
  } else if (tid == kTmaThread) {   // the chunk's q, k rows into [q; k] by TMA
    mbar_arrive_expect_tx(bar_qk, 2 * 16384);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      tma_load_3d(sm + OFF_QK + hh * 16384, &tmQ, bar_qk, 64 * hh, hq, t0);
      tma_load_3d(sm + OFF_QK + hh * 16384 + 8192, &tmK, bar_qk, 64 * hh, hq, t0);
    }
  }
  if (warp == kTmemWarp) {
    tmem_alloc(tslot, T_COLS);
    tmem_relinquish();
  }
  for (int e = tid; e < 8192 / 16; e += kThreads)      // the zero tile
    reinterpret_cast<uint4*>(sm + OFF_ZERO)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;
  bool ok = true, failed = false;
  int last_a = 0, last_b = 0;   // the last heads whose part A / part B tiles were requested

  for (int hi = 0; hi < grp; ++hi) {
    const int h = hq * grp + hi;
    const size_t ch = (size_t)c * Hv + h;
    const uint32_t ph = (uint32_t)hi & 1u;   // phase of the head's loads
    // the gates (warp 1) and the row dots (warps 2-3) load while the copies land
    if (warp == 1) load_gates(a, t0, L, h, G, bt, lane);
    if (tid >= 64 && tid < 128)   // the row dots dX_i . v_i of the reverse pass (slot 0)
      xvr[tid - 64] = ws.XV[ch * 4 * 64 + tid - 64];
    GDN_GSTAMP(hi, 0);
    if (tid == kIssuer)   // landed
      ok = mbar_wait(bar_a, ph, kWaitNs) && mbar_wait(bar_b, ph, kWaitNs) &&
           (hi > 0 || mbar_wait(bar_qk, 0, kWaitNs));
    if (__syncthreads_or(!ok)) { failed = true; break; }
    GDN_GSTAMP(hi, 1);
    if (hi == 0 && tid < kWorkThreads) {  // [q; k] rows normalised in place (thread: one row
                                          // half, 128 rows x 2 halves)
      const int r = tid >> 1, hh = tid & 1, i = r & 63;
      uint8_t* rowq = sm + OFF_QK + hh * 16384 + r * 128;
      float ss = 0.f;
      // 16-byte chunks in an order rotated by the row (the warp's accesses spread over the
      // banks), kept in registers for the scaling
      uint4 u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) u[j] = *reinterpret_cast<const uint4*>(rowq + 16 * ((j + r) & 7));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      const float rn = i < L ? (l2 ? 1.0f / sqrtf(ss + kL2Eps) : 1.f) : 0.f;
      if (hh == 0) rnv[r] = rn;
#pragma unroll
      for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(rowq + 16 * ((j + r) & 7)) = scaled8(u[j], rn);
    }
    GDN_GSTAMP(hi, 2);
    if (L < C) {   // dO rows past the chunk end (the next sequence's) cleared
      for (int e = tid; e < 2 * 64 * 8; e += kThreads) {
        const int hf = e >> 9, ii = (e >> 3) & 63, c8 = e & 7;
        if (ii >= L)
          *reinterpret_cast<uint4*>(sm + OFF_OX + hf * 16384 + ii * 128 + 16 * c8) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    GDN_GSTAMP(hi, 3);
    // ---- R1, R2 (and R3 for the first head), issued first: the dot below runs meanwhile
    if (tid == kIssuer) {
      const uint32_t i1 = idesc_bf16(128, 256, false, true), i2 = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ko = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tb + T_R1, kdesc(sb + OFF_QK + ko), mndesc(sb + OFF_S0 + ks * 2048, 16384), i1, ks > 0);
        mma_bf16(tb + T_R2, kdesc(sb + OFF_OX + ko),
                 kdesc(sb + OFF_U + (ks >> 2) * 8192 + (ks & 3) * 32), i2, ks > 0);
        if (hi == 0)
          mma_bf16(tb + T_R3, kdesc(sb + OFF_QK + ko), kdesc(sb + OFF_QK + 8192 + ko), i2, ks > 0);
      }
      mma_commit(bar);
    }
    GDN_GSTAMP(hi, 4);
    if (tid < kWorkThreads) {  // <S0, dS> over the two tiles (same layout, element by element)
      float sd = 0.f;
      const uint4* p0 = reinterpret_cast<const uint4*>(sm + OFF_S0);
      const uint4* p1 = reinterpret_cast<const uint4*>(sm + OFF_DS);
#pragma unroll 4
      for (int e = tid; e < 32768 / 16; e += kWorkThreads) {
        const uint4 u0 = p0[e], u1 = p1[e];
        const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w}, w1[4] = {u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w0[q]));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w1[q]));
          sd = fmaf(f0.x, f1.x, fmaf(f0.y, f1.y, sd));
        }
      }
      sd = warp_sum(sd);
      if (lane == 0) red[warp] = sd;
    }
    if (tid < 64) {
      gm[tid] = expf(G[tid]);
      lm[tid] = expf(G[L - 1] - G[tid]);
      g2[tid] = G[tid] * kLog2eG;   // base-2 log-decay for the F / E factors
    }
    GDN_GSTAMP(hi, 5);
    if (tid == kIssuer) ok = mbar_wait(bar, 0, kWaitNs);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    GDN_GSTAMP(hi, 6);
    // ---- row dots from R1 (warps 0-3: the S0 columns; warps 6-7: the dS columns of k rows)
    if (warp < 4 || warp == 6 || warp == 7) {   // 8 columns of the bf16 row per 16-byte load
      const bool s0 = warp < 4;
      const uint8_t* tile = s0 ? sm + OFF_OX : sm + OFF_U;
      const uint32_t half = s0 ? 16384u : 8192u;
      const int r = s0 ? row : row - 64;
      float acc = 0.f;
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        float x[32];
        tmem_ld32(tb + loff + T_R1 + (s0 ? 0 : 128) + 32 * part, x);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int col = 32 * part + 8 * m;
          const uint4 u = *reinterpret_cast<const uint4*>(tile + (col >> 6) * half + sw128_offset(r, col & 63));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
            acc = fmaf(x[8 * m + 2 * q], f.x, fmaf(x[8 * m + 2 * q + 1], f.y, acc));
          }
        }
      }
      if (!s0) kh3[row - 64] = acc;
      else if (row < 64) qh1[row] = acc;
      else kh2[row - 64] = acc;
    }
    tc_fence_before();
    __syncthreads();   // R1 has been read out: its columns take R4's operand
    tc_fence_after();
    GDN_GSTAMP(hi, 7);
    // ---- R4's A operand in TMEM, in R1's columns (read out by the row dots):
    //      [scale gamma dO | 0 ; -gamma beta dX | lambda U'] as bf16 pairs, K = 256 (the v of S0,
    //      then the v of dS); thread: its TMEM lane's row, the v half warp / 4 of each part.  A
    //      row's 16-byte chunks sit at chunk ^ (row % 8), so the warp's reads of one chunk index
    //      spread over the banks.
    if (warp < 8) {
      const int g = warp >> 2;
      float pk[32];
      {
        const float sc = row < 64 ? a.scale * gm[row] : -gm[row - 64] * bt[row - 64];
        const uint8_t* orow = sm + OFF_OX + g * 16384 + row * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint4 u = *reinterpret_cast<const uint4*>(orow + ((c8 ^ (row & 7)) << 4));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
            pk[4 * c8 + q] = __uint_as_float(pack2(sc * f.x, sc * f.y));
          }
        }
        tmem_st32(tb + loff + T_R1 + 32 * g, pk);
      }
      if (row < 64) {
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = 0.f;
      } else {
        const int i = row - 64;
        const float li = lm[i];
        const uint8_t* urow = sm + OFF_U + g * 8192 + i * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint4 u = *reinterpret_cast<const uint4*>(urow + ((c8 ^ (i & 7)) << 4));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
            pk[4 * c8 + q] = __uint_as_float(pack2(li * f.x, li * f.y));
          }
        }
      }
      tmem_st32(tb + loff + T_R1 + 64 + 32 * g, pk);
    }
    tc_fence_before();
    __syncthreads();   // [dO; dX] and U' have been read: the next head's load into their space
    tc_fence_after();
    if (tid == kIssuer) {
      if (hi + 1 < grp) issue_loads_a(sm, ws, &tmO, bar_a, ch + 1, h + 1, t0);
      // R4's part over [S0 | dS], beside F and E: [scale gamma dO | 0 ; -gamma beta dX |
      // lambda U'] [S0 | dS]^T
      const uint32_t i4 = idesc_bf16(128, 128, false, false);
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        const uint32_t ko = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16_ta(tb + T_R4, tb + T_R1 + 8 * ks, kdesc(sb + OFF_S0 + ko), i4, ks > 0 || hi > 0);
      }
    }
    if (hi + 1 < grp) last_a = hi + 1;
    GDN_GSTAMP(hi, 8);
    // ---- F (rows i < 64 of R2 / R3) and E (rows 64-127), warps 0-7 at once: a warp reaches
    //      the TMEM lanes 32 (warp % 4) .. + 31 and takes the column half warp / 4
    if (warp < 8) {
      const int part = warp >> 2;
      float x[32], y[32], v[32];
      tmem_ld32(tb + loff + T_R2 + 32 * part, x);   // dO U'^T or dX U'^T
      tmem_ld32(tb + loff + T_R3 + 32 * part, y);   // Q K^T or K K^T
      float racc = 0.f, db = 0.f;
      float fe[32];
      if (row < 64) {   // F = scale (dO U'^T) * Gamma on and below the diagonal
        const int i = row;
        const float gi = g2[i];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * part + jj;
          const float e = a.scale * x[jj] * ex2g(gi - g2[j]);
          fe[jj] = j <= i ? e : 0.f;
          v[jj] = fe[jj] * y[jj];
          racc += v[jj];
        }
      } else {          // dA = -(dX U'^T) strictly below, E = beta dA * Gamma
        const int i = row - 64;
        const float gi = g2[i];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * part + jj;
          const float e2 = ex2g(gi - g2[j]);
          const float gij = j < i ? e2 : 0.f;
          const float dA = -x[jj];
          fe[jj] = bt[i] * gij * dA;
          v[jj] = fe[jj] * y[jj];
          racc += v[jj];
          db = fmaf(dA * gij, y[jj], db);
        }
        dbp[part * 64 + i] = db;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {   // the F / E row as bf16, 8 columns per 16-byte store
        uint4 u;
        u.x = pack2(fe[8 * m], fe[8 * m + 1]);
        u.y = pack2(fe[8 * m + 2], fe[8 * m + 3]);
        u.z = pack2(fe[8 * m + 4], fe[8 * m + 5]);
        u.w = pack2(fe[8 * m + 6], fe[8 * m + 7]);
        *reinterpret_cast<uint4*>(sm + OFF_FE + sw128_offset(row, 32 * part + 8 * m)) = u;
      }
      rowp[part * 128 + row] = racc;
      // column sums over this warp's 32 rows: a transpose-reduce across the lanes (31 shuffles);
      // lane l ends with the sum of column 32 part + l
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < o; ++k) {
          const float send = up ? v[k] : v[k + o];
          const float keep = up ? v[k + o] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      colp[(warp & 3) * 64 + 32 * part + lane] = v[0];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    GDN_GSTAMP(hi, 9);
    // ---- the rest of R4 += [dQ; dK] of this value head (the issuer), and beside it (warps 2-3) dG,
    //      dbeta per token, then dg by a suffix sum
    if (tid == kIssuer) {
      const uint32_t i4c = idesc_bf16(128, 128, false, true), i4d = idesc_bf16(128, 128, true, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        // [F; E] K
        mma_bf16(tb + T_R4, kdesc(sb + OFF_FE + ks * 32), mndesc(sb + OFF_QK + 8192 + ks * 2048, 16384), i4c, 1);
        // [0; F^T] Q
        mma_bf16(tb + T_R4, mndesc(sb + OFF_ZERO + ks * 2048, OFF_FE - OFF_ZERO),
                 mndesc(sb + OFF_QK + ks * 2048, 16384), i4d, 1);
        // [0; E^T] K
        mma_bf16(tb + T_R4, mndesc(sb + OFF_ZERO + ks * 2048, OFF_FE + 8192 - OFF_ZERO),
                 mndesc(sb + OFF_QK + 8192 + ks * 2048, 16384), i4d, 1);
      }
      mma_commit(bar);
    } else if (warp == 2 || warp == 3) {
      const int i = tid - 64;
      // per-token sums in a fixed order
      const float rzi = (rowp[i] + rowp[64 + i]) + (rowp[128 + i] + rowp[192 + i]);
      const float dbai = dbp[i] + dbp[64 + i];
      const float csi = (colp[i] + colp[64 + i]) + (colp[128 + i] + colp[192 + i]);
      const float omega = i < L ? lm[i] * kh3[i] : 0.f;
      om[i] = omega;
      dGv[i] = i < L ? a.scale * gm[i] * qh1[i] - bt[i] * gm[i] * kh2[i] - omega + rzi - csi : 0.f;
      if (i < L) b.dbeta[(size_t)(t0 + i) * Hv + h] = xvr[i] - gm[i] * kh2[i] + dbai;
      group_sync(1, 64);   // warps 2-3: every token's dG is in place
    }
    if (warp == 2) {
      float sdt = 0.f;
      for (int w = 0; w < kWorkThreads / 32; ++w) sdt += red[w];
      const float omsum = warp_sum(om[lane] + om[lane + 32]);
      float x0 = dGv[lane], x1 = dGv[lane + 32];
      const float extra = gm[L - 1] * sdt + omsum;
      if (lane == L - 1) x0 += extra;
      if (lane + 32 == L - 1) x1 += extra;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_down_sync(0xffffffffu, x0, o);
        const float y1 = __shfl_down_sync(0xffffffffu, x1, o);
        if (lane + o < 32) { x0 += y0; x1 += y1; }
      }
      x0 += __shfl_sync(0xffffffffu, x1, 0);
      const size_t base = (size_t)t0 * Hv + h;
      if (lane < L) b.dg[base + (size_t)lane * Hv] = x0;
      if (lane + 32 < L) b.dg[base + (size_t)(lane + 32) * Hv] = x1;
    }
    GDN_GSTAMP(hi, 10);
    if (tid == kIssuer) ok = mbar_wait(bar, 1, kWaitNs);
    // (the barrier also orders the per-token vectors' last reads before the next head's writes)
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    GDN_GSTAMP(hi, 11);
    // S0, dS have been read: the next head's load into their space meanwhile
    if (hi + 1 < grp) {
      if (tid == kIssuer) issue_loads_b(sm, ws, bar_b, ch + 1);
      last_b = hi + 1;
    }
    GDN_GSTAMP(hi, 12);
  }
  if (failed) {
    if (tid == kIssuer) {   // copies still in flight land before the shared memory is released
      mbar_wait(bar_a, (uint32_t)last_a & 1u, kWaitNs);
      mbar_wait(bar_b, (uint32_t)last_b & 1u, kWaitNs);
      mbar_wait(bar_qk, 0, kWaitNs);
      report(a.dev_status, GDN_DEV_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTmemWarp) {
      tc_fence_after();
      tmem_dealloc(tb, T_COLS);
    }
    return;
  }
  GDN_GSTAMP(0, 13);
  // ---- dq, dk: the L2 norm's Jacobian on the group sums in R4 (rows 0-63: q, 64-127: k),
  //      dx = r (dx^ - x^ (x^ . dx^)) with x^ the normalised row in [q; k]; warp group g takes
  //      the columns 64 g .. 64 g + 63 (the k-half g of [q; k]) and the halves' partial dots
  //      meet in shared memory.  The bf16 rows are staged (128-byte-swizzled [64 tokens][64
  //      features] halves: dq at OFF_S0, dk at OFF_S0 + 16 KB) for TMA stores.
  const bool epi = warp < 8;   // (the issuer warp has no TMEM lanes here)
  const int g = warp >> 2, i = row & 63;
  float* pd = colp;   // [2][128]
  float d0[32], d1[32];   // the row's 64 columns of R4
  float xh[64];
  if (epi) {
    const uint8_t* xrow = sm + OFF_QK + g * 16384 + row * 128;
    tmem_ld32(tb + loff + T_R4 + 64 * g, d0);
    tmem_ld32(tb + loff + T_R4 + 64 * g + 32, d1);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {   // the row's 16-byte chunk c8 sits at c8 ^ (row % 8)
      const uint4 u = *reinterpret_cast<const uint4*>(xrow + ((c8 ^ (row & 7)) << 4));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
        xh[8 * c8 + 2 * q] = f.x;
        xh[8 * c8 + 2 * q + 1] = f.y;
      }
    }
    float p = 0.f;
#pragma unroll
    for (int e = 0; e < 64; ++e) p = fmaf(xh[e], e < 32 ? d0[e] : d1[e - 32], p);
    pd[g * 128 + row] = p;
  }
  __syncthreads();
  if (epi) {
    const float r = rnv[row];
    const float xd = pd[row] + pd[128 + row];
    uint8_t* srow = sm + OFF_S0 + (row >> 6) * 16384 + g * 8192 + i * 128;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = 8 * c8 + e;
        const float dk = k < 32 ? d0[k] : d1[k - 32];
        o[e] = l2 ? r * fmaf(-xd, xh[k], dk) : dk;
      }
      uint4 u;
      u.x = pack2(o[0], o[1]);
      u.y = pack2(o[2], o[3]);
      u.z = pack2(o[4], o[5]);
      u.w = pack2(o[6], o[7]);
      *reinterpret_cast<uint4*>(srow + ((c8 ^ (i & 7)) << 4)) = u;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (warp == kTmemWarp) {
    tc_fence_after();
    tmem_dealloc(tb, T_COLS);
  }
  GDN_GSTAMP(0, 14);
  if (L == C) {   // four TMA stores
    if (tid == kTmaThread) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        tma_store_3d(&tmDQ, sm + OFF_S0 + hh * 8192, 64 * hh, hq, t0);
        tma_store_3d(&tmDK, sm + OFF_S0 + 16384 + hh * 8192, 64 * hh, hq, t0);
      }
      tma_store_commit();
      tma_store_wait_read();   // the staged rows have left shared memory
    }
  } else {   // a chunk ending early: rows i < L only (the next ones are another sequence's)
    for (int e = tid; e < 2 * 64 * 16; e += kThreads) {
      const int hf = e >> 10, i = (e >> 4) & 63, hh = (e >> 3) & 1, c8 = e & 7;
      if (i < L)
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(hf ? b.dk : b.dq) +
                                  (((size_t)(t0 + i) * Hqk + hq) * 128 + 64 * hh + 8 * c8) * 2) =
            *reinterpret_cast<const uint4*>(sm + OFF_S0 + hf * 16384 + hh * 8192 + i * 128 + ((c8 ^ (i & 7)) << 4));
    }
  }
}
}  // namespace tcg

// ---------------------------------------------------------------- 4b. reverse on the tensor cores
// bf16 I/O with K = V = 128: one CTA (8 warps) per (sequence, value head), chunks last to
// first, with dS^T (TMEM lane = value index v, column = key index d) resident in TMEM like the
// forward's state.  Per chunk (tiles double-buffered one chunk ahead: q, k, v, dO by TMA; the
// prep pass's T and P tiles and per-token vectors by bulk copy):
//   Y^T   = dS^T K^T                        M=128 N=64  K=128  (A: bf16 dS^T from TMEM; raw k)
//   dUp^T = dO^T P                          M=128 N=64  K=64   (P carries scale)
//   dU'^T = dUp^T + Y^T diag(lambda r_k)    -> bf16 into TMEM
//   dX^T  = dU'^T T                         M=128 N=64  K=64
//   dS^T <- gamma_L dS^T + dO^T (scale diag(gamma r_q) Q) + (dX^T diag(-gamma beta r_k)) K
//                                           M=128 N=128 K=64 + 64
// The l2-norm reciprocals r_q, r_k and the gates enter as per-token fp32 factors: the k rows
// stay raw, the q rows are scaled in shared memory while the first products run, and
// -gamma beta r_k is folded into the bf16 dX^T operand.  It writes, per chunk, the bf16 dS (the
// gradient of the chunk's exit state) and dX tiles of the grad pass (staged in shared memory,
// bulk copies), dv = diag(beta) dX (staged over the v tile, TMA store) and the row dots
// dX_i . v_i (slot 0 of ws.XV).
namespace tcr {
using namespace sm100;
constexpr int kThreads = 256;    // two warps per TMEM lane quarter
constexpr int kStorer = 32;      // the thread that issues (and waits for) the bulk stores
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t ST_Q = 0, ST_K = 16384, ST_V = 32768, ST_DO = 49152, ST_T = 65536, ST_P = 73728;
constexpr uint32_t ST_VEC = 81920;                        // the prep pass's per-token vectors
constexpr uint32_t VEC_BYTES = kRvFloats * 4;
constexpr uint32_t STAGE = (ST_VEC + VEC_BYTES + 1023) / 1024 * 1024;
constexpr uint32_t STAGE_TX = 4 * 16384 + 16384 + VEC_BYTES;
constexpr uint32_t OFF_RED = 2 * STAGE;              // [4 lane quarters][64]
constexpr uint32_t OFF_BAR = OFF_RED + 4 * 64 * 4;
constexpr uint32_t OFF_STG_S = (OFF_BAR + 64 + 1023) / 1024 * 1024;   // staging: the dS tile (32 KB)
constexpr uint32_t OFF_STG_X = OFF_STG_S + 32768;                     // and the dX tile (16 KB)
constexpr uint32_t SMEM = OFF_STG_X + 16384 + 1024;
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(ST_P == ST_T + 8192, "T and P arrive by one bulk copy");
constexpr uint32_t C_S = 0, C_SB = 128, C_Y = 192, C_U = 256, C_X = 320, T_COLS = 512;

// Shared-memory offset, within a 128-byte-swizzled tile of 64-element halves `half` bytes
// apart, of the 8 x 8 block that lane `lane` of warp quarter wq addresses for stmatrix /
// ldmatrix .trans in column group 0: matrix i = lane / 8 covers elements 32 wq + 8 i .. + 7 of
// rows r = lane % 8 (add 1024 per further group of 8 rows).
__device__ __forceinline__ uint32_t frag_off(int wq, int lane, uint32_t half) {
  const int mblk = lane >> 3, rr = lane & 7;
  const int d0 = 32 * wq + 8 * mblk;
  return (d0 >> 6) * half + rr * 128 + ((((d0 & 63) >> 3) ^ rr) << 4);
}

// dS^T (fp32, C_S; lane = v, column = d) as the bf16 rows d of the grad pass's dS tile (two
// 16 KB halves), then scaled in TMEM by gamma_L.  Passes 2 p, 2 p + 1 of 32 columns (p = warp
// group).  16x256b loads hand each thread the fragment of stmatrix .trans (columns j, 2 (t%4)
// and + 1 of each 8-column group; v = t / 4 and t / 4 + 8 of each 16-lane half), which writes
// the 8 x 8 blocks transposed.
__device__ __forceinline__ void stage_state(uint32_t tb, uint32_t loff, int p, uint32_t tile,
                                            float gl, int wq, int lane) {
  const uint32_t st_base = tile + frag_off(wq, lane, 16384);
#pragma unroll 1
  for (int pass = 2 * p; pass < 2 * p + 2; ++pass) {
    uint32_t a0[16], a1[16];
    tmem_ld16x256b_x4(tb + loff + C_S + 32 * pass, a0);                 // v 0-15 of the warp
    tmem_ld16x256b_x4(tb + loff + (16u << 16) + C_S + 32 * pass, a1);   // v 16-31
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // column group 4 pass + j
      uint32_t f[4];
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const uint32_t* x = (mm >> 1) ? a1 : a0;
        const int k = 4 * j + 2 * (mm & 1);
        f[mm] = tcg::pack2(__uint_as_float(x[k]), __uint_as_float(x[k + 1]));
      }
      stmatrix_x4_trans(st_base + (4 * pass + j) * 1024, f);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      a0[e] = __float_as_uint(gl * __uint_as_float(a0[e]));
      a1[e] = __float_as_uint(gl * __uint_as_float(a1[e]));
    }
    tmem_st16x256b_x4(tb + loff + C_S + 32 * pass, a0);
    tmem_st16x256b_x4(tb + loff + (16u << 16) + C_S + 32 * pass, a1);
  }
  tmem_wait_st();
}

// dX^T (fp32, C_X; column = token) for tokens 32 p .. 32 p + 31 (p = warp group): the bf16 dX
// rows of the grad pass's tile at `xtile`, dv = beta_i dX_i written over the v rows at `vtile`
// (the same fragment positions, read first), and the row dots dX_i . v_i over this warp's 32 v
// into red[wq][i].
__device__ __forceinline__ void stage_dx(uint32_t tb, uint32_t loff, int p, uint32_t xtile,
                                         uint32_t vtile, const float* beta, float* red, int wq,
                                         int lane) {
  const uint32_t off = frag_off(wq, lane, 8192);
  uint32_t a0[16], a1[16];
  tmem_ld16x256b_x4(tb + loff + C_X + 32 * p, a0);
  tmem_ld16x256b_x4(tb + loff + (16u << 16) + C_X + 32 * p, a1);
  tmem_wait_ld();
  const int tq = 2 * (lane & 3);
  float dot[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {   // column group 4 p + j: this thread's tokens i0, i0 + 1
    const int i0 = 32 * p + 8 * j + tq;
    const float b0 = beta[i0], b1 = beta[i0 + 1];
    const uint32_t blk = (4 * p + j) * 1024 + off;
    uint32_t vv[4], fx[4], fv[4];
    ldmatrix_x4_trans(vtile + blk, vv);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const uint32_t* x = (mm >> 1) ? a1 : a0;
      const int k = 4 * j + 2 * (mm & 1);
      const float x0 = __uint_as_float(x[k]), x1 = __uint_as_float(x[k + 1]);
      const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv[mm]));
      fx[mm] = tcg::pack2(x0, x1);
      fv[mm] = tcg::pack2(b0 * x0, b1 * x1);
      s0 = fmaf(x0, vf.x, s0);
      s1 = fmaf(x1, vf.y, s1);
    }
    stmatrix_x4_trans(xtile + blk, fx);
    stmatrix_x4_trans(vtile + blk, fv);
    dot[2 * j] = s0;
    dot[2 * j + 1] = s1;
  }
  // sum over the 8 lanes of equal lane % 4 (the warp's 32 v), as a transpose: lane l ends
  // with the total of dot[l / 4]
#pragma unroll
  for (int o = 16, n = 4; o >= 4; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float send = up ? dot[k] : dot[k + n];
      const float keep = up ? dot[k + n] : dot[k];
      dot[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  const int idx = lane >> 2;
  red[wq * 64 + 32 * p + 8 * (idx >> 1) + tq + (idx & 1)] = dot[0];
}

__device__ __forceinline__ void issue_stage(uint8_t* st, uint64_t* bar, const CUtensorMap* tq,
                                            const CUtensorMap* tk, const CUtensorMap* tv,
                                            const CUtensorMap* to, const uint8_t* tp,
                                            const float* rv, int t, int hq, int h) {
  mbar_arrive_expect_tx(bar, STAGE_TX);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    tma_load_3d(st + ST_Q + hh * 8192, tq, bar, 64 * hh, hq, t);
    tma_load_3d(st + ST_K + hh * 8192, tk, bar, 64 * hh, hq, t);
    tma_load_3d(st + ST_V + hh * 8192, tv, bar, 64 * hh, h, t);
    tma_load_3d(st + ST_DO + hh * 8192, to, bar, 64 * hh, h, t);
  }
  bulk_load(st + ST_T, tp, 16384, bar);
  bulk_load(st + ST_VEC, rv, VEC_BYTES, bar);
}

// dS^T (fp32, C_S) -> bf16 pairs in C_SB, the A operand of the next Y product: columns
// 64 p2 .. 64 p2 + 63 for warp group p2.
__device__ __forceinline__ void pack_state(uint32_t tb, uint32_t loff, int p2) {
  {
    float x[32], y[32], pk[32];
    tmem_ld32(tb + loff + C_S + 64 * p2, x);
    tmem_ld32(tb + loff + C_S + 64 * p2 + 32, y);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      pk[j] = __uint_as_float(tcg::pack2(x[2 * j], x[2 * j + 1]));
      pk[16 + j] = __uint_as_float(tcg::pack2(y[2 * j], y[2 * j + 1]));
    }
    tmem_st32(tb + loff + C_SB + 32 * p2, pk);
  }
}

__global__ void __launch_bounds__(kThreads, 1) bwd_reverse_tc_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
    const __grid_constant__ CUtensorMap tmDV, const ChunkArgs a, const BwdArgs b, BwdWs ws) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  float* red = reinterpret_cast<float*>(sm + OFF_RED);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BAR);   // [2]
  uint64_t* mmab = full + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 24);
  const int Hv = a.Hv, h = blockIdx.x % Hv, n = blockIdx.x / Hv, hq = h / (Hv / a.Hqk);
  // warp group wg = warp / 4 takes half of the columns of every TMEM pass; wq = warp % 4 is the
  // lane quarter (the value indices v) the warp may access
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, wg = warp >> 2;
  const int v = 32 * wq + lane;
  const size_t st_off = ((size_t)n * Hv + h) * 128 * 128;
  if (!ws.chunk_off[a.num_seqs + 1]) {   // invalid cu_seqlens: zero gradient
    if (b.d_initial)
      for (int d = wg; d < 128; d += 2) b.d_initial[st_off + (size_t)d * 128 + v] = 0.f;
    return;
  }
  int bos, eos;
  seq_bounds(a, n, &bos, &eos);
  const int first = ws.chunk_off[n];
  const int nch = (eos - bos + C - 1) / C;
  const uint32_t loff = (uint32_t)(32 * wq) << 16;
  // the tiles of iteration it (chunk nch - 1 - it) into stage it % 2
  auto issue = [&](int it) {
    const int qc = nch - 1 - it;
    const size_t ch = (size_t)(first + qc) * Hv + h;
    issue_stage(sm + (it & 1) * STAGE, &full[it & 1], &tmQ, &tmK, &tmV, &tmO,
                reinterpret_cast<const uint8_t*>(ws.T + ch * 64 * 64), ws.G + ch * kRvFloats,
                bos + qc * C, hq, h);
  };
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(mmab, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
    tma_prefetch_desc(&tmDV);
    for (int it = 0; it < 2 && it < nch; ++it) issue(it);
  }
  int issued = nch < 2 ? nch : 2;   // iterations whose tiles were requested (uniform)
  if (warp == 0) {
    tmem_alloc(tslot, T_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;
  {  // dS^T <- d_final^T (warp group wg: columns 64 wg .. 64 wg + 63)
#pragma unroll
    for (int part = 2 * wg; part < 2 * wg + 2; ++part) {
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        x[j] = b.d_final ? b.d_final[st_off + (size_t)(32 * part + j) * 128 + v] : 0.f;
      tmem_st32(tb + loff + C_S + 32 * part, x);
    }
    pack_state(tb, loff, wg);
  }
  uint32_t ph = 0;
  bool failed = false;
  int it = 0;
  for (; it < nch; ++it) {
    const int qc = nch - 1 - it, s = it & 1;
    const int t0 = bos + qc * C, L = min(C, eos - t0);
    const size_t ch = (size_t)(first + qc) * Hv + h;
    uint8_t* st = sm + s * STAGE;
    const uint32_t sst = sb + s * STAGE;
    const float* vec = reinterpret_cast<const float*>(st + ST_VEC);
    bool ok = true;
    GDN_RSTAMP(0);
    if (tid == 0) ok = mbar_wait(&full[s], (uint32_t)(it >> 1) & 1u, kWaitNs);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    GDN_RSTAMP(1);
    if (L < C) {   // the sequence's last chunk: rows past its end (the next sequence's) cleared
      for (int e = tid; e < 2 * 64 * 8; e += kThreads) {
        const int hh = e >> 9, i = (e >> 3) & 63, c8 = e & 7;
        if (i >= L) {
          const uint32_t o = hh * 8192 + i * 128 + 16 * c8;
          *reinterpret_cast<uint4*>(st + ST_Q + o) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(st + ST_K + o) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(st + ST_DO + o) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
    }
    tc_fence_after();
    GDN_RSTAMP(2);
    if (tid == 0) {   // Y^T = dS^T K^T;  dUp^T = dO^T P
      const uint32_t iy = idesc_bf16(128, 64, false, false), iu = idesc_bf16(128, 64, true, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16_ta(tb + C_Y, tb + C_SB + 8 * ks,
                    tcg::kdesc(sst + ST_K + (ks >> 2) * 8192 + (ks & 3) * 32), iy, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tb + C_U, tcg::mndesc(sst + ST_DO + ks * 2048, 8192),
                 tcg::mndesc(sst + ST_P + ks * 2048, 8192), iu, ks > 0);
      mma_commit(mmab);
    } else {
      // while the products run: the next iteration's tiles into the other stage (its last
      // reads, and the dv store out of it, finished before the previous iteration ended) and
      // the q rows scaled by scale gamma_i r_q,i for the dS update
      if (tid == kThreads - 32 && it >= 1 && it + 1 < nch) issue(it + 1);
      if (warp > 0) {
        for (int e = tid - 32; e < 64 * 16; e += kThreads - 32) {
          const int i = e >> 4, hh = (e >> 3) & 1, c8 = e & 7;
          tcg::scale8(st + ST_Q + hh * 8192 + i * 128 + 16 * c8, vec[kRvCq + i]);
        }
        fence_proxy_async_smem();
      }
    }
    GDN_RSTAMP(3);
    if (it >= 1 && it + 1 < nch) issued = it + 2;
    if (tid == 0) ok = mbar_wait(mmab, ph, kWaitNs);
    ph ^= 1u;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    GDN_RSTAMP(4);
    {  // dU'^T = dUp^T + Y^T diag(lambda r_k) -> bf16 pairs in C_U
      const float* w = vec + kRvW;
      float pk[16];
      {
        const int p = wg;   // tokens 32 p .. 32 p + 31
        float y[32], u[32];
        tmem_ld32(tb + loff + C_Y + 32 * p, y);
        tmem_ld32(tb + loff + C_U + 32 * p, u);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j0 = 32 * p + 2 * jj;
          pk[jj] = __uint_as_float(tcg::pack2(fmaf(w[j0], y[2 * jj], u[2 * jj]),
                                              fmaf(w[j0 + 1], y[2 * jj + 1], u[2 * jj + 1])));
        }
      }
      tc_fence_before();
      __syncthreads();   // both groups have read their fp32 columns
      tc_fence_after();
      tcg::tmem_st16(tb + loff + C_U + 16 * wg, pk);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    GDN_RSTAMP(5);
    if (tid == 0) {   // dX^T = dU'^T T (the stage holds T^T: a K-major B operand)
      const uint32_t ix = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ta(tb + C_X, tb + C_U + 8 * ks, tcg::kdesc(sst + ST_T + ks * 32), ix, ks > 0);
      mma_commit(mmab);
    }
    if (tid == 0) ok = mbar_wait(mmab, ph, kWaitNs);
    if (tid == kStorer) tma_store_wait_read();   // the previous tiles have left the staging buffers
    ph ^= 1u;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    // the grad pass's bf16 tiles, staged for bulk copies: dX (rows = the chunk's tokens, 64 v
    // per 128-byte row in two 8 KB halves) and dS, the gradient of the chunk's exit state (rows d,
    // two 16 KB halves), both 128-byte swizzled; dv over the v tile; dS^T <- gamma_L dS^T
    GDN_RSTAMP(6);
    stage_dx(tb, loff, wg, sb + OFF_STG_X, sst + ST_V, vec + kRvBeta, red, wq, lane);
    GDN_RSTAMP(7);
    stage_state(tb, loff, wg, sb + OFF_STG_S, vec[kRvGl], wq, lane);
    fence_proxy_async_smem();
    GDN_RSTAMP(8);
    {  // bf16 dX^T diag(-gamma beta r_k) in C_X, the A operand of the dS update
      const float* fv = vec + kRvF;
      float pk[16];
      {
        const int p = wg;
        float x[32];
        tmem_ld32(tb + loff + C_X + 32 * p, x);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int i = 32 * p + 2 * jj;
          pk[jj] = __uint_as_float(tcg::pack2(x[2 * jj] * fv[i], x[2 * jj + 1] * fv[i + 1]));
        }
      }
      tc_fence_before();
      __syncthreads();   // both groups have read their fp32 columns
      tc_fence_after();
      tcg::tmem_st16(tb + loff + C_X + 16 * wg, pk);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    GDN_RSTAMP(9);
    if (tid == kStorer) {   // beside the dS update: dv first (its own group), then dS and dX
      if (L == C) {   // dv rows by TMA (a chunk ending earlier must not touch the next sequence)
        tma_store_3d(&tmDV, st + ST_V, 0, h, t0);
        tma_store_3d(&tmDV, st + ST_V + 8192, 64, h, t0);
      }
      tma_store_commit();
      uint8_t* gs = reinterpret_cast<uint8_t*>(ws.dS + ch * ws.sdS);
      bulk_store(gs, sm + OFF_STG_S, 16384);
      bulk_store(gs + 16384, sm + OFF_STG_S + 16384, 16384);
      bulk_store(ws.dX + ch * ws.sdX, sm + OFF_STG_X, 16384);
      tma_store_commit();
    }
    if (L < C) {   // dv rows i < L of the sequence's last chunk, 16 bytes a store
      for (int e = tid; e < 64 * 16; e += kThreads) {
        const int i = e >> 4, hh = (e >> 3) & 1, c8 = e & 7;
        if (i < L)
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(b.dv) +
                                    (((size_t)(t0 + i) * Hv + h) * 128 + 64 * hh + 8 * c8) * 2) =
              *reinterpret_cast<const uint4*>(st + ST_V + hh * 8192 + i * 128 + ((c8 ^ (i & 7)) << 4));
      }
    }
    if (tid >= 64 && tid < 128) {   // the row dots, summed over the lane quarters in a fixed order
      const int i = tid - 64;
      ws.XV[ch * 4 * 64 + i] = (red[i] + red[64 + i]) + (red[128 + i] + red[192 + i]);
    }
    GDN_RSTAMP(10);
    if (tid == 0) {   // dS^T += dO^T (scale gamma r_q q) + (dX^T diag(-gamma beta r_k)) k
      const uint32_t iq = idesc_bf16(128, 128, true, true), ik = idesc_bf16(128, 128, false, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tb + C_S, tcg::mndesc(sst + ST_DO + ks * 2048, 8192),
                 tcg::mndesc(sst + ST_Q + ks * 2048, 8192), iq, 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ta(tb + C_S, tb + C_X + 8 * ks, tcg::mndesc(sst + ST_K + ks * 2048, 8192), ik, 1);
      mma_commit(mmab);
    }
    if (tid == 0) ok = mbar_wait(mmab, ph, kWaitNs);
    // the dv rows have left the stage, which the next iteration refills (the staged dS and dX
    // tiles may still be in flight: they are waited for before the next staging)
    if (tid == kStorer) tma_store_wait_read_allbut1();
    ph ^= 1u;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    GDN_RSTAMP(11);
    pack_state(tb, loff, wg);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    GDN_RSTAMP(12);
  }
  if (tid == kStorer) tma_store_wait_all();   // the stored tiles are written before the CTA exits
  if (tid == 0) {
    if (failed) {   // tiles still in flight land before the shared memory is released
      for (int k = it; k < issued; ++k) mbar_wait(&full[k & 1], (uint32_t)(k >> 1) & 1u, kWaitNs);
      report(a.dev_status, GDN_DEV_TIMEOUT);
    }
  }
  if (!failed && b.d_initial) {
#pragma unroll
    for (int part = 2 * wg; part < 2 * wg + 2; ++part) {
      float x[32];
      tmem_ld32(tb + loff + C_S + 32 * part, x);
#pragma unroll
      for (int j = 0; j < 32; ++j) b.d_initial[st_off + (size_t)(32 * part + j) * 128 + v] = x[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, T_COLS);
  }
}
}  // namespace tcr

// ---------------------------------------------------------------- 6. qk
// One warp per (token, query/key head), four features per lane: the group sum of the
// per-value-head dQ, dK in a fixed order, then the L2 norm's Jacobian.  Tokens outside every
// sequence get zero gradients (dq, dk here; dv, dg, dbeta of the group's value heads too).
constexpr int kQkThreads = 256;

__global__ void __launch_bounds__(kQkThreads) bwd_qk_kernel(const ChunkArgs a, const BwdArgs b,
                                                            BwdWs ws, int T_total) {
  const long long item = (long long)blockIdx.x * (kQkThreads / 32) + (threadIdx.x >> 5);
  if (item >= (long long)T_total * a.Hqk) return;
  const int lane = threadIdx.x & 31;
  const int t = (int)(item / a.Hqk), hq = (int)(item - (long long)t * a.Hqk);
  const int N = a.num_seqs, K = a.K, V = a.V, grp = a.Hv / a.Hqk;
  int covered = 0;
  if (ws.chunk_off[N + 1]) covered = a.cu_seqlens ? a.cu_seqlens[N] : N * a.T;
  const bool in = t < covered;
  const bool l2 = a.use_qk_l2norm != 0;
  const int d = 4 * lane;
  const bool act = d < K;   // K % 4 == 0
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const void* x_src = which ? a.k : a.q;
    const float* dsrc = which ? ws.dK : ws.dQ;
    float dx[4] = {0.f, 0.f, 0.f, 0.f}, x[4] = {0.f, 0.f, 0.f, 0.f};
    if (in && act) {
      for (int hh = hq * grp; hh < (hq + 1) * grp; ++hh) {
        const float4 v = ld4(dsrc + ((size_t)t * a.Hv + hh) * K + d);
        dx[0] += v.x; dx[1] += v.y; dx[2] += v.z; dx[3] += v.w;
      }
      load4(x_src, ((size_t)t * a.Hqk + hq) * K + d, a.io_dtype, x);
    }
    if (l2) {
      float ss = 0.f, xd = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        ss = fmaf(x[m], x[m], ss);
        xd = fmaf(x[m], dx[m], xd);
      }
      ss = warp_sum(ss);
      xd = warp_sum(xd);
      const float rho = 1.0f / sqrtf(ss + kL2Eps);
      const float c3 = rho * rho * rho * xd;
#pragma unroll
      for (int m = 0; m < 4; ++m) dx[m] = rho * dx[m] - c3 * x[m];
    }
    if (act) store4(which ? b.dk : b.dq, ((size_t)t * a.Hqk + hq) * K + d, a.io_dtype, dx);
  }
  if (!in) {   // zero dv, dg, dbeta of this group's value heads
    const float z[4] = {0.f, 0.f, 0.f, 0.f};
    for (int hh = hq * grp; hh < (hq + 1) * grp; ++hh) {
      for (int e = 4 * lane; e < V; e += 128) store4(b.dv, ((size_t)t * a.Hv + hh) * V + e, a.io_dtype, z);
      if (lane == 0) {
        b.dg[(size_t)t * a.Hv + hh] = 0.f;
        b.dbeta[(size_t)t * a.Hv + hh] = 0.f;
      }
    }
  }
}

// Tokens outside every sequence (past cu_seqlens[N], or every token when cu_seqlens is
// invalid) get zero gradients: dq, dk and the group's dv, dg, dbeta.  The tensor-core path's
// passes write every token inside a sequence; this one clears the rest, one warp per (token,
// query/key head) in a grid-stride loop.
constexpr int kUncoveredBlocks = 256;
__global__ void __launch_bounds__(kQkThreads) bwd_uncovered_kernel(const ChunkArgs a, const BwdArgs b,
                                                                   BwdWs ws, int T_total) {
  const int N = a.num_seqs, K = a.K, V = a.V, grp = a.Hv / a.Hqk;
  int covered = 0;
  if (ws.chunk_off[N + 1]) covered = a.cu_seqlens ? a.cu_seqlens[N] : N * a.T;
  covered = min(max(covered, 0), T_total);
  const long long items = (long long)(T_total - covered) * a.Hqk;
  const long long step = (long long)gridDim.x * (kQkThreads / 32);
  const int lane = threadIdx.x & 31;
  const float z[4] = {0.f, 0.f, 0.f, 0.f};
  for (long long it = (long long)blockIdx.x * (kQkThreads / 32) + (threadIdx.x >> 5); it < items; it += step) {
    const int t = covered + (int)(it / a.Hqk), hq = (int)(it % a.Hqk);
    for (int e = 4 * lane; e < K; e += 128) {
      store4(b.dq, ((size_t)t * a.Hqk + hq) * K + e, a.io_dtype, z);
      store4(b.dk, ((size_t)t * a.Hqk + hq) * K + e, a.io_dtype, z);
    }
    for (int hh = hq * grp; hh < (hq + 1) * grp; ++hh) {
      for (int e = 4 * lane; e < V; e += 128) store4(b.dv, ((size_t)t * a.Hv + hh) * V + e, a.io_dtype, z);
      if (lane == 0) {
        b.dg[(size_t)t * a.Hv + hh] = 0.f;
        b.dbeta[(size_t)t * a.Hv + hh] = 0.f;
      }
    }
  }
}

}  // namespace

#ifdef GDN_CHUNK_STAMPS
// The stage timestamps of the last tensor-core backward of the stamped build: the reverse pass's
// [8 CTAs][iterations 32 .. 95][16] and the grad pass's [8 CTAs][2 heads][16] clock64 values;
// returns a cudaError_t.
extern "C" int gdn_bwd_stamps_read(void* rev, void* grad) {
  cudaError_t e = cudaMemcpyFromSymbol(rev, g_rev_stamps, sizeof(g_rev_stamps));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(grad, g_grad_stamps, sizeof(g_grad_stamps));
  return (int)e;
}
#endif

size_t chunk_bwd_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V, bool tc) {
  size_t total = 0;
  bwd_layout(nullptr, max_chunks(T_total, num_seqs), num_seqs, Hv, K, V, T_total, tc, &total);
  return total;
}

bool chunk_bwd_uses_tc(int K, int V, int io_dtype, int beta_dtype) {
  return chunk_tc_supported(K, V, io_dtype, beta_dtype);
}

cudaError_t launch_chunk_bwd(const ChunkArgs& a_in, const BwdArgs& b) {
  ChunkArgs a = a_in;
  a.final_state = nullptr;  // the forward state pass records entry states only
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  const long long NC = max_chunks(T_total, a.num_seqs);
  // bf16 with K = V = 128 (given gates): every product on the tensor cores
  const bool tc = chunk_bwd_uses_tc(a.K, a.V, a.io_dtype, a.beta_dtype) && a.gates.mode == kGatesGiven;
  BwdWs ws = bwd_layout(a.workspace, NC, a.num_seqs, a.Hv, a.K, a.V, T_total, tc, nullptr);
  cudaError_t err;
  if ((err = cudaFuncSetAttribute(bwd_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem))) return err;
  if ((err = cudaFuncSetAttribute(tcr::bwd_reverse_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcr::SMEM))) return err;
  if ((err = cudaFuncSetAttribute(bwd_reverse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRevSmem))) return err;
  if ((err = cudaFuncSetAttribute(bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmem))) return err;
  if ((err = cudaFuncSetAttribute(tcg::bwd_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcg::SMEM))) return err;
  chunk_table_kernel<<<1, 1024, 0, a.stream>>>(a, ws.chunk_off);
  if ((err = cudaGetLastError())) return err;
  // Forward recompute of the state entering every chunk and of U'.  bf16 with K = V = 128:
  // the tensor-core kernel in record mode (no output); otherwise the fp32 state pass on W, U
  // from the prep kernel.
  if (tc && T_total > 0) {
    ChunkArgs f = a;
    f.o = nullptr;
    f.rec_states = ws.S;
    f.rec_u = ws.U;
    f.rec_tp = ws.T;      // T^T and P for the reverse pass
    f.rec_vec = ws.G;     // and its per-token vectors
    f.rec_chunk_off = ws.chunk_off;
    if ((err = launch_chunk_tc(f))) return err;
  }
  if (!tc) {   // fp32 state pass on W, U of the fp32 path's own prep pass
    if ((err = launch_chunk_prep(a, ws.chunk_off, ws.W, ws.U, ws.G))) return err;
    if ((err = launch_chunk_states(a, ws.chunk_off, ws.W, ws.U, ws.G, ws.S))) return err;
  }
  if (tc && NC * a.Hv > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (tc && a.Hv % a.Hqk != 0) return cudaErrorInvalidValue;
  if (NC > 0 && !tc) {   // (the tensor-core path's record-mode forward wrote T, P and the vectors)
    bwd_prep_kernel<<<dim3((unsigned)NC, a.Hv), kPrepThreads, kPrepSmem, a.stream>>>(a, b, ws);
    if ((err = cudaGetLastError())) return err;
  }
  const unsigned vtiles = (unsigned)((a.V + VT - 1) / VT);
  if (a.num_seqs > 0) {
    const long long blocks = (long long)vtiles * a.Hv * a.num_seqs;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (tc) {
      CUtensorMap mq, mk, mv, mo, mdv;
      memset(&mq, 0, sizeof(mq));
      memset(&mk, 0, sizeof(mk));
      memset(&mv, 0, sizeof(mv));
      memset(&mo, 0, sizeof(mo));
      memset(&mdv, 0, sizeof(mdv));
      if (!encode_rows_map_bf16(&mq, a.q, a.Hqk, T_total) || !encode_rows_map_bf16(&mk, a.k, a.Hqk, T_total) ||
          !encode_rows_map_bf16(&mv, a.v, a.Hv, T_total) || !encode_rows_map_bf16(&mo, b.d_o, a.Hv, T_total) ||
          !encode_rows_map_bf16(&mdv, b.dv, a.Hv, T_total))
        return cudaErrorInvalidValue;
      const long long ctas = (long long)a.num_seqs * a.Hv;
      if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      tcr::bwd_reverse_tc_kernel<<<(unsigned)ctas, tcr::kThreads, tcr::SMEM, a.stream>>>(mq, mk, mv, mo, mdv, a, b, ws);
    } else {
      bwd_reverse_kernel<<<(unsigned)blocks, kRevThreads, kRevSmem, a.stream>>>(a, b, ws);
    }
    if ((err = cudaGetLastError())) return err;
  }
  if (NC > 0) {
    if (tc) {
      CUtensorMap gq, gk, go, gdq, gdk;
      memset(&gq, 0, sizeof(gq));
      memset(&gk, 0, sizeof(gk));
      memset(&go, 0, sizeof(go));
      memset(&gdq, 0, sizeof(gdq));
      memset(&gdk, 0, sizeof(gdk));
      if (!encode_rows_map_bf16(&gq, a.q, a.Hqk, T_total) || !encode_rows_map_bf16(&gk, a.k, a.Hqk, T_total) ||
          !encode_rows_map_bf16(&go, b.d_o, a.Hv, T_total) || !encode_rows_map_bf16(&gdq, b.dq, a.Hqk, T_total) ||
          !encode_rows_map_bf16(&gdk, b.dk, a.Hqk, T_total))
        return cudaErrorInvalidValue;
      // one CTA per (chunk, query/key head)
      tcg::bwd_grad_tc_kernel<<<(unsigned)(NC * a.Hqk), tcg::kThreads, tcg::SMEM, a.stream>>>(gq, gk, go, gdq, gdk, a, b, ws);
    } else {
      bwd_grad_kernel<<<dim3((unsigned)NC, a.Hv), kGradThreads, kGradSmem, a.stream>>>(a, b, ws);
    }
    if ((err = cudaGetLastError())) return err;
  }
  if (T_total > 0) {
    if (tc) {   // the grad pass wrote dq, dk of every token in a sequence; clear the rest
      bwd_uncovered_kernel<<<kUncoveredBlocks, kQkThreads, 0, a.stream>>>(a, b, ws, T_total);
    } else {
      const long long items = (long long)T_total * a.Hqk;
      const long long blocks = (items + kQkThreads / 32 - 1) / (kQkThreads / 32);
      if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      bwd_qk_kernel<<<(unsigned)blocks, kQkThreads, 0, a.stream>>>(a, b, ws, T_total);
    }
    if ((err = cudaGetLastError())) return err;
  }
  return cudaSuccess;
}

}  // namespace gdn
