// gdn_chunk_util.cuh -- device helpers shared by the fp32 chunk kernels (forward and
// backward): sequence bounds, the device-side chunk table built from cu_seqlens,
// chunk -> (sequence, first token, length) lookup, row loads with the optional
// q/k L2 norm, and the per-chunk gate values with their in-chunk cumulative sum.
#pragma once

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

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
      if (!bad) cnt = (eos - bos + kChunk - 1) / kChunk;
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
  *t0 = bos + (c - chunk_off[lo]) * kChunk;
  *L = min(kChunk, eos - *t0);
  return true;
}

// Load rows [t0, t0 + L) of a [T, H, D] tensor (head hd) into dst[kChunk][ld] fp32
// (ld >= D; the first D entries of each row), L2-normalised per row when asked;
// rows >= L are zero.  D <= 128; any whole number of warps, each taking its rows four at a
// time with every load of the four issued before the norms.  Needs a __syncthreads after
// return before the tile is read.
__device__ void load_rows(const void* src, int dtype, int t0, int L, int H, int hd, int D,
                          bool l2, float* dst, int ld) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int r0 = warp; r0 < kChunk; r0 += 4 * nw) {
    float x[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * nw;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = lane + 32 * m;
        x[u][m] = (r < kChunk && r < L && e < D)
                      ? load_elem(src, ((size_t)(t0 + r) * H + hd) * D + e, dtype) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * nw;
      if (r >= kChunk) break;   // uniform over the warp
      float rn = 1.f;
      if (l2 && r < L) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(x[u][m], x[u][m], ss);
        rn = 1.0f / sqrtf(warp_sum(ss) + kL2Eps);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = lane + 32 * m;
        if (e < D) dst[r * ld + e] = x[u][m] * rn;
      }
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
// (zero for rows >= L).  Done by one whole warp (lane = its lane index).
__device__ void load_gates(const ChunkArgs& a, int t0, int L, int h, float* G, float* bt,
                           int lane) {
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
// The same on warp 0 of the block (the other threads return at once).
__device__ void load_gates(const ChunkArgs& a, int t0, int L, int h, float* G, float* bt) {
  if (threadIdx.x < 32) load_gates(a, t0, L, h, G, bt, (int)threadIdx.x);
}

}  // namespace
}  // namespace gdn
