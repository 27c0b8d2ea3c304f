// gdn_tc_prep.cuh -- the state-independent half of a chunk on the tensor-core path (the prep
// group of the fused chunk kernel, gdn_chunk_tc.cu, in its forward and record modes).  For one
// chunk of one (sequence, value head), bf16 I/O, K = V = 128, chunk 64, with G = in-chunk
// cumulative log-decay and r_q / r_k the inverse L2 norms:
//
//   D1 = [Q; K] [Q; K]^T                      (tcgen05, M = N = K = 128; the diagonal gives
//                                              |q|^2 and |k|^2)
//   P  = scale r_q r_k^T * Q K^T * exp(G_i - G_j) * [j <= i]   (bf16, K-major [64 i][64 j])
//   A  = beta r_k r_k^T * K K^T * exp(G_i - G_j) * [j < i]     (fp32)
//   T  = (I + A)^{-1}, written as the bf16 MMA operands
//        Tw^T = (T diag(beta exp(G) r_k))^T and Tu^T = (T diag(beta))^T   (MN-major [64 j][64 i]):
//        the 16 x 16 diagonal-block inverses by substitution on the CUDA cores, the block
//        products that assemble T from them by warp-level tf32 mma.sync
//
// These are the chunkwise (WY / UT transform) equations of the gated delta rule at the fixed
// 64-token chunking of the inference kernels ("Megatron-Core API: core.ssm.gated_delta_product",
// ssm_inference_chunk_size) with the argument set of torch_chunk_gated_delta_rule ("Megatron-Core
// API: core.ssm.gated_delta_net.gdn").  Every function here is run by one 256-thread group
// (threads 0-255 of the CTA: eight warps, two per TMEM lane quarter) that synchronises on its
// own named barrier.
#pragma once

#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kPrepThreads = 256;
constexpr int kTcDK = 128, kTcDV = 128;

// TMA stage: [dk half][Q rows 0-63 | K rows 64-127][128 B] (32 KB) and V [dv half][64][128 B]
// (16 KB), both 128-byte swizzled.
constexpr uint32_t kQkStageBytes = 32768;
constexpr uint32_t kVStageBytes = 16384;
constexpr uint32_t kStageTx = kQkStageBytes + kVStageBytes;

// Per-token fp32 vectors of a chunk, 64 entries each (offsets in floats).
constexpr uint32_t VEC_G = 0,      // in-chunk cumulative log-decay, base 2
    VEC_BETA = 64,                 // beta (zero past the chunk end)
    VEC_RQ = 128, VEC_RK = 192,    // inverse L2 norms
    VEC_SW = 256,                  // beta exp(G) r_k: the column factor of Tw
    VEC_DL = 320,                  // exp(G_last - G) r_k: the row factor of K~
    VEC_QS = 384,                  // scale exp(G) r_q: the row factor of Q S
    VEC_H = 448,                   // G - log2 r_k: column factor of P and A as an exponent
    VEC_FLOATS = 512;

// Diagonal blocks of T, column-major: [4 blocks][16 columns][TD_LD (16 rows + pad)].
constexpr int TD_LD = 20;
constexpr uint32_t kTdBytes = 4 * 16 * TD_LD * 4;
constexpr uint64_t kPrepWaitNs = 2000000000ull;

// fp32 A tile: element (i, j) at i * 64 + 4 * ((j / 4) ^ (i % 16)) + j % 4, so that
// 16-byte groups stay contiguous and the row-parallel accesses of the solve hit
// distinct banks.
__device__ __forceinline__ int a_idx(int i, int j) {
  return i * 64 + ((((j >> 2) ^ (i & 15)) << 2) | (j & 3));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ void store_bf16x8(uint8_t* p, const float* v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// 2^x and log2(x) on the special-function unit (inputs here are <= 0 or moderate).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool flag_set(const int* f) {
  return *reinterpret_cast<const volatile int*>(f) != 0;
}
__device__ __forceinline__ void set_flag(int* f) { *reinterpret_cast<volatile int*>(f) = 1; }

// Issue the TMA loads of the chunk starting at token t into one stage (without V when
// load_v is false: the stage's V tile then keeps whatever it holds, zeros for a v = 0 run).
__device__ __forceinline__ void issue_chunk_loads(uint8_t* qk, uint8_t* vv, uint64_t* bar,
                                                  const CUtensorMap* tq, const CUtensorMap* tk,
                                                  const CUtensorMap* tv, int t, int hq, int h,
                                                  bool load_v = true) {
  mbar_arrive_expect_tx(bar, load_v ? kStageTx : kQkStageBytes);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    tma_load_3d(qk + hh * 16384, tq, bar, 64 * hh, hq, t);
    tma_load_3d(qk + hh * 16384 + 8192, tk, bar, 64 * hh, hq, t);
    if (load_v) tma_load_3d(vv + hh * 8192, tv, bar, 64 * hh, h, t);
  }
}

// D1 = [Q;K][Q;K]^T of the stage at shared address qk_a: the stage holds Q rows 0-63 and
// K rows 64-127, so one descriptor serves as A and as the N = 128 B.  Issued by one thread.
__device__ __forceinline__ void issue_d1(uint32_t d_tmem, uint32_t qk_a, uint64_t* bar) {
  const uint32_t id1 = idesc_bf16(128, 128, false, false);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint64_t d = sdesc_sw128(qk_a + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
    mma_bf16(d_tmem, d, d, id1, ks > 0);
  }
  mma_commit(bar);
}

// g and beta of tokens t0 + lane and t0 + lane + 32, clamped to a valid token:
// loaded one chunk ahead and masked (zero past the chunk end) where used, so the
// loads never stall the issuing warp.
__device__ __forceinline__ float ld_f32_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_bf16_early(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return __bfloat162float(__ushort_as_bfloat16(v));
}
// (volatile loads stay where they are issued: the compiler cannot sink them to
// their use one chunk later and expose the memory latency there)
__device__ __forceinline__ float ld_early(const void* base, size_t i, int dtype) {
  return dtype == GDN_BF16 ? ld_bf16_early(reinterpret_cast<const __nv_bfloat16*>(base) + i)
                           : ld_f32_early(reinterpret_cast<const float*>(base) + i);
}
// Raw gate inputs of tokens t0 + lane and t0 + lane + 32: g and beta, or, with
// fused gates, the features a and b (turned into g and beta where used).
__device__ __forceinline__ void prefetch_gates(const ChunkArgs& a, int t0, int h, int lane,
                                               int T_total, float* g, float* b) {
  const size_t ta = (size_t)min(t0 + lane, T_total - 1), tb = (size_t)min(t0 + lane + 32, T_total - 1);
  if (a.gates.mode == kGatesFused) {
    g[0] = ld_early(a.gates.a, ta * a.Hv + h, a.gates.ab_dtype);
    g[1] = ld_early(a.gates.a, tb * a.Hv + h, a.gates.ab_dtype);
    b[0] = ld_early(a.gates.b, ta * a.Hv + h, a.gates.ab_dtype);
    b[1] = ld_early(a.gates.b, tb * a.Hv + h, a.gates.ab_dtype);
  } else {
    g[0] = ld_f32_early(a.g + ta * a.Hv + h);
    g[1] = ld_f32_early(a.g + tb * a.Hv + h);
    b[0] = ld_early(a.beta, ta * a.Hv + h, a.beta_dtype);
    b[1] = ld_early(a.beta, tb * a.Hv + h, a.beta_dtype);
  }
}

// One warp: the chunk's in-chunk cumulative log-decay (base 2) and beta into vec from the
// prefetched raw values gq / bq (fused gates: g = -exp(A_log) softplus(a + dt_bias),
// beta = sigmoid(b)); then prefetches the next chunk's raw values.
__device__ __forceinline__ void gates_step(const ChunkArgs& a, float* vec, float* gq, float* bq,
                                           int L, int lane, bool fused, float expA, float dtb,
                                           bool prefetch_next, int t_next, int h, int T_total) {
  if (fused) {
    gq[0] = -expA * softplus_f(gq[0] + dtb);
    gq[1] = -expA * softplus_f(gq[1] + dtb);
    bq[0] = sigmoid_f(bq[0]);
    bq[1] = sigmoid_f(bq[1]);
  }
  float g0 = lane < L ? gq[0] : 0.f, g1 = lane + 32 < L ? gq[1] : 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float x0 = __shfl_up_sync(0xffffffffu, g0, o);
    const float x1 = __shfl_up_sync(0xffffffffu, g1, o);
    if (lane >= o) { g0 += x0; g1 += x1; }
  }
  g1 += __shfl_sync(0xffffffffu, g0, 31);
  vec[VEC_G + lane] = g0 * kLog2e;
  vec[VEC_G + lane + 32] = g1 * kLog2e;
  vec[VEC_BETA + lane] = lane < L ? bq[0] : 0.f;
  vec[VEC_BETA + lane + 32] = lane + 32 < L ? bq[1] : 0.f;
  if (prefetch_next) prefetch_gates(a, t_next, h, lane, T_total, gq, bq);
}

// After D1 of the chunk has landed in TMEM at d1 (and the gates are in vec): the inverse
// norms from its diagonal (lane i, column i: |q_i|^2 for i < 64, |k_{i-64}|^2 above) and the
// per-token scalars built from them, then P (bf16, K-major rows i, to p_dst; none when p_dst
// is null) and A (fp32, to sA).  The row and column factors enter as exponents: x * 2^(G_i + log2 f_i - H_j).
// Synchronises the group once in the middle; the caller syncs before P, A or vec are read.
template <int kBar>
__device__ __forceinline__ void norms_p_a(const ChunkArgs& a, uint32_t d1, float* vec, float* sA,
                                          uint8_t* p_dst, int L) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, chalf = warp >> 2;
  const int row = 32 * quad + lane;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  float x[32];
  tmem_ld32(d1 + lane_off + 64 + 32 * chalf, x);   // Q K^T | K K^T, for P and A
  if (chalf == 0) {
    float dg[32];
    tmem_ld32(d1 + lane_off + 32 * quad, dg);
    float d2 = dg[0];
#pragma unroll
    for (int jj = 1; jj < 32; ++jj) d2 = (lane == jj) ? dg[jj] : d2;
    const float r = a.use_qk_l2norm ? rsqrtf(d2 + kL2Eps) : 1.0f;
    const int i = row & 63;
    const float gi = vec[VEC_G + i];
    if (quad < 2) {
      vec[VEC_RQ + i] = r;
      vec[VEC_QS + i] = a.scale * ex2(gi) * r;
    } else {
      vec[VEC_RK + i] = r;
      vec[VEC_SW + i] = vec[VEC_BETA + i] * ex2(gi) * r;
      vec[VEC_DL + i] = ex2(vec[VEC_G + L - 1] - gi) * r;
      vec[VEC_H + i] = gi - lg2(r);   // column factor r_k[j] 2^-G_j as an exponent
    }
  }
  group_sync(kBar, kPrepThreads);

  const bool is_p = quad < 2;
  if (is_p && !p_dst) return;   // no P wanted
  const int j0 = 32 * chalf;
  float hj[32];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float4 h4 = *reinterpret_cast<const float4*>(vec + VEC_H + j0 + 4 * m);
    hj[4 * m] = h4.x; hj[4 * m + 1] = h4.y; hj[4 * m + 2] = h4.z; hj[4 * m + 3] = h4.w;
  }
  // one code path for both halves: P rows (quads 0-1) keep j <= i with the row factor scale r_q[i]
  // (zero past the chunk end: lg2(0) = -inf gives exact zeros), A rows (quads 2-3) keep j < i with
  // the row factor beta r_k[i]; both as exponents
  const int i = is_p ? row : row - 64;
  const float base = vec[VEC_G + i] + lg2(is_p ? ((i < L) ? a.scale * vec[VEC_RQ + i] : 0.f)
                                               : vec[VEC_BETA + i] * vec[VEC_RK + i]);
  const int lim = is_p ? i : i - 1;
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) {
    const float e = x[jj] * ex2(base - hj[jj]);
    x[jj] = (j0 + jj <= lim) ? e : 0.f;
  }
  if (is_p) {
#pragma unroll
    for (int m = 0; m < 4; ++m) store_bf16x8(p_dst + sw128_offset(i, j0 + 8 * m), &x[8 * m]);
  } else {
#pragma unroll
    for (int m = 0; m < 8; ++m)
      *reinterpret_cast<float4*>(&sA[a_idx(i, j0 + 4 * m)]) =
          make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
  }
}

// One 16 x 16 x 16 product on the tensor cores with warp-level tf32 mma.sync (two n tiles of
// eight, two k steps of eight): acc[nt] (+)= A B, with A and B read element-wise through the
// callables fa(r, k) and fb(k, n) (fp32 in shared memory), acc in the m16n8 accumulator layout
// (g = lane / 4, t = lane % 4): acc[nt] = {C[g][8 nt + 2 t], C[g][8 nt + 2 t + 1],
// C[g + 8][8 nt + 2 t], C[g + 8][8 nt + 2 t + 1]}.
template <class FA, class FB>
__device__ __forceinline__ void mma16(float (&acc)[2][4], FA fa, FB fb, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const uint32_t a[4] = {to_tf32(fa(g, 8 * ks + t)), to_tf32(fa(g + 8, 8 * ks + t)),
                           to_tf32(fa(g, 8 * ks + t + 4)), to_tf32(fa(g + 8, 8 * ks + t + 4))};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t bb[2] = {to_tf32(fb(8 * ks + t, 8 * nt + g)), to_tf32(fb(8 * ks + t + 4, 8 * nt + g))};
      mma_tf32_16x8x8(acc[nt], a, bb);
    }
  }
}

// T = (I + A)^{-1}, with D_b = (I + A_bb)^{-1} the inverses of the 16 x 16 diagonal blocks and
// L = D A_off (block strictly lower, so L^4 = 0): T = (I - L + L^2 - L^3) D, i.e. below the
// diagonal T_bq = X_bq D_q with X_10 = -L_10, X_21 = -L_21, X_32 = -L_32, X_20 = -L_20 + L_21 L_10,
// X_31 = -L_31 + L_32 L_21, X_30 = -L_30 + L_31 L_10 - L_32 X_20.  Written as the bf16 operands
// tw = (T diag(VEC_SW))^T and tu = (T diag(VEC_BETA))^T (MN-major [64 j][64 i], 128-byte
// swizzled), and T^T itself to tt_b unless that is null.  sA is overwritten.  Synchronises the group after steps 1a and 1b; the caller
// fences and syncs before the operands are read.
template <int kBar>
__device__ void solve_t(float* sA, float* sTd, const float* vec, uint8_t* tw_b, uint8_t* tu_b,
                        uint8_t* tt_b) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // step 1a (CUDA cores): the diagonal-block inverses D_b = (I + A_bb)^{-1}, one column per
  //      thread by a right-looking substitution (warp w < 2: lanes 0-15 block 2 w, lanes 16-31
  //      block 2 w + 1).  D_b goes to sTd (column-major) and to the diagonal blocks of Tw / Tu,
  //      together with the zeros that precede them.
  if (warp < 2) {
    const int b = 2 * warp + (lane >> 4), j = lane & 15;
    // A[16 b + i][16 b + m] = ab[i / 4][64 i + 4 ((m / 4) ^ (i % 4)) + m % 4]
    const float* ab[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ab[k] = sA + 1024 * b + (((4 * b) ^ (4 * k)) << 2);
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {   // columns m = 4 g .. 4 g + 3 of A_bb, one float4 per row
      float4 ag[16];
#pragma unroll
      for (int i = 4 * g + 1; i < 16; ++i)
        ag[i] = *reinterpret_cast<const float4*>(ab[i >> 2] + 64 * i + ((g ^ (i & 3)) << 2));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 4 * g + e;
#pragma unroll
        for (int i = m + 1; i < 16; ++i) {
          const float am = e == 0 ? ag[i].x : (e == 1 ? ag[i].y : (e == 2 ? ag[i].z : ag[i].w));
          x[i] = fmaf(-am, x[m], x[i]);
        }
      }
    }
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4)
      *reinterpret_cast<float4*>(&sTd[(b * 16 + j) * TD_LD + 4 * i4]) =
          make_float4(x[4 * i4], x[4 * i4 + 1], x[4 * i4 + 2], x[4 * i4 + 3]);
    // row jr = 16 b + j of (T diag(beta exp(G) r_k))^T and (T diag(beta))^T: the zeros
    // before the diagonal block and the diagonal block itself
    const int jr = 16 * b + j;
    const float sw = vec[VEC_SW + jr], sb = vec[VEC_BETA + jr];
    float w[16], u[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) { w[i] = x[i] * sw; u[i] = x[i] * sb; }
    store_bf16x8(tw_b + sw128_offset(jr, 16 * b), w);
    store_bf16x8(tw_b + sw128_offset(jr, 16 * b + 8), w + 8);
    store_bf16x8(tu_b + sw128_offset(jr, 16 * b), u);
    store_bf16x8(tu_b + sw128_offset(jr, 16 * b + 8), u + 8);
    if (tt_b) {
      store_bf16x8(tt_b + sw128_offset(jr, 16 * b), x);
      store_bf16x8(tt_b + sw128_offset(jr, 16 * b + 8), x + 8);
    }
    const float zeros[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i8 = 0; i8 < 2 * b; ++i8) {
      store_bf16x8(tw_b + sw128_offset(jr, 8 * i8), zeros);
      store_bf16x8(tu_b + sw128_offset(jr, 8 * i8), zeros);
      if (tt_b) store_bf16x8(tt_b + sw128_offset(jr, 8 * i8), zeros);
    }
  }
  group_sync(kBar, kPrepThreads);
  // step 1b (tensor cores, warp-level tf32 mma.sync): L_bq = D_b A_bq, warp w < 6 one block
  //      ((1,0) (2,0) (3,0) (2,1) (3,1) (3,2)), written over A_bq
  if (warp < 6) {
    const int b = warp < 3 ? warp + 1 : (warp < 5 ? warp - 1 : 3);
    const int q = warp < 3 ? 0 : (warp < 5 ? 1 : 2);
    const int g = lane >> 2, t = lane & 3;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const float* db = sTd + b * 16 * TD_LD;
    mma16(acc, [db](int r, int k) { return db[k * TD_LD + r]; },
          [sA, b, q](int k, int n) { return sA[a_idx(16 * b + k, 16 * q + n)]; }, lane);
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sA[a_idx(16 * b + g, 16 * q + 8 * nt + 2 * t)] = acc[nt][0];
      sA[a_idx(16 * b + g, 16 * q + 8 * nt + 2 * t + 1)] = acc[nt][1];
      sA[a_idx(16 * b + g + 8, 16 * q + 8 * nt + 2 * t)] = acc[nt][2];
      sA[a_idx(16 * b + g + 8, 16 * q + 8 * nt + 2 * t + 1)] = acc[nt][3];
    }
  }
  group_sync(kBar, kPrepThreads);
  // steps 2-3 (tensor cores, warp-level tf32 mma.sync): warp w < 6 computes one block T_bq below
  //      the diagonal: w 0 T_30, 1 T_20, 2 T_31, 3 T_10, 4 T_21, 5 T_32.  An X that is itself a
  //      product goes back through a free upper-triangle block of sA to become an A operand:
  //      X_20 at (0, 2), which warp 1 also shares with warp 0 through a 64-thread named
  //      barrier, X_31 at (1, 2), X_30 at (1, 3).
  if (warp < 6) {
    const int b = warp == 0 ? 3 : (warp == 1 ? 2 : (warp == 2 ? 3 : warp - 2));
    const int q = warp == 0 ? 0 : (warp == 1 ? 0 : (warp == 2 ? 1 : warp - 3));
    const int g = lane >> 2, t = lane & 3;
    auto blk = [sA](int bb, int qq) {   // element (r, c) of the 16 x 16 block (bb, qq) of sA
      return [sA, bb, qq](int r, int c) { return sA[a_idx(16 * bb + r, 16 * qq + c)]; };
    };
    auto neg = [](float (&x)[2][4]) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[nt][e] = -x[nt][e];
    };
    // X_bq in the accumulator layout; the rows that X products need go through shared memory
    float x[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {   // start from -L_bq
      x[nt][0] = -sA[a_idx(16 * b + g, 16 * q + 8 * nt + 2 * t)];
      x[nt][1] = -sA[a_idx(16 * b + g, 16 * q + 8 * nt + 2 * t + 1)];
      x[nt][2] = -sA[a_idx(16 * b + g + 8, 16 * q + 8 * nt + 2 * t)];
      x[nt][3] = -sA[a_idx(16 * b + g + 8, 16 * q + 8 * nt + 2 * t + 1)];
    }
    if (warp == 1 || warp == 2) {       // X_20 = -L_20 + L_21 L_10,  X_31 = -L_31 + L_32 L_21
      mma16(x, blk(b, b - 1), blk(b - 1, q), lane);
    }
    if (warp == 1) {                    // publish X_20 for warp 0
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sA[a_idx(g, 32 + 8 * nt + 2 * t)] = x[nt][0];
        sA[a_idx(g, 32 + 8 * nt + 2 * t + 1)] = x[nt][1];
        sA[a_idx(g + 8, 32 + 8 * nt + 2 * t)] = x[nt][2];
        sA[a_idx(g + 8, 32 + 8 * nt + 2 * t + 1)] = x[nt][3];
      }
    }
    if (warp <= 1) group_sync(kBar + 3, 64);
    if (warp == 0) {                    // X_30 = -L_30 + L_31 L_10 - L_32 X_20
      mma16(x, blk(3, 1), blk(1, 0), lane);
      neg(x);
      mma16(x, blk(3, 2), blk(0, 2), lane);   // X_20 sits at block (0, 2)
      neg(x);
      // X_30 must become the A operand of the last product: through its own scratch block
      // (1, 3), read back by the same warp
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sA[a_idx(16 + g, 48 + 8 * nt + 2 * t)] = x[nt][0];
        sA[a_idx(16 + g, 48 + 8 * nt + 2 * t + 1)] = x[nt][1];
        sA[a_idx(24 + g, 48 + 8 * nt + 2 * t)] = x[nt][2];
        sA[a_idx(24 + g, 48 + 8 * nt + 2 * t + 1)] = x[nt][3];
      }
      __syncwarp();
    } else if (warp == 2) {             // X_31 back as the A operand through block (1, 2)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sA[a_idx(16 + g, 32 + 8 * nt + 2 * t)] = x[nt][0];
        sA[a_idx(16 + g, 32 + 8 * nt + 2 * t + 1)] = x[nt][1];
        sA[a_idx(24 + g, 32 + 8 * nt + 2 * t)] = x[nt][2];
        sA[a_idx(24 + g, 32 + 8 * nt + 2 * t + 1)] = x[nt][3];
      }
      __syncwarp();
    }
    // T_bq = X_bq D_q (D_q column-major in sTd)
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const float* dq = sTd + q * 16 * TD_LD;
    auto fd = [dq](int k, int n) { return dq[n * TD_LD + k]; };
    if (warp >= 3) {                    // X = -L_bq straight from step 1
      auto fx = [sA, b, q](int r, int k) { return -sA[a_idx(16 * b + r, 16 * q + k)]; };
      mma16(acc, fx, fd, lane);
    } else {
      // X_30 at block (1, 3), X_20 at (0, 2), X_31 at (1, 2)
      const int rb = warp == 1 ? 0 : 1, cb = warp == 0 ? 3 : 2;
      mma16(acc, blk(rb, cb), fd, lane);
    }
    // out: Tw^T row j = 16 q + 8 nt + r, columns i = 16 b + 8 h .. + 7 from the transposing
    // stmatrix (matrix m = 2 nt + h holds rows 8 h .. 8 h + 7 of column tile nt)
    uint32_t fw[4], fu[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int j0 = 16 * q + 8 * nt + 2 * t;
      const float sw0 = vec[VEC_SW + j0], sw1 = vec[VEC_SW + j0 + 1];
      const float sb0 = vec[VEC_BETA + j0], sb1 = vec[VEC_BETA + j0 + 1];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        fw[2 * nt + h] = pack_bf16x2(acc[nt][2 * h] * sw0, acc[nt][2 * h + 1] * sw1);
        fu[2 * nt + h] = pack_bf16x2(acc[nt][2 * h] * sb0, acc[nt][2 * h + 1] * sb1);
      }
    }
    const int m = lane >> 3, r = lane & 7;
    const uint32_t off = sw128_offset(16 * q + 8 * (m >> 1) + r, 16 * b + 8 * (m & 1));
    stmatrix_x4_trans(smem_u32(tw_b) + off, fw);
    stmatrix_x4_trans(smem_u32(tu_b) + off, fu);
    if (tt_b) {
      uint32_t ft[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) ft[2 * nt + h] = pack_bf16x2(acc[nt][2 * h], acc[nt][2 * h + 1]);
      stmatrix_x4_trans(smem_u32(tt_b) + off, ft);
    }
  }
}

}  // namespace
}  // namespace gdn
