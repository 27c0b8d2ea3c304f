// gdn_chunk_tc.cu -- fused chunkwise gated delta rule on the tcgen05 tensor cores.
//
// One CTA per (sequence, value head), bf16 I/O, K = V = 128, chunk 64.  TMA
// brings each chunk's Q, K, V tiles into 128-byte-swizzled shared memory, every
// contraction is a tcgen05.mma with its fp32 accumulator in TMEM, and the K x V
// fp32 state lives in TMEM for the whole sequence.  Per chunk (G = in-chunk
// cumulative log-decay, r_q / r_k = inverse L2 norms, S = state entering the chunk):
//
//   D1  = [Q; K] K^T                       M=128 N=64  K=128   (Q K^T and K K^T)
//   P   = r_q r_k^T * Q K^T * exp(G_i - G_j) * [j <= i]          (bf16, smem)
//   A   = beta r_k r_k^T * K K^T * exp(G_i - G_j) * [j < i]      (fp32, smem)
//   T   = (I + A)^{-1}                     16 x 16 diagonal blocks, then block rows
//   W^T = K^T (T diag(beta exp(G) r_k))^T  M=128 N=64  K=64
//   U^T = V^T (T diag(beta))^T             M=128 N=64  K=64
//   U'^T = U^T - S^T W^T                   M=128 N=64  K=128   (accumulates on U^T)
//   O1  = S^T Q^T                          M=128 N=64  K=128
//   O2  = U'^T P^T                         M=128 N=64  K=64
//   S^T <- exp(G_last) S^T + (U' * exp(G_last - G) r_k)^T K     M=128 N=128 K=64
//   o   = scale (exp(G) r_q * O1 + O2)
//
// Every product is oriented so M = 128 (value or key features on the TMEM
// lanes, tokens on the columns).  The CTA is warp-specialised: a prep group
// (warps 0-7) builds everything that does not depend on the state -- norms,
// D1, P, A, T, W, U -- for chunk c + 1 while a state group (warps 8-11) runs
// the state-dependent part of chunk c (U', O, the state update, the output);
// they hand chunks over through mbarriers, double-buffering P, U, the per-token
// vectors and the TMA stages.  These are the chunkwise (WY / UT transform)
// equations of the gated delta rule with the chunking of the inference kernels
// ("Megatron-Core API: core.ssm.gated_delta_product", ssm_inference_chunk_size:
// a fixed 64) and the argument set of torch_chunk_gated_delta_rule ("Megatron-
// Core API: core.ssm.gated_delta_net.gdn").  Every wait is bounded; a timeout
// sets GDN_DEV_TIMEOUT, drains, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kPrepThreads = 256;   // warps 0-7
constexpr int kStateThreads = 128;  // warps 8-11
constexpr int kTcThreads = kPrepThreads + kStateThreads;
constexpr int kBarPrep = 1, kBarState = 2;   // named barrier ids
constexpr int DK = 128, DV = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Shared memory map (bytes from a 1024-byte-aligned base).
constexpr uint32_t OFF_QK = 0;          // 2 stages x 32 KB: [dk half][Q rows 0-63 | K rows 64-127][128 B]
constexpr uint32_t QK_STAGE = 32768;
constexpr uint32_t OFF_V = 65536;       // 2 stages x 16 KB: [dv half][64 tokens][128 B]
constexpr uint32_t V_STAGE = 16384;
constexpr uint32_t OFF_S = 98304;       // S^T bf16, A operand: [dk half][128 dv rows][128 B]; after
                                        // the MMAs that read it, the bf16 output tile staged for a
                                        // TMA store
constexpr uint32_t OFF_W = 131072;      // -W^T bf16, MN-major B: [128 dk rows][64 tokens]
constexpr uint32_t OFF_A = 147456;      // fp32 A [64][64], 16-byte-group swizzled; the solve
                                        // overwrites its strictly-lower blocks with those of T
constexpr uint32_t OFF_P = 163840;      // 2 x P, K-major B [64 i][64 j]
constexpr uint32_t OFF_U = 180224;      // U'^T bf16, K-major A [128 dv][64 tokens]
constexpr uint32_t OFF_TW = 196608;     // (T diag(beta exp(G) r_k))^T, MN-major B [64 j][64 i]
constexpr uint32_t OFF_TU = 204800;     // (T diag(beta))^T, MN-major B
constexpr uint32_t OFF_VEC = 212992;    // 2 x per-token fp32 vectors [7][64]
constexpr uint32_t VEC_G = 0, VEC_BETA = 64, VEC_RQ = 128, VEC_RK = 192, VEC_SW = 256,
                   VEC_DL = 320, VEC_QS = 384, VEC_FLOATS = 448;
constexpr uint32_t OFF_TD = OFF_VEC + 2 * 4 * VEC_FLOATS;  // diagonal blocks of T [4][16][16]
constexpr uint32_t OFF_YS = OFF_TD + 4 * 1024;             // per-warp 16 x 8 fp32 scratch
constexpr uint32_t OFF_BAR = OFF_YS + 8 * 512;
constexpr uint32_t SMEM_USED = OFF_BAR + 256;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base

constexpr uint32_t STAGE_TX = QK_STAGE + V_STAGE;  // Q + K + V bytes per stage = 48 KB

// TMEM columns (fp32, 128 lanes).  COL_S holds S^T for the whole sequence.
constexpr uint32_t COL_D1 = 0, COL_W = 64, COL_U = 128 /* 2 x 64 */, COL_O1 = 256,
                   COL_O2 = 320, COL_S = 384, TMEM_COLS = 512;

// mbarriers (8 bytes each) at OFF_BAR.
enum {
  B_FULL = 0,       // [2] TMA stage landed
  B_MMA_P = 2,      // prep group's MMA commits
  B_MMA_S = 3,      // state group's MMA commits
  B_READY = 4,      // [2] prep -> state: chunk ready (vectors, P, U, -W^T)
  B_W_FREE = 6,     // state -> prep: MMA on -W^T done
  B_U_FREE = 7,     // [2] state -> prep: U accumulator read
  B_P_FREE = 9,     // [2] state -> prep: MMA on P done
  B_VEC_FREE = 11,  // [2] state -> prep: per-token vectors no longer needed
  B_COUNT = 13
};
constexpr uint32_t OFF_FLAG = OFF_BAR + 8 * B_COUNT;      // int: a group timed out
constexpr uint32_t OFF_TSLOT = OFF_FLAG + 8;              // TMEM base address

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_TSLOT + 4 <= SMEM_USED, "barrier block");
static_assert(STAGE_TX == 49152, "stage bytes");

// fp32 A tile: element (i, j) at i * 64 + 4 * ((j / 4) ^ (i % 16)) + j % 4, so that
// 16-byte groups stay contiguous and the row-parallel accesses of the solve hit
// distinct banks.
__device__ __forceinline__ int a_idx(int i, int j) {
  return i * 64 + ((((j >> 2) ^ (i & 15)) << 2) | (j & 3));
}

__device__ __forceinline__ void store_bf16x8(uint8_t* p, const float* v) {
  __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 b2 = __floats2bfloat162_rn(v[4], v[5]);
  __nv_bfloat162 b3 = __floats2bfloat162_rn(v[6], v[7]);
  uint4 u;
  u.x = *reinterpret_cast<uint32_t*>(&b0);
  u.y = *reinterpret_cast<uint32_t*>(&b1);
  u.z = *reinterpret_cast<uint32_t*>(&b2);
  u.w = *reinterpret_cast<uint32_t*>(&b3);
  *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float sumsq_bf16x8(uint4 u) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    s += f.x * f.x + f.y * f.y;
  }
  return s;
}

// Issue the TMA loads of the chunk starting at token t into stage s.
__device__ __forceinline__ void issue_chunk_loads(uint8_t* sm, uint64_t* bar, const CUtensorMap* tq,
                                                  const CUtensorMap* tk, const CUtensorMap* tv,
                                                  int s, int t, int hq, int h) {
  mbar_arrive_expect_tx(bar, STAGE_TX);
  uint8_t* qk = sm + OFF_QK + s * QK_STAGE;
  uint8_t* vv = sm + OFF_V + s * V_STAGE;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    tma_load_3d(qk + hh * 16384, tq, bar, 64 * hh, hq, t);
    tma_load_3d(qk + hh * 16384 + 8192, tk, bar, 64 * hh, hq, t);
    tma_load_3d(vv + hh * 8192, tv, bar, 64 * hh, h, t);
  }
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
__device__ __forceinline__ void load_gates(const ChunkArgs& a, int t0, int h, int lane,
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

// 2^x on the special-function unit (inputs here are <= 0 or moderate).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool flag_set(const int* f) {
  return *reinterpret_cast<const volatile int*>(f) != 0;
}
__device__ __forceinline__ void set_flag(int* f) { *reinterpret_cast<volatile int*>(f) = 1; }

// =================================================================== prep group
// Warps 0-7.  For each chunk: gates, norms, D1 = [Q;K]K^T, P, A, T = (I+A)^{-1},
// W^T and U^T on the tensor core, -W^T to shared memory; then hands the chunk to
// the state group.
__device__ void prep_group(const ChunkArgs& a, uint8_t* sm, uint32_t tbase, int bos, int eos,
                           int nchunks, int h) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, chalf = warp >> 2;
  const int row = 32 * quad + lane;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  int* flag = reinterpret_cast<int*>(sm + OFF_FLAG);
  float* sA = reinterpret_cast<float*>(sm + OFF_A);
  float* sTd = reinterpret_cast<float*>(sm + OFF_TD);
  const bool leader = (tid == 0);
  uint32_t pp = 0;   // parity of B_MMA_P
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  float gq[2], bq[2];
  if (warp == 0) load_gates(a, bos, h, lane, T_total, gq, bq);
  const bool fused = a.gates.mode == kGatesFused;
  const float expA = fused ? expf(a.gates.A_log[h]) : 0.f;
  const float dtb = fused ? a.gates.dt_bias[h] : 0.f;

  for (int c = 0; c < nchunks; ++c) {
    const int s = c & 1;
    const int t0 = bos + c * kChunk;
    const int L = min(kChunk, eos - t0);
    float* vec = reinterpret_cast<float*>(sm + OFF_VEC) + s * VEC_FLOATS;
    uint8_t* qk = sm + OFF_QK + s * QK_STAGE;
    const uint32_t qk_a = sbase + OFF_QK + s * QK_STAGE;
    const uint32_t v_a = sbase + OFF_V + s * V_STAGE;

    // ---- per-token vectors of chunk c - 2 released; this chunk's tiles landed
    // (one thread polls each mbarrier; the rest of the group sleeps in the named barrier)
    bool ok = true;
    if (leader) {
      if (c >= 2) ok = mbar_wait(&bars[B_VEC_FREE + s], (uint32_t)((c - 2) >> 1) & 1u, kWaitLimitNs);
      ok = ok && mbar_wait(&bars[B_FULL + s], (uint32_t)(c >> 1) & 1u, kWaitLimitNs);
    }
    if (group_sync_or(kBarPrep, kPrepThreads, !ok || flag_set(flag))) { if (leader) set_flag(flag); return; }

    // ---- MMA: D1 = [Q;K] K^T, issued as soon as the tiles are in (overlaps gates and norms)
    if (leader) {
      tc_fence_after();
      const uint32_t id1 = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tbase + COL_D1, sdesc_sw128(qk_a + off, 16, 1024),
                 sdesc_sw128(qk_a + off + 8192, 16, 1024), id1, ks > 0);
      }
      mma_commit(&bars[B_MMA_P]);
    }

    // ---- gates: in-chunk cumulative log-decay and beta; prefetch the next chunk's
    if (warp == 0) {
      if (fused) {   // g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
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
      vec[VEC_G + lane] = g0 * kLog2e; vec[VEC_G + lane + 32] = g1 * kLog2e;   // base-2 log-decay
      vec[VEC_BETA + lane] = lane < L ? bq[0] : 0.f;
      vec[VEC_BETA + lane + 32] = lane + 32 < L ? bq[1] : 0.f;
      if (c + 1 < nchunks) load_gates(a, t0 + kChunk, h, lane, T_total, gq, bq);
    }
    // ---- inverse L2 norms of q and k rows: 4 threads per row, each reading four
    //      16-byte chunks chosen so a warp's loads fall in distinct banks
    {
      const int r = tid >> 2, part = tid & 3;
      const uint8_t* qrow = qk + (part >> 1) * 16384 + r * 128;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = ((part & 1) * 4 + m) ^ (r & 7);
        sq += sumsq_bf16x8(*reinterpret_cast<const uint4*>(qrow + 16 * ch));
        sk += sumsq_bf16x8(*reinterpret_cast<const uint4*>(qrow + 8192 + 16 * ch));
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 2);
      if (part == 0) {
        vec[VEC_RQ + r] = a.use_qk_l2norm ? 1.0f / sqrtf(sq + kL2Eps) : 1.0f;
        vec[VEC_RK + r] = a.use_qk_l2norm ? 1.0f / sqrtf(sk + kL2Eps) : 1.0f;
      }
    }
    group_sync(kBarPrep, kPrepThreads);
    if (tid < kChunk) {   // per-token scalars while the tensor core works
      const float gl = vec[VEC_G + L - 1], gt = vec[VEC_G + tid];
      const float et = ex2(gt), rk = vec[VEC_RK + tid];
      vec[VEC_SW + tid] = vec[VEC_BETA + tid] * et * rk;
      vec[VEC_DL + tid] = ex2(gl - gt) * rk;
      vec[VEC_QS + tid] = a.scale * et * vec[VEC_RQ + tid];
    }
    if (leader) {
      ok = mbar_wait(&bars[B_MMA_P], pp, kWaitLimitNs);
      if (c >= 2) ok = ok && mbar_wait(&bars[B_P_FREE + s], (uint32_t)((c - 2) >> 1) & 1u, kWaitLimitNs);
    }
    pp ^= 1u;
    if (group_sync_or(kBarPrep, kPrepThreads, !ok || flag_set(flag))) { if (leader) set_flag(flag); return; }
    tc_fence_after();

    // ---- P (bf16, rows 0-63 of D1) and A (fp32, rows 64-127 of D1)
    {
      float x[32];
      tmem_ld32(tbase + lane_off + COL_D1 + 32 * chalf, x);
      const int j0 = 32 * chalf;
      const float* G = vec + VEC_G;
      float gj[32], rkj[32];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float4 g4 = *reinterpret_cast<const float4*>(G + j0 + 4 * m);
        const float4 r4 = *reinterpret_cast<const float4*>(vec + VEC_RK + j0 + 4 * m);
        gj[4 * m] = g4.x; gj[4 * m + 1] = g4.y; gj[4 * m + 2] = g4.z; gj[4 * m + 3] = g4.w;
        rkj[4 * m] = r4.x; rkj[4 * m + 1] = r4.y; rkj[4 * m + 2] = r4.z; rkj[4 * m + 3] = r4.w;
      }
      const bool zero_tile = ((quad & 1) == 0) && chalf == 1;   // rows 0-31 x cols 32-63
      if (quad < 2) {
        const int i = row;
        const float gi = G[i], ri = (i < L) ? vec[VEC_RQ + i] : 0.f;
        if (zero_tile) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) x[jj] = 0.f;
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = j0 + jj;
            x[jj] = (j <= i) ? ri * rkj[jj] * x[jj] * ex2(gi - gj[jj]) : 0.f;
          }
        }
        uint8_t* dst = sm + OFF_P + s * 8192;
#pragma unroll
        for (int m = 0; m < 4; ++m) store_bf16x8(dst + sw128_offset(i, j0 + 8 * m), &x[8 * m]);
      } else {
        const int i = row - 64;
        const float gi = G[i], bi = vec[VEC_BETA + i] * vec[VEC_RK + i];
        if (zero_tile) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) x[jj] = 0.f;
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = j0 + jj;
            x[jj] = (j < i) ? bi * rkj[jj] * x[jj] * ex2(gi - gj[jj]) : 0.f;
          }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m)
          *reinterpret_cast<float4*>(&sA[a_idx(i, j0 + 4 * m)]) =
              make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
      }
    }
    tc_fence_before();
    group_sync(kBarPrep, kPrepThreads);

    // ---- T = (I + A)^{-1}, step 1: the four 16 x 16 diagonal blocks, one column per
    //      thread; each row is a dot product with four partial sums (short dependency chain)
    if (tid < 64) {
      const int b = tid >> 4, jj = tid & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == jj) ? 1.f : 0.f;
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if (4 * g < i) {
            const float4 a4 = *reinterpret_cast<const float4*>(&sA[a_idx(16 * b + i, 16 * b + 4 * g)]);
            if (4 * g + 0 < i) p[0] += a4.x * x[4 * g + 0];
            if (4 * g + 1 < i) p[1] += a4.y * x[4 * g + 1];
            if (4 * g + 2 < i) p[2] += a4.z * x[4 * g + 2];
            if (4 * g + 3 < i) p[3] += a4.w * x[4 * g + 3];
          }
        }
        const float v = -((p[0] + p[1]) + (p[2] + p[3]));
        if (i > jj) x[i] = v;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) sTd[(b * 16 + i) * 16 + jj] = x[i];
      // row j = 16 b + jj of (T diag(beta exp(G) r_k))^T and (T diag(beta))^T: the zeros
      // before the diagonal block and the diagonal block itself
      const int j = 16 * b + jj;
      const float sw = vec[VEC_SW + j], sb = vec[VEC_BETA + j];
      float w[16], u[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) { w[i] = x[i] * sw; u[i] = x[i] * sb; }
      store_bf16x8(sm + OFF_TW + sw128_offset(j, 16 * b), w);
      store_bf16x8(sm + OFF_TW + sw128_offset(j, 16 * b + 8), w + 8);
      store_bf16x8(sm + OFF_TU + sw128_offset(j, 16 * b), u);
      store_bf16x8(sm + OFF_TU + sw128_offset(j, 16 * b + 8), u + 8);
      const float zeros[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int i8 = 0; i8 < 2 * b; ++i8) {
        store_bf16x8(sm + OFF_TW + sw128_offset(j, 8 * i8), zeros);
        store_bf16x8(sm + OFF_TU + sw128_offset(j, 8 * i8), zeros);
      }
    }
    group_sync(kBarPrep, kPrepThreads);
    // ---- step 2: block row b from the rows above it, T[b, :16b] = -T_bb (A[b, :16b] T[:16b, :16b]),
    //      on the warp-level tf32 MMA: warp w owns columns 8w..8w+7; results overwrite A in place
    {
      const int g8 = lane >> 2, t4 = lane & 3;
      float* ys = reinterpret_cast<float*>(sm + OFF_YS) + warp * 128;
#pragma unroll
      for (int b = 1; b < 4; ++b) {
        const int nt = warp;
        const bool active = nt < 2 * b;       // warp-uniform
        float z[4] = {0.f, 0.f, 0.f, 0.f};
        if (active) {
          const int cb = nt >> 1;
          const int cc = 8 * nt + g8;
          float y[4] = {0.f, 0.f, 0.f, 0.f};
          for (int ks = nt; ks < 2 * b; ++ks) {
            uint32_t af[4], bf[2];
            af[0] = to_tf32(sA[a_idx(16 * b + g8, 8 * ks + t4)]);
            af[1] = to_tf32(sA[a_idx(16 * b + g8 + 8, 8 * ks + t4)]);
            af[2] = to_tf32(sA[a_idx(16 * b + g8, 8 * ks + t4 + 4)]);
            af[3] = to_tf32(sA[a_idx(16 * b + g8 + 8, 8 * ks + t4 + 4)]);
            const int k0 = 8 * ks + t4, k1 = k0 + 4;
            float b0, b1;
            if ((ks >> 1) == cb) {            // diagonal block of T
              b0 = sTd[(cb * 16 + (k0 & 15)) * 16 + (cc & 15)];
              b1 = sTd[(cb * 16 + (k1 & 15)) * 16 + (cc & 15)];
            } else {                          // T rows of an earlier round, stored over A
              b0 = sA[a_idx(k0, cc)];
              b1 = sA[a_idx(k1, cc)];
            }
            bf[0] = to_tf32(b0);
            bf[1] = to_tf32(b1);
            mma_tf32_16x8x8(y, af, bf);
          }
          ys[g8 * 8 + 2 * t4] = y[0];
          ys[g8 * 8 + 2 * t4 + 1] = y[1];
          ys[(g8 + 8) * 8 + 2 * t4] = y[2];
          ys[(g8 + 8) * 8 + 2 * t4 + 1] = y[3];
          __syncwarp();
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            uint32_t af[4], bf[2];
            const float* tb = sTd + (b * 16) * 16 + 8 * k2;
            af[0] = to_tf32(tb[g8 * 16 + t4]);
            af[1] = to_tf32(tb[(g8 + 8) * 16 + t4]);
            af[2] = to_tf32(tb[g8 * 16 + t4 + 4]);
            af[3] = to_tf32(tb[(g8 + 8) * 16 + t4 + 4]);
            bf[0] = to_tf32(ys[(8 * k2 + t4) * 8 + g8]);
            bf[1] = to_tf32(ys[(8 * k2 + t4 + 4) * 8 + g8]);
            mma_tf32_16x8x8(z, af, bf);
          }
          __syncwarp();
        }
        if (active) {
          // T block row b, columns c0, c0 + 1 of this tile -> Tw / Tu entries (row = column of T)
          const int r0 = 16 * b + g8, c0 = 8 * nt + 2 * t4;
          const float sw0 = vec[VEC_SW + c0], sw1 = vec[VEC_SW + c0 + 1];
          const float sb0 = vec[VEC_BETA + c0], sb1 = vec[VEC_BETA + c0 + 1];
          __nv_bfloat16* tw = reinterpret_cast<__nv_bfloat16*>(sm + OFF_TW);
          __nv_bfloat16* tu = reinterpret_cast<__nv_bfloat16*>(sm + OFF_TU);
          tw[sw128_offset(c0, r0) >> 1] = __float2bfloat16_rn(-z[0] * sw0);
          tw[sw128_offset(c0 + 1, r0) >> 1] = __float2bfloat16_rn(-z[1] * sw1);
          tw[sw128_offset(c0, r0 + 8) >> 1] = __float2bfloat16_rn(-z[2] * sw0);
          tw[sw128_offset(c0 + 1, r0 + 8) >> 1] = __float2bfloat16_rn(-z[3] * sw1);
          tu[sw128_offset(c0, r0) >> 1] = __float2bfloat16_rn(-z[0] * sb0);
          tu[sw128_offset(c0 + 1, r0) >> 1] = __float2bfloat16_rn(-z[1] * sb1);
          tu[sw128_offset(c0, r0 + 8) >> 1] = __float2bfloat16_rn(-z[2] * sb0);
          tu[sw128_offset(c0 + 1, r0 + 8) >> 1] = __float2bfloat16_rn(-z[3] * sb1);
        }
        if (b < 3) {
          group_sync(kBarPrep, kPrepThreads);   // all reads of A's block row b are done
          if (active) {   // fp32 T block for the later rounds, over A in place
            const int r0 = 16 * b + g8, c0 = 8 * nt + 2 * t4;
            sA[a_idx(r0, c0)] = -z[0];
            sA[a_idx(r0, c0 + 1)] = -z[1];
            sA[a_idx(r0 + 8, c0)] = -z[2];
            sA[a_idx(r0 + 8, c0 + 1)] = -z[3];
          }
          group_sync(kBarPrep, kPrepThreads);
        }
      }
    }
    fence_proxy_async_smem();
    group_sync(kBarPrep, kPrepThreads);

    // ---- MMA: W^T = K^T Tw^T, U^T = V^T Tu^T (all operands MN-major); U into its buffer
    //      once the state group has read the one two chunks back
    if (leader) {
      bool okl = true;
      if (c >= 2) okl = mbar_wait(&bars[B_U_FREE + s], (uint32_t)((c - 2) >> 1) & 1u, kWaitLimitNs);
      if (!okl) set_flag(flag);
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_W, sdesc_sw128(qk_a + 8192 + ks * 2048, 16384, 1024),
                 sdesc_sw128(sbase + OFF_TW + ks * 2048, 8192, 1024), id, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_U + 64 * s, sdesc_sw128(v_a + ks * 2048, 8192, 1024),
                 sdesc_sw128(sbase + OFF_TU + ks * 2048, 8192, 1024), id, ks > 0);
      }
      mma_commit(&bars[B_MMA_P]);
    }
    if (leader) {
      ok = mbar_wait(&bars[B_MMA_P], pp, kWaitLimitNs);
      if (c >= 1) ok = ok && mbar_wait(&bars[B_W_FREE], (uint32_t)(c - 1) & 1u, kWaitLimitNs);
    }
    pp ^= 1u;
    if (group_sync_or(kBarPrep, kPrepThreads, !ok || flag_set(flag))) { if (leader) set_flag(flag); return; }
    tc_fence_after();

    // ---- -W^T -> bf16 MN-major B operand [dk rows][tokens]
    {
      float x[32];
      tmem_ld32(tbase + lane_off + COL_W + 32 * chalf, x);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) x[jj] = -x[jj];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        store_bf16x8(sm + OFF_W + sw128_offset(row, 32 * chalf + 8 * m), &x[8 * m]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    group_sync(kBarPrep, kPrepThreads);
    if (leader) mbar_arrive(&bars[B_READY + s]);
  }
}

// =================================================================== state group
// Warps 8-11.  For each chunk: S -> bf16 operand and decay of the TMEM state,
// U' = U - S W, O1 = S Q^T, O2 = U' P^T, S += (decayed U')^T K, output.
__device__ void state_group(const ChunkArgs& a, uint8_t* sm, uint32_t tbase, int bos, int eos,
                            int nchunks, int h, int hq, size_t st_off,
                            const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                            const CUtensorMap* to) {
  const int tid = threadIdx.x - kPrepThreads, wq = tid >> 5, lane = tid & 31;
  const int row = 32 * wq + lane;
  const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  int* flag = reinterpret_cast<int*>(sm + OFF_FLAG);
  const bool leader = (tid == 0);
  uint32_t ps = 0;   // parity of B_MMA_S
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o);
  bool failed = false;

  for (int c = 0; c < nchunks; ++c) {
    const int s = c & 1;
    const int t0 = bos + c * kChunk;
    const int L = min(kChunk, eos - t0);
    const float* vec = reinterpret_cast<const float*>(sm + OFF_VEC) + s * VEC_FLOATS;
    const uint32_t qk_a = sbase + OFF_QK + s * QK_STAGE;

    bool ok = true;
    if (leader) {
      ok = mbar_wait(&bars[B_READY + s], (uint32_t)(c >> 1) & 1u, kWaitLimitNs);
      tma_store_wait_read();   // the previous output tile (staged where S^T goes) has been read
    }
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    tc_fence_after();

    // ---- S (entry state) -> bf16 A operand S^T [dv rows][dk]; S <- exp(G_last) S in TMEM
    {
      const float dl = ex2(vec[VEC_G + L - 1]);
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        float x[32];
        const uint32_t col = COL_S + 32 * part;
        tmem_ld32(tbase + lane_off + col, x);
        uint8_t* dst = sm + OFF_S + (part >> 1) * 16384;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          store_bf16x8(dst + sw128_offset(row, 32 * (part & 1) + 8 * m), &x[8 * m]);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] *= dl;
        tmem_st32(tbase + lane_off + col, x);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    group_sync(kBarState, kStateThreads);

    // ---- MMA: U'^T = U^T + S^T (-W^T);  O1 = S^T Q^T
    if (leader) {
      tc_fence_after();
      const uint32_t id4 = idesc_bf16(128, 64, false, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_bf16(tbase + COL_U + 64 * s,
                 sdesc_sw128(sbase + OFF_S + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                 sdesc_sw128(sbase + OFF_W + ks * 2048, 8192, 1024), id4, 1);
      }
      mma_commit(&bars[B_W_FREE]);
      const uint32_t id5 = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tbase + COL_O1, sdesc_sw128(sbase + OFF_S + off, 16, 1024),
                 sdesc_sw128(qk_a + off, 16, 1024), id5, ks > 0);
      }
      mma_commit(&bars[B_MMA_S]);
    }
    if (leader) ok = mbar_wait(&bars[B_MMA_S], ps, kWaitLimitNs);
    ps ^= 1u;
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    tc_fence_after();

    // ---- U'^T -> bf16 K-major A operand [dv rows][tokens]; K tile rows scaled by
    //      exp(G_last - G_t) r_k[t] in place (the state update's B operand; the prep
    //      group is done with this K tile)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float x[32];
      tmem_ld32(tbase + lane_off + COL_U + 64 * s + 32 * half, x);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        store_bf16x8(sm + OFF_U + sw128_offset(row, 32 * half + 8 * m), &x[8 * m]);
    }
    {
      const int t = tid >> 1, kh = tid & 1;
      const float dl = vec[VEC_DL + t];
      uint8_t* krow = sm + OFF_QK + s * QK_STAGE + kh * 16384 + 8192 + t * 128;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint4 u = *reinterpret_cast<uint4*>(krow + 16 * m);
        __nv_bfloat162* b2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(b2[e]);
          b2[e] = __floats2bfloat162_rn(f.x * dl, f.y * dl);
        }
        *reinterpret_cast<uint4*>(krow + 16 * m) = u;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    group_sync(kBarState, kStateThreads);

    // ---- MMA: O2 = U'^T P^T, S^T += Ut^T K
    if (leader) {
      mbar_arrive(&bars[B_U_FREE + s]);
      tc_fence_after();
      const uint32_t id6 = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_O2, sdesc_sw128(sbase + OFF_U + ks * 32, 16, 1024),
                 sdesc_sw128(sbase + OFF_P + s * 8192 + ks * 32, 16, 1024), id6, ks > 0);
      }
      const uint32_t id7 = idesc_bf16(128, 128, false, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_S, sdesc_sw128(sbase + OFF_U + ks * 32, 16, 1024),
                 sdesc_sw128(qk_a + 8192 + ks * 2048, 16384, 1024), id7, 1);
      }
      mma_commit(&bars[B_P_FREE + s]);
      mma_commit(&bars[B_MMA_S]);
    }
    if (leader) ok = mbar_wait(&bars[B_MMA_S], ps, kWaitLimitNs);
    ps ^= 1u;
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    tc_fence_after();
    // Stage s is free again: load chunk c + 2 into it.
    if (leader && c + 2 < nchunks) {
      fence_proxy_async_smem();
      issue_chunk_loads(sm, &bars[B_FULL + s], tq, tk, tv, s, t0 + 2 * kChunk, hq, h);
    }

    // ---- o = scale (exp(G) r_q O1 + O2): a full chunk is staged as a bf16 tile (two
    //      128-byte-swizzled [64 tokens][64 dv] halves) and written by one TMA store;
    //      the last, partial chunk of a sequence is stored row by row
    if (L == kChunk) {
      uint8_t* stage = sm + OFF_S + (row >> 6) * 8192;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float x[32], y[32];
        tmem_ld32(tbase + lane_off + COL_O1 + 32 * half, x);
        tmem_ld32(tbase + lane_off + COL_O2 + 32 * half, y);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int t = 32 * half + jj;
          *reinterpret_cast<__nv_bfloat16*>(stage + sw128_offset(t, row & 63)) =
              __float2bfloat16_rn(vec[VEC_QS + t] * x[jj] + a.scale * y[jj]);
        }
      }
      fence_proxy_async_smem();
      group_sync(kBarState, kStateThreads);
      if (leader) {
        tma_store_3d(to, sm + OFF_S, 0, h, t0);
        tma_store_3d(to, sm + OFF_S + 8192, 64, h, t0);
        tma_store_commit();
      }
    } else {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float x[32], y[32];
        tmem_ld32(tbase + lane_off + COL_O1 + 32 * half, x);
        tmem_ld32(tbase + lane_off + COL_O2 + 32 * half, y);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int t = 32 * half + jj;
          if (t < L)
            out[((size_t)(t0 + t) * a.Hv + h) * DV + row] =
                __float2bfloat16_rn(vec[VEC_QS + t] * x[jj] + a.scale * y[jj]);
        }
      }
    }
    tc_fence_before();
    group_sync(kBarState, kStateThreads);
    if (leader) mbar_arrive(&bars[B_VEC_FREE + s]);
  }

  if (leader) tma_store_wait_all();   // output tiles written before the CTA exits
  if (failed) {
    if (leader) {
      set_flag(flag);
      mbar_wait(&bars[B_MMA_S], ps ^ 1u, kWaitLimitNs);   // last commit, if any, has landed
    }
  } else if (a.final_state) {
    tc_fence_after();
#pragma unroll
    for (int part = 0; part < 4; ++part) {
      float x[32];
      tmem_ld32(tbase + lane_off + COL_S + 32 * part, x);
#pragma unroll
      for (int j = 0; j < 32; ++j) a.final_state[st_off + (size_t)(32 * part + j) * DV + row] = x[j];
    }
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  int* flag = reinterpret_cast<int*>(sm + OFF_FLAG);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x % a.Hv, n = blockIdx.x / a.Hv;
  const int hq = h / (a.Hv / a.Hqk);
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  int bos, eos;
  if (a.cu_seqlens) { bos = a.cu_seqlens[n]; eos = a.cu_seqlens[n + 1]; }
  else { bos = n * a.T; eos = bos + a.T; }
  if (bos < 0 || eos < bos || eos > T_total) {
    if (tid == 0) report(a.dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  int slot = n;
  if (a.state_indices) {
    slot = a.state_indices[n];
    if (slot < 0 || slot >= a.num_slots) {   // padding sequence: zero rows, no state access
      if (slot != -1 && tid == 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
      for (int e = tid; e < (eos - bos) * DV; e += kTcThreads) {
        const int t = e / DV, d = e - t * DV;
        o[((size_t)(bos + t) * a.Hv + h) * DV + d] = __float2bfloat16_rn(0.f);
      }
      return;
    }
  }
  const size_t st_off = ((size_t)slot * a.Hv + h) * (size_t)(DK * DV);
  const int nchunks = (eos - bos + kChunk - 1) / kChunk;
  if (nchunks == 0) {   // empty sequence: the state passes through unchanged
    if (a.final_state) {
      for (int e = tid; e < DK * DV; e += kTcThreads)
        a.final_state[st_off + e] = a.initial_state ? a.initial_state[st_off + e] : 0.f;
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
    *flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (tid < kPrepThreads) {
    if (tid == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      issue_chunk_loads(sm, &bars[B_FULL + 0], &tmQ, &tmK, &tmV, 0, bos, hq, h);
      if (nchunks > 1)
        issue_chunk_loads(sm, &bars[B_FULL + 1], &tmQ, &tmK, &tmV, 1, bos + kChunk, hq, h);
    }
    prep_group(a, sm, tbase, bos, eos, nchunks, h);
  } else {
    // Initial state -> TMEM (S^T: lane = value index, columns = key index).
    const int row = 32 * ((tid - kPrepThreads) >> 5) + (tid & 31);
    const uint32_t lane_off = (uint32_t)(32 * ((tid - kPrepThreads) >> 5)) << 16;
#pragma unroll
    for (int part = 0; part < 4; ++part) {
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        x[j] = a.initial_state ? a.initial_state[st_off + (size_t)(32 * part + j) * DV + row] : 0.f;
      tmem_st32(tbase + lane_off + COL_S + 32 * part, x);
    }
    state_group(a, sm, tbase, bos, eos, nchunks, h, hq, st_off, &tmQ, &tmK, &tmV, &tmO);
  }

  __syncthreads();
  if (tid == 0 && flag_set(flag)) {
    report(a.dev_status, GDN_DEV_TIMEOUT);
    // Drain the TMA loads that may still be in flight before the CTA exits.
    mbar_wait(&bars[B_FULL + 0], 0u, kWaitLimitNs / 4);
    mbar_wait(&bars[B_FULL + 1], 0u, kWaitLimitNs / 4);
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [T_total, H, 128] bf16 -> 3-D map with 64 x 1 x 64 boxes, 128-byte swizzle,
// zero fill past the last token.
bool encode_map(CUtensorMap* m, const void* base, int H, int T_total) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T_total};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(int K, int V, int io_dtype, int beta_dtype) {
  return K == DK && V == DV && io_dtype == GDN_BF16 &&
         (beta_dtype == GDN_BF16 || beta_dtype == GDN_F32);
}

cudaError_t launch_chunk_tc(const ChunkArgs& a) {
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  CUtensorMap mq, mk, mv, mo;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  memset(&mo, 0, sizeof(mo));
  if (T_total > 0) {
    if (!encode_map(&mq, a.q, a.Hqk, T_total) || !encode_map(&mk, a.k, a.Hqk, T_total) ||
        !encode_map(&mv, a.v, a.Hv, T_total) || !encode_map(&mo, a.o, a.Hv, T_total))
      return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)a.num_seqs * a.Hv;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  chunk_tc_kernel<<<(unsigned)blocks, kTcThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, a);
  return cudaGetLastError();
}

}  // namespace gdn
