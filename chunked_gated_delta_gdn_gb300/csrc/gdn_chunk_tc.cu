// gdn_chunk_tc.cu -- fused chunkwise gated delta rule on the tcgen05 tensor cores.
//
// One CTA per (sequence, value head), bf16 I/O, K = V = 128, chunk 64.  The
// whole chunk pipeline runs on chip: TMA brings each chunk's Q, K, V tiles into
// 128-byte-swizzled shared memory (double-buffered), every contraction is a
// tcgen05.mma with its fp32 accumulator in TMEM, the 64 x 64 unit-lower-
// triangular solve runs in fp32 registers, and the K x V fp32 state lives in
// TMEM for the whole sequence.  Per chunk (G = in-chunk cumulative log-decay,
// r_q / r_k = inverse L2 norms, S = state entering the chunk):
//
//   D1  = [Q; K] K^T                       M=128 N=64  K=128   (Q K^T and K K^T)
//   O1  = S^T Q^T                          M=128 N=64  K=128
//   P   = r_q r_k^T * Q K^T * exp(G_i - G_j) * [j <= i]          (bf16, smem)
//   A   = beta r_k r_k^T * K K^T * exp(G_i - G_j) * [j < i]      (fp32, smem)
//   T   = (I + A)^{-1}                     16 x 16 diagonal blocks, then block rows
//   W^T = K^T (T diag(beta exp(G) r_k))^T  M=128 N=64  K=64
//   U^T = V^T (T diag(beta))^T             M=128 N=64  K=64
//   U'^T = U^T - S^T W^T                   M=128 N=64  K=128   (accumulates on U^T)
//   O2  = U'^T P^T                         M=128 N=64  K=64
//   S^T <- exp(G_last) S^T + (U' * exp(G_last - G) r_k)^T K     M=128 N=128 K=64
//   o   = scale (exp(G) r_q * O1 + O2)
//
// Every product is oriented so M = 128 (value or key features on the TMEM
// lanes, tokens on the columns).  These are the chunkwise (WY / UT transform)
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

constexpr int kTcThreads = 256;
constexpr int DK = 128, DV = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Shared memory map (bytes from a 1024-byte-aligned base).
constexpr uint32_t OFF_QK = 0;          // 2 stages x 32 KB: [dk half][Q rows 0-63 | K rows 64-127][128 B]
constexpr uint32_t QK_STAGE = 32768;
constexpr uint32_t OFF_V = 65536;       // 2 stages x 16 KB: [dv half][64 tokens][128 B]
constexpr uint32_t V_STAGE = 16384;
constexpr uint32_t OFF_S = 98304;       // S^T bf16, A operand: [dk half][128 dv rows][128 B]
constexpr uint32_t OFF_W = 131072;      // -W^T bf16, MN-major B: [128 dk rows][64 tokens]
constexpr uint32_t OFF_TW = 147456;     // (T diag(beta exp(G) r_k))^T, MN-major B: [64 j][64 i]
constexpr uint32_t OFF_TU = 155648;     // (T diag(beta))^T, MN-major B
constexpr uint32_t OFF_P = 163840;      // P, K-major B [64 i][64 j]
constexpr uint32_t OFF_U = 172032;      // U'^T bf16, K-major A [128 dv][64 tokens]
constexpr uint32_t OFF_UT = 188416;     // (U' exp(G_last - G) r_k)^T bf16
constexpr uint32_t OFF_A = OFF_U;       // fp32 A [64][64], 16-byte-group swizzled (aliases U'^T,
                                        // which is written later in the chunk)
constexpr uint32_t OFF_VEC = 204800;    // per-token fp32 vectors, T diagonal blocks, barriers
constexpr uint32_t VEC_G = 0, VEC_BETA = 64, VEC_RQ = 128, VEC_RK = 192, VEC_SW = 256,
                   VEC_DL = 320, VEC_QS = 384, VEC_TD = 448;   // floats; TD is [4][16][16]
constexpr uint32_t OFF_BAR = OFF_VEC + 4 * (448 + 4 * 256);    // 8-byte aligned
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base

constexpr uint32_t STAGE_TX = QK_STAGE + V_STAGE;  // Q + K + V bytes per stage = 48 KB

// TMEM columns (fp32, 128 lanes).  COL_S holds S^T for the whole sequence.
constexpr uint32_t COL_D1 = 0, COL_W = 64, COL_U = 128, COL_O1 = 192, COL_O2 = 256,
                   COL_S = 320, TMEM_COLS = 512;

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
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

// g and beta of tokens t0 + lane and t0 + lane + 32 (zero past the chunk end).
__device__ __forceinline__ void load_gates(const ChunkArgs& a, int t0, int L, int h, int lane,
                                           float* g, float* b) {
  g[0] = g[1] = b[0] = b[1] = 0.f;
  if (lane < L) {
    g[0] = a.g[(size_t)(t0 + lane) * a.Hv + h];
    b[0] = load_elem(a.beta, (size_t)(t0 + lane) * a.Hv + h, a.beta_dtype);
  }
  if (lane + 32 < L) {
    g[1] = a.g[(size_t)(t0 + lane + 32) * a.Hv + h];
    b[1] = load_elem(a.beta, (size_t)(t0 + lane + 32) * a.Hv + h, a.beta_dtype);
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* vec = reinterpret_cast<float*>(sm + OFF_VEC);
  float* sG = vec + VEC_G;
  float* sBeta = vec + VEC_BETA;
  float* sRq = vec + VEC_RQ;
  float* sRk = vec + VEC_RK;
  float* sSw = vec + VEC_SW;
  float* sDl = vec + VEC_DL;
  float* sQs = vec + VEC_QS;
  float* sTd = vec + VEC_TD;   // diagonal 16 x 16 blocks of T: [block][row][col]
  float* sA = reinterpret_cast<float*>(sm + OFF_A);
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // [2]
  uint64_t* bar_mma = bar_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_full + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  // This thread's TMEM lane (a value or key feature index) and column half.
  const int quad = warp & 3, chalf = warp >> 2;
  const int row = 32 * quad + lane;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  const size_t st_off = ((size_t)slot * a.Hv + h) * (size_t)(DK * DV);
  const int nchunks = (eos - bos + kChunk - 1) / kChunk;
  if (nchunks == 0) {   // empty sequence: the state passes through unchanged
    if (a.final_state) {
      for (int j = 0; j < 64; ++j) {
        const size_t e = st_off + (size_t)(64 * chalf + j) * DV + row;
        a.final_state[e] = a.initial_state ? a.initial_state[e] : 0.f;
      }
    }
    return;
  }

  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(bar_mma, 1);
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
  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    issue_chunk_loads(sm, &bar_full[0], &tmQ, &tmK, &tmV, 0, bos, hq, h);
    if (nchunks > 1) issue_chunk_loads(sm, &bar_full[1], &tmQ, &tmK, &tmV, 1, bos + kChunk, hq, h);
  }
  // Initial state -> TMEM (S^T: lane = value index, columns = key index).
  {
    float x[32];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int k0 = 64 * chalf + 32 * part;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        x[j] = a.initial_state ? a.initial_state[st_off + (size_t)(k0 + j) * DV + row] : 0.f;
      tmem_st32(tbase + lane_off + COL_S + k0, x);
    }
  }
  // gates of chunk 0 (warp 0), later prefetched one chunk ahead
  float gq[2], bq[2];
  if (warp == 0) load_gates(a, bos, min(kChunk, eos - bos), h, lane, gq, bq);

  const uint32_t sbase = smem_u32(sm);
  uint32_t mma_parity = 0;
  int issued = nchunks > 1 ? 2 : 1;  // chunks whose loads have been issued
  bool failed = false;

  // Wait for the tensor core's most recent commit (all threads), bounded.
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(bar_mma, mma_parity, kWaitLimitNs);
    mma_parity ^= 1u;
    return __syncthreads_or(!ok) == 0;
  };

  int c = 0;
  for (; c < nchunks; ++c) {
    const int s = c & 1;
    const int t0 = bos + c * kChunk;
    const int L = min(kChunk, eos - t0);
    uint8_t* qk = sm + OFF_QK + s * QK_STAGE;
    const uint32_t qk_a = sbase + OFF_QK + s * QK_STAGE;
    const uint32_t v_a = sbase + OFF_V + s * V_STAGE;

    // ---- gates: in-chunk cumulative log-decay and beta; prefetch the next chunk's
    if (warp == 0) {
      float g0 = gq[0], g1 = gq[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x0 = __shfl_up_sync(0xffffffffu, g0, o);
        const float x1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) { g0 += x0; g1 += x1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      sG[lane] = g0; sG[lane + 32] = g1;
      sBeta[lane] = bq[0]; sBeta[lane + 32] = bq[1];
      if (c + 1 < nchunks) load_gates(a, t0 + kChunk, min(kChunk, eos - t0 - kChunk), h, lane, gq, bq);
    }
    // ---- this chunk's Q, K, V tiles
    {
      const bool ok = mbar_wait(&bar_full[s], (uint32_t)(c >> 1) & 1u, kWaitLimitNs);
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // ---- S (entry state) -> bf16 A operand S^T [dv rows][dk]; S <- exp(G_last) S in TMEM
    {
      const float dl = __expf(sG[L - 1]);
      uint8_t* dst = sm + OFF_S + chalf * 16384;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float x[32];
        const uint32_t col = COL_S + 64 * chalf + 32 * part;
        tmem_ld32(tbase + lane_off + col, x);
#pragma unroll
        for (int m = 0; m < 4; ++m) store_bf16x8(dst + sw128_offset(row, 32 * part + 8 * m), &x[8 * m]);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] *= dl;
        tmem_st32(tbase + lane_off + col, x);
      }
    }
    // ---- inverse L2 norms of the chunk's q and k rows (4 threads per row)
    {
      const int r = tid >> 2, part = tid & 3;
      const uint8_t* qrow = qk + (part >> 1) * 16384 + r * 128 + (part & 1) * 64;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        sq += sumsq_bf16x8(*reinterpret_cast<const uint4*>(qrow + 16 * m));
        sk += sumsq_bf16x8(*reinterpret_cast<const uint4*>(qrow + 8192 + 16 * m));
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 2);
      if (part == 0) {
        sRq[r] = a.use_qk_l2norm ? 1.0f / sqrtf(sq + kL2Eps) : 1.0f;
        sRk[r] = a.use_qk_l2norm ? 1.0f / sqrtf(sk + kL2Eps) : 1.0f;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA: D1 = [Q;K] K^T, O1 = S^T Q^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id1 = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tbase + COL_D1, sdesc_sw128(qk_a + off, 16, 1024),
                 sdesc_sw128(qk_a + off + 8192, 16, 1024), id1, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tbase + COL_O1, sdesc_sw128(sbase + OFF_S + off, 16, 1024),
                 sdesc_sw128(qk_a + off, 16, 1024), id1, ks > 0);
      }
      mma_commit(bar_mma);
    }
    // per-token scalars while the tensor core works
    if (tid < kChunk) {
      const float gl = sG[L - 1];
      const float gt = sG[tid];
      const float et = __expf(gt);
      sSw[tid] = sBeta[tid] * et * sRk[tid];
      sDl[tid] = __expf(gl - gt) * sRk[tid];
      sQs[tid] = a.scale * et * sRq[tid];
    }
    if (!wait_mma()) { failed = true; break; }
    tc_fence_after();

    // ---- P (bf16, rows 0-63 of D1) and A (fp32, rows 64-127 of D1)
    {
      float x[32];
      tmem_ld32(tbase + lane_off + COL_D1 + 32 * chalf, x);
      const int j0 = 32 * chalf;
      if (quad < 2) {
        const int i = row;
        const float gi = sG[i], ri = (i < L) ? sRq[i] : 0.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = j0 + jj;
          x[jj] = (j <= i) ? ri * sRk[j] * x[jj] * __expf(gi - sG[j]) : 0.f;
        }
        uint8_t* dst = sm + OFF_P;
#pragma unroll
        for (int m = 0; m < 4; ++m) store_bf16x8(dst + sw128_offset(i, j0 + 8 * m), &x[8 * m]);
      } else {
        const int i = row - 64;
        const float gi = sG[i], bi = sBeta[i] * sRk[i];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = j0 + jj;
          x[jj] = (j < i) ? bi * sRk[j] * x[jj] * __expf(gi - sG[j]) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m)
          *reinterpret_cast<float4*>(&sA[a_idx(i, j0 + 4 * m)]) =
              make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- T = (I + A)^{-1}, step 1: the four 16 x 16 diagonal blocks (one column per thread)
    if (tid < 64) {
      const int b = tid >> 4, jj = tid & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == jj) ? 1.f : 0.f;
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < i; ++k) acc += sA[a_idx(16 * b + i, 16 * b + k)] * x[k];
        if (i > jj) x[i] = -acc;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) sTd[(b * 16 + i) * 16 + jj] = x[i];
    }
    __syncthreads();
    // ---- step 2: each column of T in registers (4 threads per column, replicated);
    //      block row b from the rows above it: T[b, c] = -T_bb A[b, :16b] T[:16b, c]
    {
      const int col = tid >> 2, q4 = tid & 3;
      const int bc = col >> 4;                 // warp-uniform (a warp holds 8 columns)
      float x[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) x[i] = 0.f;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        if (bb == bc) {
#pragma unroll
          for (int i = 0; i < 16; ++i) x[16 * bb + i] = sTd[(bb * 16 + i) * 16 + (col & 15)];
        }
      }
#pragma unroll
      for (int b = 1; b < 4; ++b) {
        if (b > bc) {
          // y[rr] = sum_k A[16b + r][k] x[k] for this thread's rows r = 4 rr + q4
          float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int g = 0; g < 4 * b; ++g) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int r = 16 * b + 4 * rr + q4;
              const float4 a4 = *reinterpret_cast<const float4*>(&sA[a_idx(r, 4 * g)]);
              y[rr] += a4.x * x[4 * g] + a4.y * x[4 * g + 1] + a4.z * x[4 * g + 2] +
                       a4.w * x[4 * g + 3];
            }
          }
          float ys[16];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int src = 0; src < 4; ++src)
              ys[4 * rr + src] = __shfl_sync(0xffffffffu, y[rr], (lane & ~3) | src);
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m <= r; ++m) acc += sTd[(b * 16 + r) * 16 + m] * ys[m];
            x[16 * b + r] = -acc;
          }
        }
      }
      // (T diag(beta exp(G) r_k))^T and (T diag(beta))^T: row `col`, this thread's 16 entries
      const float sw = sSw[col], sb = sBeta[col];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        if (qq == q4) {
          float w[16], u[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) { w[i] = x[16 * qq + i] * sw; u[i] = x[16 * qq + i] * sb; }
          store_bf16x8(sm + OFF_TW + sw128_offset(col, 16 * qq), w);
          store_bf16x8(sm + OFF_TW + sw128_offset(col, 16 * qq + 8), w + 8);
          store_bf16x8(sm + OFF_TU + sw128_offset(col, 16 * qq), u);
          store_bf16x8(sm + OFF_TU + sw128_offset(col, 16 * qq + 8), u + 8);
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA: W^T = K^T Tw^T, U^T = V^T Tu^T   (all operands MN-major)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_W, sdesc_sw128(qk_a + 8192 + ks * 2048, 16384, 1024),
                 sdesc_sw128(sbase + OFF_TW + ks * 2048, 8192, 1024), id, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_U, sdesc_sw128(v_a + ks * 2048, 8192, 1024),
                 sdesc_sw128(sbase + OFF_TU + ks * 2048, 8192, 1024), id, ks > 0);
      }
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { failed = true; break; }
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
    __syncthreads();

    // ---- MMA: U'^T = U^T + S^T (-W^T)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_bf16(tbase + COL_U,
                 sdesc_sw128(sbase + OFF_S + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                 sdesc_sw128(sbase + OFF_W + ks * 2048, 8192, 1024), id, 1);
      }
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { failed = true; break; }
    tc_fence_after();

    // ---- U'^T and (U' exp(G_last - G) r_k)^T -> bf16 K-major A operands [dv rows][tokens]
    {
      float x[32], y[32];
      tmem_ld32(tbase + lane_off + COL_U + 32 * chalf, x);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) y[jj] = x[jj] * sDl[32 * chalf + jj];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        store_bf16x8(sm + OFF_U + sw128_offset(row, 32 * chalf + 8 * m), &x[8 * m]);
        store_bf16x8(sm + OFF_UT + sw128_offset(row, 32 * chalf + 8 * m), &y[8 * m]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA: O2 = U'^T P^T, S^T += Ut^T K
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id6 = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_O2, sdesc_sw128(sbase + OFF_U + ks * 32, 16, 1024),
                 sdesc_sw128(sbase + OFF_P + ks * 32, 16, 1024), id6, ks > 0);
      }
      const uint32_t id7 = idesc_bf16(128, 128, false, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_S, sdesc_sw128(sbase + OFF_UT + ks * 32, 16, 1024),
                 sdesc_sw128(qk_a + 8192 + ks * 2048, 16384, 1024), id7, 1);
      }
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { failed = true; break; }
    tc_fence_after();

    // Stage s is free again: load chunk c + 2 into it.
    if (tid == 0 && c + 2 < nchunks) {
      fence_proxy_async_smem();
      issue_chunk_loads(sm, &bar_full[s], &tmQ, &tmK, &tmV, s, t0 + 2 * kChunk, hq, h);
      ++issued;
    }

    // ---- o = scale (exp(G) r_q O1 + O2)
    {
      float x[32], y[32];
      tmem_ld32(tbase + lane_off + COL_O1 + 32 * chalf, x);
      tmem_ld32(tbase + lane_off + COL_O2 + 32 * chalf, y);
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int t = 32 * chalf + jj;
        if (t < L)
          o[((size_t)(t0 + t) * a.Hv + h) * DV + row] =
              __float2bfloat16_rn(sQs[t] * x[jj] + a.scale * y[jj]);
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (failed) {
    if (tid == 0) report(a.dev_status, GDN_DEV_TIMEOUT);
    // Drain: bounded waits for the loads issued but not consumed and for the
    // last tensor-core commit, so no copy or MMA is in flight when TMEM is freed.
    for (int cc = c; cc < issued; ++cc) mbar_wait(&bar_full[cc & 1], (uint32_t)(cc >> 1) & 1u, kWaitLimitNs);
    mbar_wait(bar_mma, mma_parity ^ 1u, kWaitLimitNs);
    __syncthreads();
  } else if (a.final_state) {
    tc_fence_after();
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float x[32];
      const int k0 = 64 * chalf + 32 * part;
      tmem_ld32(tbase + lane_off + COL_S + k0, x);
#pragma unroll
      for (int j = 0; j < 32; ++j) a.final_state[st_off + (size_t)(k0 + j) * DV + row] = x[j];
    }
  }
  tc_fence_before();
  __syncthreads();
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
  CUtensorMap mq, mk, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (T_total > 0) {
    if (!encode_map(&mq, a.q, a.Hqk, T_total) || !encode_map(&mk, a.k, a.Hqk, T_total) ||
        !encode_map(&mv, a.v, a.Hv, T_total))
      return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)a.num_seqs * a.Hv;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  chunk_tc_kernel<<<(unsigned)blocks, kTcThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace gdn
