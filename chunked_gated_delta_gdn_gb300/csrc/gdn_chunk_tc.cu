// gdn_chunk_tc.cu -- fused chunkwise gated delta rule on the tcgen05 tensor cores.
//
// One CTA per (sequence, value head), bf16 I/O, K = V = 128, chunk 64.  TMA
// brings each chunk's Q, K, V tiles into 128-byte-swizzled shared memory, every
// contraction is a tcgen05.mma with its fp32 accumulator in TMEM, and the K x V
// fp32 state lives in TMEM for the whole sequence.  Per chunk (G = in-chunk
// cumulative log-decay, r_q / r_k = inverse L2 norms, S = state entering the chunk):
//
//   D1  = [Q; K] [Q; K]^T                  M=128 N=128 K=128   (Q K^T, K K^T; the
//                                                               diagonal gives |q|^2, |k|^2)
//   P   = scale r_q r_k^T * Q K^T * exp(G_i - G_j) * [j <= i]    (bf16, smem)
//   A   = beta r_k r_k^T * K K^T * exp(G_i - G_j) * [j < i]      (fp32, smem)
//   T   = (I + A)^{-1}                     with 16 x 16 diagonal blocks D_b = (I + A_bb)^-1 and
//                                           L = D A_off (block strictly lower):
//                                           T = (I - L + L^2 - L^3) D      (fp32, CUDA cores)
//   U^T = V^T Tu^T, Tu = T diag(beta)      M=128 N=64  K=64
//   [O1 | Y] = S^T [Q; K]^T                M=128 N=128 K=128   (O1 = S^T Q^T, Y = S^T K^T)
//   U'^T = U^T - Y Tw^T, Tw = T diag(beta exp(G) r_k)
//                                          M=128 N=64  K=64    (accumulates on U^T; this is
//                                                               U - W S with W = Tw K; -Y is
//                                                               read from TMEM as bf16)
//   O2 = U'^T P^T                          M=128 N=64  K=64
//   S^T += U'^T K~                         M=128 N=128 K=64    (K~ = diag(exp(G_last - G) r_k) K,
//                                                               S^T decayed by exp(G_last) before)
//   o   = scale exp(G) r_q * O1 + O2
//
// Every product is oriented so M = 128 (value or key features on the TMEM
// lanes, tokens on the columns).  The CTA is warp-specialised: a prep group
// (warps 0-7) builds everything that does not depend on the state -- norms,
// D1, P, A, T -- for chunk c + 1 while a state group (warps 8-11) runs the
// rest of chunk c (the U product, O1 and S K^T, U', the state update, the output);
// they hand chunks over through mbarriers, double-buffering P, the per-token
// vectors and the TMA stages.  These are the chunkwise (WY / UT transform)
// equations of the gated delta rule with the chunking of the inference kernels
// ("Megatron-Core API: core.ssm.gated_delta_product", ssm_inference_chunk_size:
// a fixed 64) and the argument set of torch_chunk_gated_delta_rule ("Megatron-
// Core API: core.ssm.gated_delta_net.gdn").  Every wait is bounded; a timeout
// sets GDN_DEV_TIMEOUT, drains, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"
#include "gdn_tc_prep.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kStateThreads = 128;  // warps 8-11
constexpr int kTcThreads = kPrepThreads + kStateThreads;
constexpr int kBarPrep = 1, kBarState = 2;   // named barrier ids
constexpr int DK = kTcDK, DV = kTcDV;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Shared memory map (bytes from a 1024-byte-aligned base).
constexpr uint32_t OFF_QK = 0;          // 2 stages x 32 KB: [dk half][Q rows 0-63 | K rows 64-127][128 B]
constexpr uint32_t QK_STAGE = 32768;
constexpr uint32_t OFF_V = 65536;       // 2 stages x 16 KB: [dv half][64 tokens][128 B]
constexpr uint32_t V_STAGE = 16384;
constexpr uint32_t OFF_S = 98304;       // the bf16 output tile staged for its TMA store (16 KB)
constexpr uint32_t OFF_RT = 114688;     // record mode: T^T and P staged for one bulk copy (16 KB)
constexpr uint32_t OFF_KT = 131072;     // K~^T: the K rows scaled by exp(G_last - G_t) r_k[t],
                                        // transposed, K-major [128 dk rows][64 tokens] (the B
                                        // operand of the state update; the 8 KB below are free)
constexpr uint32_t OFF_A = 147456;      // fp32 A [64][64], 16-byte-group swizzled; the solve
                                        // overwrites its strictly-lower blocks with those of T
constexpr uint32_t OFF_P = 163840;      // 2 x P, K-major B [64 i][64 j]
constexpr uint32_t OFF_REC = 180224;    // (forward mode: the second Tw / Tu buffer)    // record mode: staging of the entry-state tile's second
                                        // half, then of the U' tile (16 KB)
constexpr uint32_t OFF_TW = 196608;     // (T diag(beta exp(G) r_k))^T, MN-major B [64 j][64 i]
constexpr uint32_t OFF_TU = 204800;     // (T diag(beta))^T, MN-major B
constexpr uint32_t OFF_VEC = 212992;    // 2 x per-token fp32 vectors [8][64]
constexpr uint32_t OFF_TD = OFF_VEC + 2 * 4 * VEC_FLOATS;  // diagonal blocks of T
constexpr uint32_t OFF_BAR = OFF_TD + kTdBytes;
constexpr uint32_t SMEM_USED = OFF_BAR + 256;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base


// TMEM columns (fp32, 128 lanes).  COL_S holds S^T for the whole sequence.  Three products
// read their A operand from TMEM as bf16 (two per 32-bit column): S^T (in the O2 columns,
// until O2 is written), -Y (in its own first 32 columns) and U' (in the first 32 of U's).
constexpr uint32_t COL_D1 = 0 /* 128 */, COL_U = 128, COL_O1 = 192, COL_Y = 256 /* O1 | Y adjacent */,
                   COL_O2 = 320, COL_S = 384, TMEM_COLS = 512;

// mbarriers (8 bytes each) at OFF_BAR.
enum {
  B_FULL = 0,       // [2] TMA stage landed
  B_MMA_P = 2,      // prep group's D1 commits
  B_MMA_S = 3,      // state group's MMA commits
  B_READY = 4,      // [2] prep -> state: chunk ready (vectors, P, Tw / Tu in shared memory)
  B_WU = 6,         // [2 by buffer, see B_WU1] state -> prep: the MMAs reading Tw / Tu are done
  B_P_FREE = 7,     // [2] state -> prep: the O2 product has read P (its buffer free)
  B_VEC_FREE = 9,   // [2] state -> prep: chunk finished (per-token vectors free)
  B_WU1 = 11,       // forward mode: as B_WU, for the second Tw / Tu buffer
  B_COUNT = 12
};
constexpr uint32_t OFF_FLAG = OFF_BAR + 8 * B_COUNT;      // int: a group timed out
constexpr uint32_t OFF_TSLOT = OFF_FLAG + 8;              // TMEM base address

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_TSLOT + 4 <= SMEM_USED, "barrier block");
static_assert(QK_STAGE == kQkStageBytes && V_STAGE == kVStageBytes, "stage bytes");
static_assert(OFF_P + 2 * 8192 <= OFF_REC && OFF_REC + 16384 <= OFF_TW, "record staging");
static_assert(OFF_S + 16384 <= OFF_RT && OFF_RT + 16384 <= OFF_KT, "record staging of T^T, P");

// Stage timestamps for the per-chunk cycle budget (a diagnostic build, -DGDN_CHUNK_STAMPS):
// the leader of each group records clock64 at the stage boundaries of chunks 32 .. 95 in the
// first and the last CTA of a launch, in either mode (gdn_chunk_stamps_read copies them out).
// Without the define the stamps compile to nothing.
#ifdef GDN_CHUNK_STAMPS
__device__ unsigned long long g_chunk_stamps[2][2][64][16];
#define GDN_STAMP(grp, p)                                                                       \
  do {                                                                                          \
    const int stamp_cta_ = blockIdx.x == 0 ? 0 : (blockIdx.x == gridDim.x - 1 ? 1 : -1);        \
    if (leader && stamp_cta_ >= 0 && c >= 32 && c < 96)                                         \
      g_chunk_stamps[stamp_cta_][grp][c - 32][p] = clock64();                                   \
  } while (0)
#else
#define GDN_STAMP(grp, p) \
  do {                    \
  } while (0)
#endif

// The Tw / Tu operands of chunk c: two buffers by chunk parity, the second in space the mode
// does not use otherwise (forward mode: the record staging; record mode, which writes no
// output: the P buffers).
template <bool kRecord>
__device__ __forceinline__ uint32_t tw_off(int c) { return (c & 1) ? (kRecord ? OFF_P : OFF_REC) : OFF_TW; }
template <bool kRecord>
__device__ __forceinline__ uint32_t tu_off(int c) {
  return (c & 1) ? (kRecord ? OFF_P + 8192 : OFF_REC + 8192) : OFF_TU;
}
__device__ __forceinline__ int wu_bar(int c) { return (c & 1) ? B_WU1 : B_WU; }

// =================================================================== prep group
// Warps 0-7.  For each chunk: D1 = [Q;K][Q;K]^T, gates, norms (from the diagonal of
// D1), P, A, and T = (I+A)^{-1} as bf16 Tw / Tu operands; then hands the chunk to the
// state group and moves on.
template <bool kRecord>
__device__ void prep_group(const ChunkArgs& a, uint8_t* sm, uint32_t tbase, int bos, int eos,
                           int nchunks, int h, long long rec0) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  int* flag = reinterpret_cast<int*>(sm + OFF_FLAG);
  float* sA = reinterpret_cast<float*>(sm + OFF_A);
  float* sTd = reinterpret_cast<float*>(sm + OFF_TD);
  const bool leader = (tid == 0);
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  constexpr int kGateWarp = 1;   // not the leader's warp: gates overlap the MMA issue
  float gq[2], bq[2];
  if (warp == kGateWarp) prefetch_gates(a, bos, h, lane, T_total, gq, bq);
  const bool fused = a.gates.mode == kGatesFused;
  const float expA = fused ? expf(a.gates.A_log[h]) : 0.f;
  const float dtb = fused ? a.gates.dt_bias[h] : 0.f;

  for (int c = 0; c < nchunks; ++c) {
    const int s = c & 1;
    const int t0 = bos + c * kChunk;
    const int L = min(kChunk, eos - t0);
    float* vec = reinterpret_cast<float*>(sm + OFF_VEC) + s * VEC_FLOATS;
    const uint32_t qk_a = sbase + OFF_QK + s * QK_STAGE;
    GDN_STAMP(0, 0);

    // ---- per-token vectors of chunk c - 2 released; this chunk's tiles landed
    // (one thread polls each mbarrier; the rest of the group sleeps in the named barrier)
    bool ok = true;
    if (leader) {
      if (c >= 2) ok = mbar_wait(&bars[B_VEC_FREE + s], (uint32_t)((c - 2) >> 1) & 1u, kWaitLimitNs);
      ok = ok && mbar_wait(&bars[B_FULL + s], (uint32_t)(c >> 1) & 1u, kWaitLimitNs);
    }
    if (group_sync_or(kBarPrep, kPrepThreads, !ok || flag_set(flag))) { if (leader) set_flag(flag); return; }
    GDN_STAMP(0, 1);

    // ---- MMA: D1 = [Q;K][Q;K]^T.  (Issuing it earlier, during the previous chunk, measured
    //      slower: an MMA issue into the busy tensor pipe stalls the issuing thread.)
    if (leader) {
      tc_fence_after();
      issue_d1(tbase + COL_D1, qk_a, &bars[B_MMA_P]);
      GDN_STAMP(0, 2);
    }
    // ---- gates: in-chunk cumulative log-decay and beta; prefetch the next chunk's
    if (warp == kGateWarp)
      gates_step(a, vec, gq, bq, L, lane, fused, expA, dtb, c + 1 < nchunks, t0 + kChunk, h, T_total);
    if (leader) {
      ok = mbar_wait(&bars[B_MMA_P], (uint32_t)c & 1u, kWaitLimitNs);   // one D1 commit per chunk
      if (kRecord) tma_store_wait_read();   // the previous chunk's T^T, P have left the staging
      if (!kRecord && c >= 2) ok = ok && mbar_wait(&bars[B_P_FREE + s], (uint32_t)((c - 2) >> 1) & 1u, kWaitLimitNs);
    }
    if (group_sync_or(kBarPrep, kPrepThreads, !ok || flag_set(flag))) { if (leader) set_flag(flag); return; }
    tc_fence_after();
    GDN_STAMP(0, 3);

    // ---- norms, P (to this chunk's P buffer; in record mode to the staging for the backward)
    //      and A from D1
    norms_p_a<kBarPrep>(a, tbase + COL_D1, vec, sA, kRecord ? sm + OFF_RT + 8192 : sm + OFF_P + s * 8192, L);
    tc_fence_before();
    GDN_STAMP(0, 4);
    // Tw, Tu free: this buffer released by chunk c - 2
    if (leader && c >= 2) ok = mbar_wait(&bars[wu_bar(c)], (uint32_t)((c - 2) >> 1) & 1u, kWaitLimitNs);
    if (group_sync_or(kBarPrep, kPrepThreads, !ok || flag_set(flag))) { if (leader) set_flag(flag); return; }
    if (kRecord && tid < 64) {   // the reverse pass's per-token vectors (zero past the chunk end)
      const int i = tid;
      const bool in = i < L;
      float* rv = a.rec_vec + ((size_t)(rec0 + c) * a.Hv + h) * kRvFloats;
      rv[kRvCq + i] = in ? vec[VEC_QS + i] : 0.f;
      rv[kRvW + i] = in ? vec[VEC_DL + i] : 0.f;
      rv[kRvF + i] = in ? -vec[VEC_SW + i] : 0.f;
      rv[kRvBeta + i] = in ? vec[VEC_BETA + i] : 0.f;
      if (i == 0) rv[kRvGl] = ex2(vec[VEC_G + L - 1]);
    }

    // ---- T = (I + A)^{-1} as the Tw / Tu operands
    GDN_STAMP(0, 5);
    solve_t<kBarPrep>(sA, sTd, vec, sm + tw_off<kRecord>(c), sm + tu_off<kRecord>(c),
                      kRecord ? sm + OFF_RT : nullptr);
    fence_proxy_async_smem();
    group_sync(kBarPrep, kPrepThreads);
    if (kRecord && leader) {   // T^T and P of the chunk for the backward's reverse pass
      bulk_store(reinterpret_cast<uint8_t*>(a.rec_tp) + ((size_t)(rec0 + c) * a.Hv + h) * 16384,
                 sm + OFF_RT, 16384);
      tma_store_commit();
    }

    // ---- hand chunk c to the state group (which runs the W / U products) and move on
    GDN_STAMP(0, 6);
    if (leader) mbar_arrive(&bars[B_READY + s]);
  }
}

// Cold paths of the state group, kept out of line so the per-chunk code stays compact.
__device__ __noinline__ void load_state_tmem(uint32_t taddr, int row, const float* init, bool identity) {
#pragma unroll 1
  for (int part = 0; part < 4; ++part) {
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      x[j] = identity ? (32 * part + j == row ? 1.f : 0.f)
                      : (init ? init[(size_t)(32 * part + j) * DV + row] : 0.f);
    tmem_st32(taddr + 32 * part, x);
  }
}

__device__ __noinline__ void store_state_tmem(uint32_t taddr, int row, float* fin, bool transposed) {
#pragma unroll 1
  for (int part = 0; part < 4; ++part) {
    float x[32];
    tmem_ld32(taddr + 32 * part, x);
    if (transposed) {   // [V][K]: this thread's row, 32 consecutive floats
      float4* dst = reinterpret_cast<float4*>(fin + (size_t)row * DK + 32 * part);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) fin[(size_t)(32 * part + j) * DV + row] = x[j];
    }
  }
}

// The last, partial chunk of a sequence: o rows t < L written one by one.
__device__ __noinline__ void store_partial_output(__nv_bfloat16* out, uint32_t o1, uint32_t o2,
                                                  const float* qs, int L, size_t row0, size_t stride) {
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    float x[32], y[32];
    tmem_ld32(o1 + 32 * half, x);
    tmem_ld32(o2 + 32 * half, y);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int t = 32 * half + jj;
      if (t < L) out[row0 + (size_t)t * stride] = __float2bfloat16_rn(fmaf(qs[t], x[jj], y[jj]));
    }
  }
}

// =================================================================== state group
// Warps 8-11.  For each chunk: U^T = V^T Tu^T, S -> bf16 operand and decay of the TMEM
// state, [O1 | Y] = S^T [Q; K]^T, U' = U - Y Tw^T, O2 = U'^T P^T, S^T += U'^T K~, output.
template <bool kRecord>
__device__ void state_group(const ChunkArgs& a, uint8_t* sm, uint32_t tbase, int bos, int eos,
                            int nchunks, int h, int hq, float* fin, int uflags, long long rec0,
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
    float* vec = reinterpret_cast<float*>(sm + OFF_VEC) + s * VEC_FLOATS;
    const uint32_t qk_a = sbase + OFF_QK + s * QK_STAGE;
    const uint32_t v_a = sbase + OFF_V + s * V_STAGE;
    GDN_STAMP(1, 0);

    bool ok = true;
    if (leader) {
      ok = mbar_wait(&bars[B_READY + s], (uint32_t)(c >> 1) & 1u, kWaitLimitNs);
      // the previous chunk's staged tiles (output; in record mode also U') have been read
      tma_store_wait_read();
    }
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    tc_fence_after();
    GDN_STAMP(1, 1);

    // ---- MMA: U^T = V^T Tu^T (operands MN-major), running while the state is converted
    if (leader) {
      const uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tbase + COL_U, sdesc_sw128(v_a + ks * 2048, 8192, 1024),
                 sdesc_sw128(sbase + tu_off<kRecord>(c) + ks * 2048, 8192, 1024), id, ks > 0);
      }
      GDN_STAMP(1, 2);
    }
    // ---- record mode: the entry state as a bf16 tile, rows dk, 64 dv per 128-byte row in two
    //      16 KB halves, 128-byte swizzled (element (dk, dv) at (dv / 64) 16384 + dk 128 +
    //      ((dv % 64 / 8) xor (dk % 8)) 16 + (dv % 8) 2): 16x256b TMEM loads give each thread the
    //      stmatrix .trans fragment (as in the output epilogue), the halves are staged at OFF_S
    //      and OFF_REC and leave by two bulk copies
    if (kRecord) {
      const int mblk = lane >> 3, rr = lane & 7;
      const int d0 = 32 * wq + 8 * mblk;
      const uint32_t st_base = sbase + (d0 < 64 ? OFF_S : OFF_REC) + rr * 128 +
                               ((((d0 & 63) >> 3) ^ rr) << 4);
#pragma unroll 1
      for (int pass = 0; pass < 4; ++pass) {   // dk 32 pass .. 32 pass + 31
        uint32_t a0[16], a1[16];
        tmem_ld16x256b_x4(tbase + lane_off + COL_S + 32 * pass, a0);                 // dv 0-15
        tmem_ld16x256b_x4(tbase + lane_off + (16u << 16) + COL_S + 32 * pass, a1);   // dv 16-31
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // dk group 4 pass + j
          uint32_t f[4];
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const uint32_t* x = (mm >> 1) ? a1 : a0;
            const int k = 4 * j + 2 * (mm & 1);
            __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(x[k]), __uint_as_float(x[k + 1]));
            f[mm] = *reinterpret_cast<uint32_t*>(&p);
          }
          stmatrix_x4_trans(st_base + (4 * pass + j) * 1024, f);
        }
      }
      fence_proxy_async_smem();
      group_sync(kBarState, kStateThreads);
      if (leader) {
        uint8_t* g = reinterpret_cast<uint8_t*>(a.rec_states +
                                                ((size_t)(rec0 + c) * a.Hv + h) * (size_t)(DK * DV / 2));
        bulk_store(g, sm + OFF_S, 16384);
        bulk_store(g + 16384, sm + OFF_REC, 16384);
        tma_store_commit();
      }
    }
    // ---- S (entry state) -> bf16 S^T in the O2 columns (the next product's A operand);
    //      S <- exp(G_last) S in TMEM
    {
      const float dl = ex2(vec[VEC_G + L - 1]);
#pragma unroll 1
      for (int pair = 0; pair < 2; ++pair) {
        float pk[32];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          float x[32];
          const uint32_t col = COL_S + 32 * (2 * pair + sub);
          tmem_ld32(tbase + lane_off + col, x);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pk[16 * sub + jj] = __uint_as_float(pack_bf16x2(x[2 * jj], x[2 * jj + 1]));
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] *= dl;
          tmem_st32(tbase + lane_off + col, x);
        }
        tmem_st32(tbase + lane_off + COL_O2 + 32 * pair, pk);
      }
    }
    tc_fence_before();
    group_sync(kBarState, kStateThreads);
    GDN_STAMP(1, 3);

    // ---- MMA: [O1 | Y] = S^T [Q; K]^T, one N = 128 product over the stage as loaded (A, the
    //      bf16 S^T, from TMEM); record mode, without output: Y = S^T K^T alone (N = 64)
    if (leader) {
      tc_fence_after();
      const uint32_t id5 = kRecord ? idesc_bf16(128, 64, false, false) : idesc_bf16(128, 128, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32 + (kRecord ? 8192 : 0);
        mma_bf16_ta(tbase + (kRecord ? COL_Y : COL_O1), tbase + COL_O2 + 8 * ks,
                    sdesc_sw128(qk_a + off, 16, 1024), id5, ks > 0);
      }
      mma_commit(&bars[B_MMA_S]);
      GDN_STAMP(1, 4);
    }
    // ---- while [O1 | Y] runs: K~^T built from the stage's K rows,
    //      scaled by exp(G_last - G_t) r_k[t] and transposed in 8 x 8 blocks (ldmatrix,
    //      stmatrix .trans); warp wq takes tokens 16 wq .. 16 wq + 15.  Then the stage is free.
    {
      const int mi = lane >> 3, rr = lane & 7;   // matrix this lane addresses, row within it
      const int tg = 2 * wq + (mi & 1);          // its token group (8 tokens)
      const uint32_t kst = sbase + OFF_QK + s * QK_STAGE + 8192;
      // fragment register m holds token 8 (2 wq + (m & 1)) + lane / 4
      const float dl0 = vec[VEC_DL + 16 * wq + (lane >> 2)];
      const float dl1 = vec[VEC_DL + 16 * wq + 8 + (lane >> 2)];
#pragma unroll 2
      for (int it = 0; it < 8; ++it) {
        const int dg = 2 * it + (mi >> 1);       // dk group of the matrix this lane addresses
        const int tok = 8 * tg + rr, dk = 8 * dg;
        uint32_t f[4];
        ldmatrix_x4(kst + (dk >> 6) * 16384 + tok * 128 + ((((dk & 63) >> 3) ^ (tok & 7)) << 4), f);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162*>(&f[m]);
          const float2 x2 = __bfloat1622float2(b2);
          const float d = (m & 1) ? dl1 : dl0;
          b2 = __floats2bfloat162_rn(x2.x * d, x2.y * d);
          f[m] = *reinterpret_cast<uint32_t*>(&b2);
        }
        const int dkr = 8 * dg + rr;             // K~^T row this lane addresses
        stmatrix_x4_trans(sbase + OFF_KT + dkr * 128 + ((tg ^ (dkr & 7)) << 4), f);
      }
    }
    fence_proxy_async_smem();
    GDN_STAMP(1, 5);
    if (leader) ok = mbar_wait(&bars[B_MMA_S], ps, kWaitLimitNs);
    ps ^= 1u;
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    GDN_STAMP(1, 6);
    // every read of stage s is done (U, D1, [O1 | Y], the K copy): load chunk c + 2 into it
    if (leader) {
      if (c + 2 < nchunks)
        issue_chunk_loads(sm + OFF_QK + s * QK_STAGE, sm + OFF_V + s * V_STAGE, &bars[B_FULL + s], tq, tk,
                          tv, t0 + 2 * kChunk, hq, h, !(uflags & kUnitZeroV));
    }
    tc_fence_after();

    // ---- -Y -> bf16, packed into the first 32 of its own TMEM columns (A operand from TMEM)
    {
      float x[32], y[32], pk[32];
      tmem_ld32(tbase + lane_off + COL_Y, x);
      tmem_ld32(tbase + lane_off + COL_Y + 32, y);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(-x[2 * jj], -x[2 * jj + 1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(-y[2 * jj], -y[2 * jj + 1]);
        pk[jj] = __uint_as_float(*reinterpret_cast<uint32_t*>(&p0));
        pk[16 + jj] = __uint_as_float(*reinterpret_cast<uint32_t*>(&p1));
      }
      tmem_st32(tbase + lane_off + COL_Y, pk);
    }
    tc_fence_before();
    group_sync(kBarState, kStateThreads);
    GDN_STAMP(1, 7);

    // ---- MMA: U'^T = U^T + (-Y) Tw^T (Tw MN-major); then Tw / Tu are free for the prep group
    if (leader) {
      tc_fence_after();
      const uint32_t id4 = idesc_bf16(128, 64, false, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16_ta(tbase + COL_U, tbase + COL_Y + 8 * ks,
                    sdesc_sw128(sbase + tw_off<kRecord>(c) + ks * 2048, 8192, 1024), id4, 1);
      }
      mma_commit(&bars[wu_bar(c)]);
      mma_commit(&bars[B_MMA_S]);
      GDN_STAMP(1, 8);
    }
    if (leader) ok = mbar_wait(&bars[B_MMA_S], ps, kWaitLimitNs);
    ps ^= 1u;
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    tc_fence_after();
    GDN_STAMP(1, 9);

    // ---- record mode: U' as a bf16 tile, rows = the chunk's 64 tokens (zero from L on), 64 dv
    //      per 128-byte row in two 8 KB halves, 128-byte swizzled; staged at OFF_REC once the
    //      entry-state tile has left it, then one bulk copy
    if (kRecord) {
      if (leader) tma_store_wait_read();
      group_sync(kBarState, kStateThreads);
      const int mblk = lane >> 3, rr = lane & 7;
      const int d0 = 32 * wq + 8 * mblk;
      const uint32_t st_base = sbase + OFF_REC + (d0 >> 6) * 8192 + rr * 128 +
                               ((((d0 & 63) >> 3) ^ rr) << 4);
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {   // tokens 32 pass .. 32 pass + 31
        uint32_t a0[16], a1[16];
        tmem_ld16x256b_x4(tbase + lane_off + COL_U + 32 * pass, a0);
        tmem_ld16x256b_x4(tbase + lane_off + (16u << 16) + COL_U + 32 * pass, a1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // token group 4 pass + j; this lane's tokens t, t + 1
          const int t = 32 * pass + 8 * j + 2 * (lane & 3);
          uint32_t f[4];
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const uint32_t* x = (mm >> 1) ? a1 : a0;
            const int k = 4 * j + 2 * (mm & 1);
            __nv_bfloat162 p = __floats2bfloat162_rn(t < L ? __uint_as_float(x[k]) : 0.f,
                                                     t + 1 < L ? __uint_as_float(x[k + 1]) : 0.f);
            f[mm] = *reinterpret_cast<uint32_t*>(&p);
          }
          stmatrix_x4_trans(st_base + (4 * pass + j) * 1024, f);
        }
      }
      fence_proxy_async_smem();
      group_sync(kBarState, kStateThreads);
      if (leader) {
        bulk_store(a.rec_u + ((size_t)(rec0 + c) * a.Hv + h) * (size_t)(kChunk * DV / 2), sm + OFF_REC, 16384);
        tma_store_commit();
      }
    }
    // ---- U'^T -> bf16, packed into the first 32 of its own TMEM columns (A operand)
    {
      float x[32], y[32], pk[32];
      tmem_ld32(tbase + lane_off + COL_U, x);
      tmem_ld32(tbase + lane_off + COL_U + 32, y);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(x[2 * jj], x[2 * jj + 1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(y[2 * jj], y[2 * jj + 1]);
        pk[jj] = __uint_as_float(*reinterpret_cast<uint32_t*>(&p0));
        pk[16 + jj] = __uint_as_float(*reinterpret_cast<uint32_t*>(&p1));
      }
      tmem_st32(tbase + lane_off + COL_U, pk);
    }
    tc_fence_before();
    group_sync(kBarState, kStateThreads);
    GDN_STAMP(1, 10);

    // ---- MMA: O2 = U'^T P^T (from zero; not in record mode) and S^T += U'^T K~ (A, the bf16
    //      U', from TMEM)
    if (leader) {
      tc_fence_after();
      const uint32_t id2 = idesc_bf16(128, 64, false, false), idS = idesc_bf16(128, 128, false, false);
      if (!kRecord) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_ta(tbase + COL_O2, tbase + COL_U + 8 * ks,
                      sdesc_sw128(sbase + OFF_P + s * 8192 + ks * 32, 16, 1024), id2, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ta(tbase + COL_S, tbase + COL_U + 8 * ks,
                    sdesc_sw128(sbase + OFF_KT + ks * 32, 16, 1024), idS, 1);
      mma_commit(&bars[B_MMA_S]);
      GDN_STAMP(1, 11);
    }
    if (leader) ok = mbar_wait(&bars[B_MMA_S], ps, kWaitLimitNs);
    ps ^= 1u;
    if (group_sync_or(kBarState, kStateThreads, !ok || flag_set(flag))) { failed = true; break; }
    tc_fence_after();
    if (!kRecord && leader) mbar_arrive(&bars[B_P_FREE + s]);   // the O2 product has read P
    GDN_STAMP(1, 12);

    // ---- o = scale exp(G) r_q O1 + O2 (P carries scale r_q): a full chunk is staged as a
    //      bf16 tile (two 128-byte-swizzled [64 tokens][64 dv] halves) and written by one
    //      TMA store; the last, partial chunk of a sequence is stored row by row (neither for a
    //      unit that writes no output, nor in record mode)
    if (kRecord || (uflags & kUnitNoOut)) {
    } else if (L == kChunk) {
      // 16x256b loads hand each thread dv (t/4, t/4 + 8 of a 16-lane half) x tokens
      // (2 (t%4), +1 of each 8-token group): the fragment of stmatrix .trans, which writes
      // 8 x 8 (token, dv) blocks as 16-byte rows of the swizzled staging tile.  Lane l gives
      // the row address of block l / 8 (dv 8 (l / 8) of this warp's 32) at token l % 8.
      const int mblk = lane >> 3, rr = lane & 7;
      const int d0 = 32 * wq + 8 * mblk;
      const uint32_t st_base = sbase + OFF_S + (d0 >> 6) * 8192 + rr * 128 +
                               ((((d0 & 63) >> 3) ^ rr) << 4);
      const float* qs = vec + VEC_QS + 2 * (lane & 3);   // scale r_q exp(G): factor of O1
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {   // tokens 32 pass .. 32 pass + 31
        uint32_t a0[16], a1[16], b0[16], b1[16];
        tmem_ld16x256b_x4(tbase + lane_off + COL_O1 + 32 * pass, a0);                  // dv 0-15
        tmem_ld16x256b_x4(tbase + lane_off + (16u << 16) + COL_O1 + 32 * pass, a1);    // dv 16-31
        tmem_ld16x256b_x4(tbase + lane_off + COL_O2 + 32 * pass, b0);
        tmem_ld16x256b_x4(tbase + lane_off + (16u << 16) + COL_O2 + 32 * pass, b1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // token group 4 pass + j
          const float2 q2 = *reinterpret_cast<const float2*>(qs + 8 * (4 * pass + j));
          uint32_t f[4];
          const uint32_t* src[2] = {a0, a1};
          const uint32_t* srb[2] = {b0, b1};
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {   // block mm: dv 8 mm .. 8 mm + 7 of the warp
            const uint32_t* x = src[mm >> 1];
            const uint32_t* y = srb[mm >> 1];
            const int k = 4 * j + 2 * (mm & 1);
            __nv_bfloat162 p = __floats2bfloat162_rn(
                fmaf(q2.x, __uint_as_float(x[k]), __uint_as_float(y[k])),
                fmaf(q2.y, __uint_as_float(x[k + 1]), __uint_as_float(y[k + 1])));
            f[mm] = *reinterpret_cast<uint32_t*>(&p);
          }
          stmatrix_x4_trans(st_base + (4 * pass + j) * 1024, f);
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
      store_partial_output(out, tbase + lane_off + COL_O1, tbase + lane_off + COL_O2, vec + VEC_QS, L,
                           ((size_t)t0 * a.Hv + h) * DV + row, (size_t)a.Hv * DV);
    }
    tc_fence_before();
    group_sync(kBarState, kStateThreads);
    GDN_STAMP(1, 13);
    if (leader) mbar_arrive(&bars[B_VEC_FREE + s]);
  }

  if (leader) tma_store_wait_all();   // output tiles written before the CTA exits
  if (failed) {
    if (leader) {
      set_flag(flag);
      mbar_wait(&bars[B_MMA_S], ps ^ 1u, kWaitLimitNs);   // last commit, if any, has landed
    }
  } else if (fin) {
    tc_fence_after();
    store_state_tmem(tbase + lane_off + COL_S, row, fin, (uflags & kUnitFinT) != 0);
  }
}

template <bool kRecord>
__global__ void __launch_bounds__(kTcThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const ChunkArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  int* flag = reinterpret_cast<int*>(sm + OFF_FLAG);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);

  const int tid = threadIdx.x, warp = tid >> 5;
  int n, h, bos, eos, uflags = 0;
  const float* init;   // entry state [K][V] (NULL: zero)
  float* fin;          // exit state [K][V] (NULL: not written)
  bool padding = false;
  if (a.units) {   // planned launch: the unit table says what this CTA runs
    if ((int)blockIdx.x >= *a.unit_count) return;
    const TcUnit u = a.units[blockIdx.x];
    n = u.n; h = u.h; bos = u.bos; eos = u.eos; uflags = u.flags;
    init = u.init; fin = u.fin;
    if (uflags & kUnitSkip) return;
    padding = (uflags & kUnitPadding) != 0;
  } else {
    h = blockIdx.x % a.Hv; n = blockIdx.x / a.Hv;
    const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
    if (a.cu_seqlens) { bos = a.cu_seqlens[n]; eos = a.cu_seqlens[n + 1]; }
    else { bos = n * a.T; eos = bos + a.T; }
    if (bos < 0 || eos < bos || eos > T_total) {
      if (tid == 0) report(a.dev_status, GDN_DEV_BAD_CU_SEQLENS);
      return;
    }
    int slot = n;
    if (a.state_indices) {
      slot = a.state_indices[n];
      if (slot < 0 || slot >= a.num_slots) {   // padding sequence
        if (slot != -1 && tid == 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
        padding = true;
        slot = 0;
      }
    }
    const size_t st_off = ((size_t)slot * a.Hv + h) * (size_t)(DK * DV);
    init = a.initial_state ? a.initial_state + st_off : nullptr;
    fin = a.final_state ? a.final_state + st_off : nullptr;
  }
  if (padding) {   // padding sequence: zero rows (no output in record mode), no state access
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
    for (int e = tid; !kRecord && e < (eos - bos) * DV; e += kTcThreads) {
      const int t = e / DV, d = e - t * DV;
      o[((size_t)(bos + t) * a.Hv + h) * DV + d] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int hq = h / (a.Hv / a.Hqk);
  const bool identity = (uflags & kUnitIdentity) != 0;
  const int nchunks = (eos - bos + kChunk - 1) / kChunk;
  if (nchunks == 0) {   // empty range: the state passes through unchanged
    if (fin) {
      for (int e = tid; e < DK * DV; e += kTcThreads)
        fin[e] = identity ? ((e / DV == e % DV) ? 1.f : 0.f) : (init ? init[e] : 0.f);
    }
    return;
  }
  const bool load_v = !(uflags & kUnitZeroV);
  if (!load_v) {   // v = 0: both V stages stay zero (no V loads are issued)
    uint4* vz = reinterpret_cast<uint4*>(sm + OFF_V);
    for (int e = tid; e < (int)(2 * V_STAGE / 16); e += kTcThreads) vz[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
      issue_chunk_loads(sm + OFF_QK, sm + OFF_V, &bars[B_FULL + 0], &tmQ, &tmK, &tmV, bos, hq, h, load_v);
      if (nchunks > 1)
        issue_chunk_loads(sm + OFF_QK + QK_STAGE, sm + OFF_V + V_STAGE, &bars[B_FULL + 1], &tmQ, &tmK,
                          &tmV, bos + kChunk, hq, h, load_v);
    }
    prep_group<kRecord>(a, sm, tbase, bos, eos, nchunks, h, kRecord ? a.rec_chunk_off[n] : 0);
    if (kRecord && tid == 0) tma_store_wait_all();   // the staged T^T, P tiles are written
  } else {
    // Initial state -> TMEM (S^T: lane = value index, columns = key index).
    const int row = 32 * ((tid - kPrepThreads) >> 5) + (tid & 31);
    const uint32_t lane_off = (uint32_t)(32 * ((tid - kPrepThreads) >> 5)) << 16;
    load_state_tmem(tbase + lane_off + COL_S, row, init, identity);
    const long long rec0 = kRecord ? a.rec_chunk_off[n] : 0;
    state_group<kRecord>(a, sm, tbase, bos, eos, nchunks, h, hq, fin, uflags, rec0, &tmQ, &tmK, &tmV,
                         &tmO);
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

bool encode_rows_map_bf16(CUtensorMap* m, const void* base, int H, int T_total) {
  return encode_map(m, base, H, T_total);
}

bool chunk_tc_supported(int K, int V, int io_dtype, int beta_dtype) {
  return K == DK && V == DV && io_dtype == GDN_BF16 &&
         (beta_dtype == GDN_BF16 || beta_dtype == GDN_F32);
}

cudaError_t launch_chunk_tc(const ChunkArgs& a) {
  const bool rec = a.rec_states && a.rec_u && a.rec_chunk_off;
  const int T_total = a.cu_seqlens ? a.T : a.B * a.T;
  CUtensorMap mq, mk, mv, mo;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  memset(&mo, 0, sizeof(mo));
  if (T_total > 0) {   // (record mode writes no output: no map for it)
    if (!encode_map(&mq, a.q, a.Hqk, T_total) || !encode_map(&mk, a.k, a.Hqk, T_total) ||
        !encode_map(&mv, a.v, a.Hv, T_total) || (!rec && !encode_map(&mo, a.o, a.Hv, T_total)))
      return cudaErrorInvalidValue;
  }
  // the shared-memory attribute, set once per device and kernel
  static std::atomic<bool> attr_set[2][64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !attr_set[rec][dev].load(std::memory_order_relaxed)) {
    err = rec ? cudaFuncSetAttribute(chunk_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_BYTES)
              : cudaFuncSetAttribute(chunk_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_set[rec][dev].store(true, std::memory_order_relaxed);
  }
  const long long blocks = a.units ? (long long)a.unit_cap : (long long)a.num_seqs * a.Hv;
  if (a.units && rec) return cudaErrorInvalidValue;   // record mode runs whole sequences
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (rec)
    chunk_tc_kernel<true><<<(unsigned)blocks, kTcThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, a);
  else
    chunk_tc_kernel<false><<<(unsigned)blocks, kTcThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, a);
  return cudaGetLastError();
}

}  // namespace gdn

#ifdef GDN_CHUNK_STAMPS
// The stage timestamps of the last forward-mode launch of the stamped build
// ([2 CTAs][prep, state][chunks 32 .. 95][16] clock64 values); returns a cudaError_t.
extern "C" int gdn_chunk_stamps_read(void* host) {
  return (int)cudaMemcpyFromSymbol(host, gdn::g_chunk_stamps, sizeof(gdn::g_chunk_stamps));
}
#endif
