// gdn_decode.cu -- single-token decode on a slot-indexed recurrent-state cache.
//
// One CTA per (request i, value head h).  The CTA reads slot s = batch_indices[i]
// of the fp32 cache once, forms the two reductions r = S^T k and p = S^T q, and
// writes the updated state back once:
//
//   a  = exp(g);  u = beta (v - a r);  o = scale (a p + (k . q) u);
//   S' = a S + k u^T
//
// which is the gated delta rule step (decay, delta-rule write, read-out with the
// updated state) rearranged so the state is streamed exactly once in each
// direction.  Slot -1 is padding: the output row is written as zeros and the
// state is never touched ("Megatron-Core API: core.ssm.gated_delta_product",
// GatedDeltaProductMixer.ssm_decode; the in-kernel skip discussed on "Add GDN
// dynamic inference", review thread).  The kernel is HBM-bound: 2 * K * V * 4
// bytes of state traffic per real (request, head), under 1 FLOP per byte.
//
// With L > 1 the L tokens of a request are applied in order with the state held in
// registers.  In product mode (the Gated Delta Product's decode step, same page) the L
// entries are the n_h writes of one token: the decay goes with the first write, the
// request's single query reads the state after the last, and only that output is written.
#include <atomic>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 256;

// g and beta of element i = request * Hv + h: given, or computed from the raw gate
// features (fused gates).
__device__ __forceinline__ void gate_values(const DecodeArgs& a, size_t i, int h, float* g,
                                            float* beta) {
  if (a.gates.mode == kGatesFused) {
    fused_gates(a.gates, i, h, g, beta);
  } else {
    *g = a.g[i];
    *beta = load_elem(a.beta, i, a.beta_dtype);
  }
}

// Zero the V-vector o[i, h, :] (padding or skipped slot).
__device__ __forceinline__ void zero_output(const DecodeArgs& a, int i, int h) {
  for (int c = threadIdx.x; c < a.V; c += blockDim.x)
    store_elem(a.o, ((size_t)i * a.Hv + h) * a.V + c, 0.0f, a.io_dtype);
}

// Resolve the slot of request i; returns -1 for padding / skipped requests.
__device__ __forceinline__ int resolve_slot(const DecodeArgs& a, int i) {
  const int s = a.batch_indices ? a.batch_indices[i] : i;
  if (s < 0 || s >= a.num_slots) {
    if (s != -1 && threadIdx.x == 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
    return -1;
  }
  return s;
}

// K = V = 128.  256 threads = 8 warps; warp w owns columns [32 (w & 3), +32) and
// rows [64 (w >> 2), +64).  Lane l owns the float4 column group l & 7 and rows
// r0 + (l >> 3) + 4 m, m = 0..15, so every warp-wide load covers four whole
// 512-byte rows (fully coalesced) and each thread keeps 64 state values in
// registers between the read and the write.  Three CTAs per SM (80 registers, a few
// spilled): more state reads in flight while the resident CTAs compute; 3% faster than
// two CTAs at 103 registers.
__global__ void __launch_bounds__(kDecodeThreads, 3) decode128_kernel(const DecodeArgs a) {
  constexpr int K = 128, V = 128;
  const int h = blockIdx.x % a.Hv;
  const int i = blockIdx.x / a.Hv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = resolve_slot(a, i);
  if (s < 0) {
    if (a.product) zero_output(a, i, h);
    else for (int t = 0; t < a.L; ++t) zero_output(a, i * a.L + t, h);
    return;
  }
  const int hq = h / (a.Hv / a.Hqk);
  const int col = 32 * (warp & 3) + 4 * (lane & 7);
  const int row0 = 64 * (warp >> 2) + (lane >> 3);
  float* Sp = a.state + ((size_t)s * a.Hv + h) * (K * V);

  float4 S[16];
#pragma unroll
  for (int m = 0; m < 16; ++m)
    S[m] = __ldcs(reinterpret_cast<const float4*>(Sp + (size_t)(row0 + 4 * m) * V + col));

  __shared__ float sq[K], sk[K];
  __shared__ float wsum[8], wdot[4];
  __shared__ float red[2][2][V];

  for (int t = 0; t < a.L; ++t) {
    const int it = i * a.L + t;   // row of this token in the [n * L, ...] inputs
    if (t > 0) __syncthreads();   // sq / sk / red of the previous token fully consumed
    // q and k: threads 0..127 take q, 128..255 take k; per-vector sums of squares.
    const size_t qk_off = ((size_t)it * a.Hqk + hq) * K;
    const size_t q_off = a.product ? ((size_t)i * a.Hqk + hq) * K : qk_off;
    const float x = tid < K ? load_elem(a.q, q_off + tid, a.io_dtype)
                            : load_elem(a.k, qk_off + tid - K, a.io_dtype);
    const float ss = warp_sum(x * x);
    if (lane == 0) wsum[warp] = ss;
    __syncthreads();
    float rn = 1.0f;
    if (a.use_qk_l2norm) {
      const float tot = tid < K ? wsum[0] + wsum[1] + wsum[2] + wsum[3]
                                : wsum[4] + wsum[5] + wsum[6] + wsum[7];
      rn = 1.0f / sqrtf(tot + kL2Eps);
    }
    if (tid < K) sq[tid] = x * rn; else sk[tid - K] = x * rn;
    __syncthreads();
    if (tid < K) {
      const float d = warp_sum(sq[tid] * sk[tid]);
      if (lane == 0) wdot[warp] = d;
    }

    // Partial r = S^T k and p = S^T q over this thread's 16 rows.
    float4 pr = make_float4(0.f, 0.f, 0.f, 0.f), pq = pr;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float kr = sk[row0 + 4 * m], qr = sq[row0 + 4 * m];
      pr.x += S[m].x * kr; pr.y += S[m].y * kr; pr.z += S[m].z * kr; pr.w += S[m].w * kr;
      pq.x += S[m].x * qr; pq.y += S[m].y * qr; pq.z += S[m].z * qr; pq.w += S[m].w * qr;
    }
    // Reduce over the four row lanes of the warp (lane bits 3 and 4).
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
      pr.x += __shfl_xor_sync(0xffffffffu, pr.x, o); pr.y += __shfl_xor_sync(0xffffffffu, pr.y, o);
      pr.z += __shfl_xor_sync(0xffffffffu, pr.z, o); pr.w += __shfl_xor_sync(0xffffffffu, pr.w, o);
      pq.x += __shfl_xor_sync(0xffffffffu, pq.x, o); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, o);
      pq.z += __shfl_xor_sync(0xffffffffu, pq.z, o); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, o);
    }
    if (lane < 8) {
      *reinterpret_cast<float4*>(&red[warp >> 2][0][col]) = pr;
      *reinterpret_cast<float4*>(&red[warp >> 2][1][col]) = pq;
    }
    __syncthreads();

    const size_t hv_off = (size_t)it * a.Hv + h;
    float gv, bt;
    if (a.product) {   // the token's decay on its first write only
      gv = (t == 0) ? a.g[(size_t)i * a.Hv + h] : 0.f;
      bt = load_elem(a.beta, hv_off, a.beta_dtype);
    } else {
      gate_values(a, hv_off, h, &gv, &bt);
    }
    const float dec = expf(gv);
    const bool write_o = !a.product || t == a.L - 1;
    const size_t o_row = a.product ? (size_t)i * a.Hv + h : hv_off;
    const float kq = wdot[0] + wdot[1] + wdot[2] + wdot[3];
    float u[4], o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float r = red[0][0][col + c] + red[1][0][col + c];
      const float p = red[0][1][col + c] + red[1][1][col + c];
      const float vv = load_elem(a.v, hv_off * V + col + c, a.io_dtype);
      u[c] = bt * (vv - dec * r);
      o[c] = a.scale * (dec * p + kq * u[c]);
    }
    if (write_o && warp < 4 && lane < 8) {
      if (a.io_dtype == GDN_BF16) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(o[2], o[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.o) + o_row * V + col) = pk;
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.o) + o_row * V + col) =
            make_float4(o[0], o[1], o[2], o[3]);
      }
    }
    float* inter = a.intermediate ? a.intermediate + hv_off * (size_t)(K * V) : nullptr;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float kr = sk[row0 + 4 * m];
      S[m].x = dec * S[m].x + kr * u[0];
      S[m].y = dec * S[m].y + kr * u[1];
      S[m].z = dec * S[m].z + kr * u[2];
      S[m].w = dec * S[m].w + kr * u[3];
      if (inter) __stcs(reinterpret_cast<float4*>(inter + (size_t)(row0 + 4 * m) * V + col), S[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < 16; ++m)
    __stcs(reinterpret_cast<float4*>(Sp + (size_t)(row0 + 4 * m) * V + col), S[m]);
}

// 16-byte asynchronous copy global -> shared (no register round trip), and the wait for them.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Any K, V (the boundary holds both to multiples of 4 floats): the K x V fp32 state is staged in
// shared memory once per (request, value head) by 16-byte cp.async copies, every token of the
// request updates it there, and it is written back once.  S^T k and S^T q: thread t takes column
// t % V of the rows t / V + G j (G = threads / V row groups: 128 threads for a state of at most
// 4096 floats, else 256); the groups' partial sums meet in shared memory.  Dynamic shared
// memory: K V + 2 * 256 floats.
__global__ void __launch_bounds__(kDecodeThreads) decode_generic_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) float dsm[];
  const int K = a.K, V = a.V;
  const int h = blockIdx.x % a.Hv;
  const int i = blockIdx.x / a.Hv;
  const int tid = threadIdx.x, nt = blockDim.x;   // 256, or 128 for a small state
  const int s = resolve_slot(a, i);
  if (s < 0) {
    if (a.product) zero_output(a, i, h);
    else for (int t = 0; t < a.L; ++t) zero_output(a, i * a.L + t, h);
    return;
  }
  const int hq = h / (a.Hv / a.Hqk);
  float* S = dsm;                        // [K][V]
  float* pr = S + K * V;                 // [G][V] partial S^T k
  float* pp = pr + kDecodeThreads;       // [G][V] partial S^T q
  __shared__ float sq[GDN_MAX_HEAD_DIM], sk[GDN_MAX_HEAD_DIM], su[GDN_MAX_HEAD_DIM];
  __shared__ float part[3][kDecodeThreads / 32];
  float* Sp = a.state + ((size_t)s * a.Hv + h) * (size_t)K * V;
  const int n4 = K * V / 4;
  float4* S4 = reinterpret_cast<float4*>(S);
  // the state streams into shared memory while the first token's q, k are read and normalised
  for (int e = tid; e < n4; e += nt) cp_async16(S4 + e, reinterpret_cast<const float4*>(Sp) + e);
  const int G = nt / V, c = tid % V, g = tid / V;
  for (int t = 0; t < a.L; ++t) {
    const int it = i * a.L + t;
    __syncthreads();   // the previous token's sq / sk / su settled
    const size_t qk_off = ((size_t)it * a.Hqk + hq) * K;
    const size_t q_off = a.product ? ((size_t)i * a.Hqk + hq) * K : qk_off;
    float xq = 0.f, xk = 0.f;
    if (tid < K) {
      xq = load_elem(a.q, q_off + tid, a.io_dtype);
      xk = load_elem(a.k, qk_off + tid, a.io_dtype);
    }
    float s1 = warp_sum(xq * xq), s2 = warp_sum(xk * xk), s3 = warp_sum(xq * xk);
    if ((tid & 31) == 0) { part[0][tid >> 5] = s1; part[1][tid >> 5] = s2; part[2][tid >> 5] = s3; }
    __syncthreads();
    float nq = 0.f, nk = 0.f, dqk = 0.f;
    for (int w = 0; w < nt / 32; ++w) { nq += part[0][w]; nk += part[1][w]; dqk += part[2][w]; }
    float rq = 1.f, rk = 1.f;
    if (a.use_qk_l2norm) { rq = 1.0f / sqrtf(nq + kL2Eps); rk = 1.0f / sqrtf(nk + kL2Eps); }
    if (tid < K) { sq[tid] = xq * rq; sk[tid] = xk * rk; }
    const float kq = dqk * rq * rk;
    __syncthreads();
    const size_t hv_off = (size_t)it * a.Hv + h;
    float gv, bt;
    if (a.product) {   // the token's decay on its first write only
      gv = (t == 0) ? a.g[(size_t)i * a.Hv + h] : 0.f;
      bt = load_elem(a.beta, hv_off, a.beta_dtype);
    } else {
      gate_values(a, hv_off, h, &gv, &bt);
    }
    const float dec = expf(gv);
    const bool write_o = !a.product || t == a.L - 1;
    const size_t o_row = a.product ? (size_t)i * a.Hv + h : hv_off;
    if (t == 0) {   // the staged state landed (each thread waits for its own copies, then all)
      cp_async_wait_all();
      __syncthreads();
    }
    if (g < G) {
      float r = 0.f, p = 0.f;
      for (int row = g; row < K; row += G) {
        const float x = S[row * V + c];
        r = fmaf(x, sk[row], r);
        p = fmaf(x, sq[row], p);
      }
      pr[g * V + c] = r;
      pp[g * V + c] = p;
    }
    __syncthreads();
    if (tid < V) {
      float r = 0.f, p = 0.f;
      for (int gg = 0; gg < G; ++gg) { r += pr[gg * V + tid]; p += pp[gg * V + tid]; }
      const float u = bt * (load_elem(a.v, hv_off * V + tid, a.io_dtype) - dec * r);
      su[tid] = u;
      if (write_o) store_elem(a.o, o_row * V + tid, a.scale * (dec * p + kq * u), a.io_dtype);
    }
    __syncthreads();
    float4* inter = a.intermediate ? reinterpret_cast<float4*>(a.intermediate + hv_off * (size_t)K * V) : nullptr;
    for (int e = tid; e < n4; e += nt) {
      const int row = (4 * e) / V, c0 = 4 * e - row * V;
      const float kr = sk[row];
      float4 x = S4[e];
      x.x = fmaf(dec, x.x, kr * su[c0]);
      x.y = fmaf(dec, x.y, kr * su[c0 + 1]);
      x.z = fmaf(dec, x.z, kr * su[c0 + 2]);
      x.w = fmaf(dec, x.w, kr * su[c0 + 3]);
      S4[e] = x;
      if (inter) __stcs(inter + e, x);
    }
  }
  __syncthreads();
  for (int e = tid; e < n4; e += nt) __stcs(reinterpret_cast<float4*>(Sp) + e, S4[e]);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a) {
  if (a.n == 0 || a.L == 0) return cudaSuccess;
  const long long blocks = (long long)a.n * a.Hv;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.K == 128 && a.V == 128) {
    decode128_kernel<<<(unsigned)blocks, kDecodeThreads, 0, a.stream>>>(a);
  } else {
    const int smem = (a.K * a.V + 2 * kDecodeThreads) * (int)sizeof(float);
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
      err = cudaFuncSetAttribute(decode_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (GDN_MAX_HEAD_DIM * GDN_MAX_HEAD_DIM + 2 * kDecodeThreads) * (int)sizeof(float));
      if (err != cudaSuccess) return err;
      if (dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
    }
    // a small state (K V <= 4096 floats) takes 128 threads: twice the resident CTAs per SM
    const int threads = a.K * a.V <= 4096 ? 128 : kDecodeThreads;
    decode_generic_kernel<<<(unsigned)blocks, threads, smem, a.stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
