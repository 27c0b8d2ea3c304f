// gdn_chunk_split.cu -- the planned launch of the tensor-core chunk forward: sequences sorted
// longest first and, when the batch has too few (sequence, value head) chains to fill the GPU,
// each long chain split into segments that run concurrently.
//
// The chunkwise gated delta rule maps the state entering a token range affinely to the state
// leaving it (every token applies S <- exp(g) (I - beta k k^T) S + beta k v^T, "Megatron-Core
// API: core.ssm.gated_delta_net.gdn", torch_chunk_gated_delta_rule), and the output of every
// token is linear in the state entering its chunk.  A sequence cut into segments 0 .. s-1 is
// therefore computed exactly by
//   pass 1 (concurrent): segment 0 from the caller's entry state, keeping its exit state E_1;
//          for each middle segment j = 1 .. s-2 its K x K transition M_j (the run with v = 0
//          from S = I) and its contribution B_j (the run with the true v from S = 0);
//   scan:   E_{j+1} = M_j E_j + B_j, j = 1 .. s-2 (fp32, one launch a step, four CTAs a chain);
//   pass 2 (concurrent): segments 1 .. s-1 from E_j, writing their outputs and, for the last,
//          the caller's final state.
// The plan (which sequences split, the unit tables, the scan list) is built on the device from
// cu_seqlens, so a captured graph replays it for any lengths.  The segment count s comes from
// the host-known chain count N Hv and the SM count alone.  Context parallelism over the
// sequence dimension is what the pages' Gated Delta Product mixer does across GPUs ("Megatron-
// Core API: core.ssm.gated_delta_product", GatedDeltaProductMixer, packed_sequence_cp_metadata);
// here the segments share one GPU.
#include <algorithm>
#include <atomic>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kKV = 128 * 128;        // floats of one [K][V] state (K = V = 128)
constexpr int kBuckets = 4096;        // length buckets of the sort (chunks, capped)
constexpr int kPlanThreads = 1024;
constexpr int kScanThreads = 256;
constexpr int kScanSlabs = 4;        // CTAs per chain in a scan step (32 rows each)
constexpr int kMaxSegments = 16;
constexpr int kMaxDevices = 64;

struct ScanEntry {
  float* E;          // E_1 .. E_{s-1}, consecutive [K][V] blocks
  const float* MT;   // M_1^T .. M_{s-2}^T
  const float* Bc;   // B_1 .. B_{s-2}
  int steps;         // s - 2
  int pad_;
};

struct PlanArgs {
  const int32_t* cu_seqlens;   // NULL: B rows of T tokens
  int B, T, N, Hv;
  const int32_t* state_indices;
  int num_slots;
  const float* initial_state;
  float* final_state;
  int s;                       // segments of a split sequence (>= 3), 1: no splitting
  int* counters;               // [0] pass-1 units, [1] pass-2 units, [2] scan entries
  TcUnit* units1;
  TcUnit* units2;
  ScanEntry* scans;
  float* mats;
  int* place;                  // [N] scratch: each sequence's place in the sorted order
  int* dev_status;
};

struct SeqInfo {
  int bos, eos, nch;
  bool valid, padding;
  const float* init;
  float* fin;
  int report;   // status bit to report for this sequence, or 0
};

__device__ SeqInfo seq_info(const PlanArgs& p, int n) {
  SeqInfo r;
  const int T_total = p.cu_seqlens ? p.T : p.B * p.T;
  if (p.cu_seqlens) { r.bos = p.cu_seqlens[n]; r.eos = p.cu_seqlens[n + 1]; }
  else { r.bos = n * p.T; r.eos = r.bos + p.T; }
  r.valid = !(r.bos < 0 || r.eos < r.bos || r.eos > T_total);
  r.report = r.valid ? 0 : GDN_DEV_BAD_CU_SEQLENS;
  r.nch = r.valid ? (r.eos - r.bos + 63) / 64 : 0;
  r.padding = false;
  int slot = n;
  if (r.valid && p.state_indices) {
    slot = p.state_indices[n];
    if (slot < 0 || slot >= p.num_slots) {
      r.padding = true;
      if (slot != -1) r.report = GDN_DEV_BAD_SLOT;
      slot = 0;
    }
  }
  const size_t base = (size_t)slot * p.Hv * kKV;
  r.init = p.initial_state ? p.initial_state + base : nullptr;
  r.fin = p.final_state ? p.final_state + base : nullptr;
  return r;
}

__device__ __forceinline__ bool splits(const PlanArgs& p, const SeqInfo& q) {
  return p.s >= 3 && q.valid && !q.padding && q.nch >= 2 * p.s;
}

__device__ __forceinline__ TcUnit make_unit(const float* init, float* fin, int n, int h, int bos,
                                            int eos, int flags) {
  TcUnit u;
  u.init = init; u.fin = fin; u.n = n; u.h = h; u.bos = bos; u.eos = eos; u.flags = flags; u.pad_ = 0;
  return u;
}

// One CTA.  Sorts the sequences by chunk count, longest first (a counting sort over capped
// lengths; the order of equal lengths is whichever thread claims its place first, which
// changes no result), then writes the units of every (sequence, head) at the sequence's place
// in that order.  The split sequences (at least 2 s chunks) sort ahead of all others, so
// place p < n_split identifies them and their unit offsets follow from p alone.
__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const PlanArgs p) {
  __shared__ int hist[kBuckets];
  __shared__ int warp_sum[kPlanThreads / 32];
  __shared__ int n_split;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int b = tid; b < kBuckets; b += kPlanThreads) hist[b] = 0;
  if (tid == 0) n_split = 0;
  __syncthreads();
  for (int n = tid; n < p.N; n += kPlanThreads) {
    const SeqInfo q = seq_info(p, n);
    const int key = (q.valid && !q.padding) ? min(q.nch, kBuckets - 1) : 0;
    atomicAdd(&hist[kBuckets - 1 - key], 1);
    if (splits(p, q)) atomicAdd(&n_split, 1);
  }
  __syncthreads();
  // exclusive prefix sum over the buckets in descending length order (4 buckets a thread)
  int v[4], local = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) { v[i] = hist[4 * tid + i]; local += v[i]; }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sum[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += x;
    }
    warp_sum[lane] = wi - w;   // exclusive over warps
  }
  __syncthreads();
  int run = warp_sum[warp] + incl - local;
#pragma unroll
  for (int i = 0; i < 4; ++i) { hist[4 * tid + i] = run; run += v[i]; }
  __syncthreads();
  // every sequence's place in the order
  for (int n = tid; n < p.N; n += kPlanThreads) {
    const SeqInfo q = seq_info(p, n);
    if (q.report) report(p.dev_status, q.report);
    const int key = (q.valid && !q.padding) ? min(q.nch, kBuckets - 1) : 0;
    p.place[n] = atomicAdd(&hist[kBuckets - 1 - key], 1);
  }
  __syncthreads();   // the places, written to global memory, are visible to the whole CTA

  const int s = p.s, Hv = p.Hv, ns = n_split;
  const int u1_split = 2 * s - 3, mats_split = 3 * s - 5;
  for (long long idx = tid; idx < (long long)p.N * Hv; idx += kPlanThreads) {
    const int n = (int)(idx / Hv), h = (int)(idx % Hv);
    const SeqInfo q = seq_info(p, n);
    const int pos = p.place[n];
    const float* init = q.init ? q.init + (size_t)h * kKV : nullptr;
    float* fin = q.fin ? q.fin + (size_t)h * kKV : nullptr;
    if (!splits(p, q)) {
      const long long off1 = (long long)Hv * ((long long)u1_split * min(pos, ns) + max(pos - ns, 0));
      const int flags = !q.valid ? kUnitSkip : (q.padding ? kUnitPadding : 0);
      p.units1[off1 + h] = make_unit(init, fin, n, h, q.bos, q.eos, flags);
      continue;
    }
    // split sequence at place pos < n_split: segment j covers chunks [j nch / s, (j+1) nch / s)
    float* m = p.mats + ((size_t)pos * Hv + h) * mats_split * kKV;
    float* E = m;                              // E_1 .. E_{s-1}
    float* M = m + (size_t)(s - 1) * kKV;      // M_1^T .. M_{s-2}^T
    float* Bc = M + (size_t)(s - 2) * kKV;     // B_1 .. B_{s-2}
    TcUnit* u1 = p.units1 + (long long)Hv * u1_split * pos + (long long)h * u1_split;
    TcUnit* u2 = p.units2 + (long long)Hv * (s - 1) * pos + (long long)h * (s - 1);
    for (int j = 0; j < s; ++j) {
      const int t0 = q.bos + 64 * (int)(((long long)j * q.nch) / s);
      const int t1 = (j == s - 1) ? q.eos : q.bos + 64 * (int)(((long long)(j + 1) * q.nch) / s);
      if (j == 0) {
        u1[0] = make_unit(init, E, n, h, t0, t1, 0);
        continue;
      }
      if (j <= s - 2) {
        u1[1 + 2 * (j - 1)] = make_unit(nullptr, M + (size_t)(j - 1) * kKV, n, h, t0, t1,
                                        kUnitZeroV | kUnitIdentity | kUnitNoOut | kUnitFinT);
        u1[2 + 2 * (j - 1)] = make_unit(nullptr, Bc + (size_t)(j - 1) * kKV, n, h, t0, t1, kUnitNoOut);
      }
      u2[j - 1] = make_unit(E + (size_t)(j - 1) * kKV, j == s - 1 ? fin : nullptr, n, h, t0, t1, 0);
    }
    ScanEntry e;
    e.E = E; e.MT = M; e.Bc = Bc; e.steps = s - 2; e.pad_ = 0;
    p.scans[(size_t)pos * Hv + h] = e;
  }
  if (tid == 0) {
    p.counters[0] = Hv * (u1_split * ns + (p.N - ns));
    p.counters[1] = Hv * (s - 1) * ns;
    p.counters[2] = Hv * ns;
  }
}

// One step of the scan, E_{j+2} = M_{j+1} E_{j+1} + B_{j+1} ([K][V] fp32 row-major; M given
// transposed), fp32 on the CUDA cores.  Four CTAs per chain, each 32 rows of the result: E and
// 32 columns of M^T staged in shared memory, each thread a 4 x 4 block.
__global__ void __launch_bounds__(kScanThreads) scan_step_kernel(const ScanEntry* scans,
                                                                 const int* count, int j) {
  const int chain = blockIdx.x / kScanSlabs, slab = blockIdx.x % kScanSlabs;
  if (chain >= *count) return;
  const ScanEntry e = scans[chain];
  extern __shared__ __align__(16) float sh[];
  float* Es = sh;          // [k][v]
  float* Ms = sh + kKV;    // [k][r] = M[32 slab + r][k]
  const int tid = threadIdx.x;
  const int r0 = 4 * (tid >> 5), v0 = 4 * (tid & 31);
  const float* Ein = e.E + (size_t)j * kKV;
  const float* MT = e.MT + (size_t)j * kKV;
  for (int x = tid; x < kKV / 4; x += kScanThreads)
    reinterpret_cast<float4*>(Es)[x] = reinterpret_cast<const float4*>(Ein)[x];
  for (int x = tid; x < 128 * 8; x += kScanThreads) {   // 8 float4 of each M^T row
    const int k = x >> 3, c = x & 7;
    reinterpret_cast<float4*>(Ms)[x] = *reinterpret_cast<const float4*>(MT + (size_t)k * 128 + 32 * slab + 4 * c);
  }
  const int i0 = 32 * slab + r0;
  const float* Bc = e.Bc + (size_t)j * kKV;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float4 b = *reinterpret_cast<const float4*>(Bc + (size_t)(i0 + r) * 128 + v0);
    acc[r][0] = b.x; acc[r][1] = b.y; acc[r][2] = b.z; acc[r][3] = b.w;
  }
  __syncthreads();
#pragma unroll 8
  for (int k = 0; k < 128; ++k) {
    const float4 a = *reinterpret_cast<const float4*>(Ms + k * 32 + r0);   // one address a warp
    const float4 c = *reinterpret_cast<const float4*>(Es + k * 128 + v0);
    const float av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(av[r], cv[q], acc[r][q]);
  }
  float* Eout = e.E + (size_t)(j + 1) * kKV;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    *reinterpret_cast<float4*>(Eout + (size_t)(i0 + r) * 128 + v0) =
        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PlanLayout {
  size_t counters, place, units1, units2, scans, mats, total;
  long long cap1, cap2, cap_scan;
};

PlanLayout plan_layout(int N, int Hv, int s) {
  PlanLayout L;
  const long long P = (long long)N * Hv;
  L.cap1 = P * (s >= 3 ? 2 * s - 3 : 1);
  L.cap2 = s >= 3 ? P * (s - 1) : 0;
  L.cap_scan = s >= 3 ? P : 0;
  const long long nmats = s >= 3 ? P * (3 * s - 5) : 0;
  size_t off = 0;
  L.counters = off; off += align256(4 * sizeof(int));
  L.place = off; off += align256((size_t)N * sizeof(int));
  L.units1 = off; off += align256((size_t)L.cap1 * sizeof(TcUnit));
  L.units2 = off; off += align256((size_t)L.cap2 * sizeof(TcUnit));
  L.scans = off; off += align256((size_t)L.cap_scan * sizeof(ScanEntry));
  L.mats = off; off += (size_t)nmats * kKV * sizeof(float);
  L.total = off;
  return L;
}

}  // namespace

int device_sm_count(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int sms = cache[dev].load(std::memory_order_relaxed);
  if (sms > 0) return sms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

int chunk_tc_segments(int num_seqs, int Hv, int num_sms) {
  const long long P = (long long)num_seqs * Hv;
  if (P <= 0 || num_sms <= 0) return 1;
  // pass 1 runs 2 s - 3 units per chain; keep them within one wave of one CTA per SM
  const long long s = (num_sms / P + 3) / 2;
  if (s < 3) return 1;
  return (int)std::min<long long>(s, kMaxSegments);
}

size_t chunk_tc_plan_bytes(int num_seqs, int Hv, int segments) {
  return plan_layout(num_seqs, Hv, segments).total;
}

cudaError_t launch_chunk_tc_planned(const ChunkArgs& a0) {
  const bool rec = a0.rec_states && a0.rec_u && a0.rec_chunk_off;
  if (rec || a0.num_seqs <= 0) return launch_chunk_tc(a0);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int s = chunk_tc_segments(a0.num_seqs, a0.Hv, device_sm_count(dev));
  if (s == 1 && !a0.cu_seqlens) return launch_chunk_tc(a0);   // equal rows: nothing to plan
  const PlanLayout L = plan_layout(a0.num_seqs, a0.Hv, s);
  if (!a0.workspace || a0.workspace_bytes < L.total || ((uintptr_t)a0.workspace & 255u))
    return launch_chunk_tc(a0);
  if (L.cap1 > 0x7fffffffLL || L.cap2 > 0x7fffffffLL) return launch_chunk_tc(a0);
  uint8_t* w = reinterpret_cast<uint8_t*>(a0.workspace);
  PlanArgs p;
  p.cu_seqlens = a0.cu_seqlens;
  p.B = a0.B; p.T = a0.T; p.N = a0.num_seqs; p.Hv = a0.Hv;
  p.state_indices = a0.state_indices;
  p.num_slots = a0.num_slots;
  p.initial_state = a0.initial_state;
  p.final_state = a0.final_state;
  p.s = s;
  p.counters = reinterpret_cast<int*>(w + L.counters);
  p.units1 = reinterpret_cast<TcUnit*>(w + L.units1);
  p.units2 = reinterpret_cast<TcUnit*>(w + L.units2);
  p.scans = reinterpret_cast<ScanEntry*>(w + L.scans);
  p.mats = reinterpret_cast<float*>(w + L.mats);
  p.place = reinterpret_cast<int*>(w + L.place);
  p.dev_status = a0.dev_status;
  plan_kernel<<<1, kPlanThreads, 0, a0.stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  ChunkArgs a = a0;
  a.units = p.units1;
  a.unit_count = p.counters;
  a.unit_cap = (int)L.cap1;
  err = launch_chunk_tc(a);
  if (err != cudaSuccess || s < 3) return err;

  const int scan_smem = (kKV + 128 * 32) * (int)sizeof(float);
  static std::atomic<bool> scan_attr[kMaxDevices];
  if (dev >= kMaxDevices || !scan_attr[dev].load(std::memory_order_relaxed)) {
    err = cudaFuncSetAttribute(scan_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, scan_smem);
    if (err != cudaSuccess) return err;
    if (dev < kMaxDevices) scan_attr[dev].store(true, std::memory_order_relaxed);
  }
  for (int j = 0; j < s - 2; ++j) {
    scan_step_kernel<<<(unsigned)(L.cap_scan * kScanSlabs), kScanThreads, scan_smem, a0.stream>>>(
        p.scans, p.counters + 2, j);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }

  a.units = p.units2;
  a.unit_count = p.counters + 1;
  a.unit_cap = (int)L.cap2;
  return launch_chunk_tc(a);
}

}  // namespace gdn
