// tcgen05_rates.cu -- one-CTA rates of the tensor-core operations the fused chunk kernel issues.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -I chunked_gated_delta_gdn_gb300/csrc -I include -o tcgen05_rates \
//        chunked_gated_delta_gdn_gb300/microbench/tcgen05_rates.cu && ./tcgen05_rates
//
// Part A: tcgen05.mma kind::f16 (bf16 in, fp32 accumulate), M = 128, K = 16 per instruction,
//   for each operand source and major-ness the kernel uses (A and B in shared memory, K-major or
//   MN-major; A from TMEM) and N = 64 .. 256: 64 back-to-back instructions issued by one thread
//   (cycles per instruction and FLOP per SM clock), and the latency of a group of 4 / 8
//   instructions followed by tcgen05.commit and the mbarrier wait (the kernel's hand-off unit).
// Part B: 64 N = 128 instructions while eight other warps issue warp-level mma.sync (tf32
//   m16n8k8) -- the legacy tensor path the chunk kernel's triangular solve uses -- and how many
//   of those mma.sync complete meanwhile.
// Every wait is bounded (1 s); the results are clock64 cycles of the SM clock.
#include <cstdio>
#include <cstdint>
#include <cuda_bf16.h>

#include "gdn_sm100.cuh"

using namespace gdn::sm100;

namespace {

__device__ __forceinline__ unsigned long long clk() {
  unsigned long long c;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
  return c;
}

constexpr int kSmem = 65536 + 1024 + 256;
struct Out { unsigned long long v[128]; };

// operand sources (the chunk kernel's products in brackets)
enum Src { SS_KK = 0,   // A, B in smem, K-major           [D1 = [Q;K][Q;K]^T]
           SS_MM = 1,   // A, B in smem, MN-major          [U^T = V^T Tu^T]
           TS_K = 2,    // A in TMEM, B smem K-major       [[O1|Y] = S^T [Q;K]^T, O2, S^T update]
           TS_MN = 3 }; // A in TMEM, B smem MN-major      [U'^T += (-Y) Tw^T]

template <int kSrc, int kN>
__device__ __forceinline__ void issue(uint32_t tb, uint32_t sa, uint32_t sb, int ks, bool acc) {
  constexpr bool a_mn = (kSrc == SS_MM), b_mn = (kSrc == SS_MM || kSrc == TS_MN);
  constexpr uint32_t id = idesc_bf16(128, kN, a_mn, b_mn);
  // K-major: 128-byte rows along K, k-step = 32 bytes; MN-major: 16 K-rows of 128 bytes a k-step,
  // 64-element MN blocks 8192 bytes apart
  const uint64_t bd = b_mn ? sdesc_sw128(sb + ks * 2048, 8192, 1024) : sdesc_sw128(sb + ks * 32, 16, 1024);
  if (kSrc == TS_K || kSrc == TS_MN) {
    mma_bf16_ta(tb, tb + 256 + 8 * ks, bd, id, acc);
  } else {
    const uint64_t ad = a_mn ? sdesc_sw128(sa + ks * 2048, 8192, 1024) : sdesc_sw128(sa + ks * 32, 16, 1024);
    mma_bf16(tb, ad, bd, id, acc);
  }
}

// Part A, one configuration (operand source, N, group size G): out[0] = 64 back-to-back
// instructions, out[1] = a group of G; both up to the completion the mbarrier reports.
template <int kSrc, int kN, int kG>
__global__ void __launch_bounds__(128, 1) rates_kernel(unsigned long long* out) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 65536);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 65536 + 64);
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 65536 / 2; i += 128)
    reinterpret_cast<__nv_bfloat16*>(sm)[i] = __float2bfloat16_rn((float)((i * 37) % 17) * 0.01f);
  if (tid == 0) { mbar_init(bar, 1); fence_mbar_init(); }
  if (warp == 0) { tmem_alloc(slot, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *slot;
  const uint32_t sa = smem_u32(sm), sb = smem_u32(sm + 32768);
  if (tid == 0) {
    tc_fence_after();
    unsigned long long t0 = clk();
#pragma unroll
    for (int r = 0; r < 64; ++r) issue<kSrc, kN>(tb, sa, sb, r & 3, r > 0);
    mma_commit(bar);
    bool ok = mbar_wait(bar, 0u, 1000000000ull);
    out[0] = ok ? clk() - t0 : 0ull;
    t0 = clk();
#pragma unroll
    for (int r = 0; r < kG; ++r) issue<kSrc, kN>(tb, sa, sb, r & 3, r > 0);
    mma_commit(bar);
    ok = mbar_wait(bar, 1u, 1000000000ull);
    out[1] = ok ? clk() - t0 : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tb, 512);
}

// Part B: warp 0 times 64 N = 128 SS instructions (three repetitions) while warps 4-11 run
// mma.sync tf32 (mode 1; mode 0: idle), stopping when warp 0 is done or after 2^20 rounds.  Mode
// 2: no tcgen05 work; warp 0 only waits 14,100 cycles (about the time of mode 1) and the other
// warps run mma.sync meanwhile.
__global__ void __launch_bounds__(384, 1) interference_kernel(Out* out, int mode) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 65536);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 65536 + 64);
  volatile int* stop = reinterpret_cast<volatile int*>(sm + 65536 + 128);
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 65536 / 2; i += 384)
    reinterpret_cast<__nv_bfloat16*>(sm)[i] = __float2bfloat16_rn((float)((i * 37) % 17) * 0.01f);
  if (tid == 0) { mbar_init(bar, 1); fence_mbar_init(); *stop = 0; }
  if (warp == 0) { tmem_alloc(slot, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *slot;
  if (warp == 0) {
    const uint32_t sa = smem_u32(sm), sb = smem_u32(sm + 32768);
    const unsigned long long tw = clk();
    while (clk() - tw < 2000) {}   // let the other warps start
    uint32_t phase = 0;
    if (mode == 2) {
      const unsigned long long t0 = clk();
      while (clk() - t0 < 14100) {}
      out->v[80] = clk() - t0;
    }
    for (int rep = 0; rep < 3 && mode != 2; ++rep) {
      if (tid == 0) {
        tc_fence_after();
        const unsigned long long t0 = clk();
#pragma unroll
        for (int r = 0; r < 64; ++r) issue<SS_KK, 128>(tb, sa, sb, r & 3, r > 0);
        mma_commit(bar);
        const bool ok = mbar_wait(bar, phase, 1000000000ull);
        out->v[80 + rep] = ok ? clk() - t0 : 0ull;
      }
      __syncwarp();
      phase ^= 1u;
    }
    if (tid == 0) *stop = 1;
  } else if (warp >= 4 && mode >= 1) {
    float d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};
    uint32_t a[4], b[2];
    for (int j = 0; j < 4; ++j) a[j] = to_tf32(0.001f * (tid + j));
    b[0] = to_tf32(0.5f);
    b[1] = to_tf32(0.25f);
    unsigned long long n = 0;
    while (!*stop && n < (1ull << 20)) {
      mma_tf32_16x8x8(d0, a, b);
      mma_tf32_16x8x8(d1, a, b);
      n += 2;
    }
    if ((tid & 31) == 0) out->v[96 + warp - 4] = n + (d0[0] + d1[1] == 1234.5f ? 1 : 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tb, 512);
}

int check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    printf("%s: %s\n", what, cudaGetErrorString(e));
    return 1;
  }
  return 0;
}

}  // namespace

template <int kSrc, int kN, int kG>
int run_config(unsigned long long* d, const char* name, const char* use) {
  cudaFuncSetAttribute(rates_kernel<kSrc, kN, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  cudaMemset(d, 0, 2 * sizeof(unsigned long long));
  rates_kernel<kSrc, kN, kG><<<1, 128, kSmem>>>(d);
  if (check(cudaDeviceSynchronize(), "rates_kernel")) return 1;
  unsigned long long h[2];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  const double per = h[0] / 64.0;
  printf("| %s | %d | %s | %llu | %.1f | %.0f | %d instr: %llu |\n", name, kN, use, h[0], per,
         2.0 * 128 * kN * 16 / per, kG, h[1]);
  return 0;
}

int main() {
  const char* ss_kk = "A, B smem, K-major";
  const char* ss_mm = "A, B smem, MN-major";
  const char* ts_k = "A TMEM, B smem K-major";
  const char* ts_mn = "A TMEM, B smem MN-major";
  unsigned long long* dv;
  if (check(cudaMalloc(&dv, 2 * sizeof(unsigned long long)), "cudaMalloc")) return 1;
  printf("## A. tcgen05.mma kind::f16, M = 128, K = 16 per instruction (cycles, SM clock)\n\n");
  printf("| operands | N | chunk-kernel use | 64 back-to-back | per instr | FLOP/clk | group + commit + wait |\n");
  printf("|---|---|---|---|---|---|---|\n");
  int bad = 0;
  bad |= run_config<SS_KK, 64, 8>(dv, ss_kk, "-");
  bad |= run_config<SS_KK, 128, 8>(dv, ss_kk, "D1 = [Q;K][Q;K]^T");
  bad |= run_config<SS_KK, 192, 8>(dv, ss_kk, "-");
  bad |= run_config<SS_KK, 256, 8>(dv, ss_kk, "-");
  bad |= run_config<SS_MM, 64, 4>(dv, ss_mm, "U^T = V^T Tu^T");
  bad |= run_config<SS_MM, 128, 4>(dv, ss_mm, "-");
  bad |= run_config<TS_K, 64, 4>(dv, ts_k, "O2 = U'^T P^T");
  bad |= run_config<TS_K, 128, 8>(dv, ts_k, "[O1|Y] = S^T [Q;K]^T; S^T += U'^T K~ (4 instr)");
  bad |= run_config<TS_K, 192, 4>(dv, ts_k, "-");
  bad |= run_config<TS_K, 256, 8>(dv, ts_k, "-");
  bad |= run_config<TS_MN, 64, 4>(dv, ts_mn, "U'^T = U^T + (-Y) Tw^T");
  bad |= run_config<TS_MN, 128, 4>(dv, ts_mn, "-");
  cudaFree(dv);
  if (bad) return 1;
  Out* d;
  if (check(cudaMalloc(&d, sizeof(Out)), "cudaMalloc")) return 1;
  Out h;
  cudaMemset(d, 0, sizeof(Out));
  cudaFuncSetAttribute(interference_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  printf("\n## B. 64 N = 128 tcgen05.mma while other warps run mma.sync (tf32 m16n8k8)\n\n");
  printf("| other warps | 64 MMAs (3 repetitions) | mma.sync completed meanwhile (8 warps) |\n");
  printf("|---|---|---|\n");
  for (int mode = 0; mode < 3; ++mode) {
    cudaMemset(d, 0, sizeof(Out));
    interference_kernel<<<1, 384, kSmem>>>(d, mode);
    if (check(cudaDeviceSynchronize(), "interference_kernel")) return 1;
    cudaMemcpy(&h, d, sizeof(Out), cudaMemcpyDeviceToHost);
    unsigned long long n = 0;
    for (int w = 0; w < 8; ++w) n += h.v[96 + w];
    if (mode == 2)
      printf("| 8 warps of mma.sync, no tcgen05 work (window %llu cycles) | - | %llu |\n", h.v[80], n);
    else
      printf("| %s | %llu %llu %llu | %llu |\n", mode ? "8 warps of mma.sync" : "idle", h.v[80],
             h.v[81], h.v[82], n);
  }
  cudaFree(d);
  return 0;
}
