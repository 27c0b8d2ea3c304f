// gdn_common.cuh -- small device helpers shared by the libgdn kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Epsilon inside the square root of the in-kernel q/k L2 norm:
// x_hat = x / sqrt(sum x^2 + kL2Eps).
constexpr float kL2Eps = 1e-6f;

// Chunk length of the chunkwise evaluation (fixed at 64 for the inference
// kernels: "Megatron-Core API: core.ssm.gated_delta_product",
// ssm_inference_chunk_size).
constexpr int kChunk = 64;

__device__ __forceinline__ float load_elem(const void* p, size_t i, int dtype) {
  if (dtype == GDN_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_elem(void* p, size_t i, float x, int dtype) {
  if (dtype == GDN_BF16)
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float*>(p)[i] = x;
}

__device__ __forceinline__ void report(int* dev_status, int bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

// softplus(x) = log(1 + e^x), written as max(x, 0) + log1p(e^{-|x|}) so that it
// neither overflows nor loses the tail.
__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// Gate values of element i (= token * Hv + h) from the raw gate features (the
// fused-gate mode): g = -exp(A_log[h]) softplus(a + dt_bias[h]), beta = sigmoid(b).
template <class GA>
__device__ __forceinline__ void fused_gates(const GA& ga, size_t i, int h, float* g, float* beta) {
  const float av = load_elem(ga.a, i, ga.ab_dtype), bv = load_elem(ga.b, i, ga.ab_dtype);
  *g = -expf(ga.A_log[h]) * softplus_f(av + ga.dt_bias[h]);
  *beta = sigmoid_f(bv);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace gdn
