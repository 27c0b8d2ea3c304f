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

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace gdn
