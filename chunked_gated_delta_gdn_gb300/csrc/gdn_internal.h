// gdn_internal.h -- launchers behind the C ABI (not part of the public header).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const void* beta;
  int B, T, Hqk, Hv, K, V;
  int io_dtype, beta_dtype;
  float scale;
  const float* initial_state;
  float* final_state;  // NULL when no final state is requested
  int use_qk_l2norm;
  const int32_t* cu_seqlens;  // NULL: uniform rows of T tokens
  int num_seqs;               // N
  const int32_t* state_indices;
  int num_slots;
  void* o;
  void* workspace;
  size_t workspace_bytes;
  int* dev_status;
  cudaStream_t stream;
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const void* beta;
  float* state;
  int num_slots;
  const int32_t* batch_indices;
  int n, Hqk, Hv, K, V;
  int io_dtype, beta_dtype;
  float scale;
  int use_qk_l2norm;
  void* o;
  int* dev_status;
  cudaStream_t stream;
};

// Upper bound on the number of 64-token chunks over all sequences.
inline long long max_chunks(int T_total, int num_seqs) {
  return ((long long)T_total + 63) / 64 + (long long)num_seqs;
}

// fp32 CUDA-core chunk path (any accepted K, V, dtype).
size_t chunk_generic_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V);
cudaError_t launch_chunk_generic(const ChunkArgs& a);

// Fused tcgen05 / TMEM / TMA path (bf16, K = V = 128).
bool chunk_tc_supported(int K, int V, int io_dtype, int beta_dtype);
cudaError_t launch_chunk_tc(const ChunkArgs& a);

cudaError_t launch_decode(const DecodeArgs& a);

}  // namespace gdn
