// gdn_noalloc.cu -- gdn_chunk_fwd for callers that cannot allocate device memory.
//
// The CUDA-core chunk kernels keep their per-chunk intermediates (W, U, U', the
// entry state of every chunk and the chunk table) in caller-provided scratch.
// Some callers have no way to provide it: a plugin running inside another
// runtime whose device memory is fully reserved by that runtime, a C caller
// without an allocator of its own, or code that must not call cudaMalloc in the
// middle of a step because it would synchronise the device.  This entry point
// gives them the same computation with the scratch taken from one file-scope
// device array instead, so nothing is allocated per call.
#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

// The scratch: one array per device that loads the library, held until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device, with that device current, and cached.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], [dev] {
    g_scratch_err[dev] = cudaGetSymbolAddress(&g_scratch_addr[dev], g_noalloc_scratch);
  });
  if (g_scratch_err[dev] != cudaSuccess) return g_scratch_err[dev];
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" gdn_status_t gdn_chunk_fwd_noalloc(
    const void* q, const void* k, const void* v, const float* g, const void* beta, int B, int T,
    int Hqk, int Hv, int K, int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
    int chunk_size, const float* initial_state, int output_final_state, float* final_state,
    int use_qk_l2norm, const int32_t* cu_seqlens, int num_seqs, const int32_t* state_indices,
    int num_slots, void* o, int* dev_status, void* stream) {
  const int N = cu_seqlens ? num_seqs : B;
  const size_t need =
      gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, K, V, N, io_dtype, beta_dtype);
  if (need == (size_t)-1) {
    // Let gdn_chunk_fwd name the argument error.
    return gdn_chunk_fwd(q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, beta_dtype, scale,
                         chunk_size, initial_state, output_final_state, final_state,
                         use_qk_l2norm, cu_seqlens, num_seqs, state_indices, num_slots, o,
                         nullptr, 0, dev_status, stream);
  }
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn_chunk_fwd(q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, beta_dtype, scale,
                       chunk_size, initial_state, output_final_state, final_state, use_qk_l2norm,
                       cu_seqlens, num_seqs, state_indices, num_slots, o, scratch,
                       (size_t)GDN_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
