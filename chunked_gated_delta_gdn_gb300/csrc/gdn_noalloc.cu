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
#include "gdn.h"
#include "gdn_internal.h"

namespace {

// The scratch: one array per device that loads the library, held until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current context, looked up on every call.  In host
// code the array's name is only a host-side stand-in; cudaGetSymbolAddress, with the device
// current, gives the address in that device's context.  Nothing is cached: after a context is
// torn down and created again (cudaDeviceReset) the module is loaded anew, possibly at another
// address, and a lookup that failed once is simply tried again on the next call.  The lookup
// is a host-side table query once the module is loaded; the first call on a device may load
// the module, which is why that first call must come before any stream capture.
cudaError_t scratch_on_current_device(void** out) {
  return cudaGetSymbolAddress(out, g_noalloc_scratch);
}

// The stream's device, which must be the current one: the scratch address is the current
// device's.  The NULL stream is the current device's.
bool stream_on_current_device(void* stream) {
  if (!stream) return true;
  int cur = 0, sdev = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return false;
  if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return false;
  return sdev == cur;
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
  // the tensor-core path runs without its launch plan when the plan does not fit
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES && gdn_chunk_fwd_path(K, V, io_dtype, beta_dtype) != 1)
    return GDN_ERR_WORKSPACE;
  if (!stream_on_current_device(stream)) return GDN_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn_chunk_fwd(q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, beta_dtype, scale,
                       chunk_size, initial_state, output_final_state, final_state, use_qk_l2norm,
                       cu_seqlens, num_seqs, state_indices, num_slots, o, scratch,
                       (size_t)GDN_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
