// gdn_selftest.cu -- the bounded-wait path of the fused kernels, exercised on its own.
//
// Every mbarrier wait in the tensor-core kernels goes through sm100::mbar_wait with a time
// limit; when a wait gives up, the kernel sets GDN_DEV_TIMEOUT in the caller's status word,
// drains what it has in flight and returns instead of hanging.  This entry point runs that wait
// in a one-thread kernel with nothing in flight: on an mbarrier that nobody arrives on (the
// wait must give up after limit_ns and report the timeout), or on one the thread has already
// arrived on (the wait must succeed and report nothing).
#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_sm100.cuh"

namespace {

__global__ void wait_selftest_kernel(int* dev_status, unsigned long long limit_ns, int arrive_first,
                                     unsigned long long* waited_ns) {
  using namespace gdn::sm100;
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (arrive_first) mbar_arrive(&bar);
  const uint64_t t0 = globaltimer_ns();
  const bool ok = mbar_wait(&bar, 0u, limit_ns);
  if (waited_ns) *waited_ns = globaltimer_ns() - t0;
  if (!ok) gdn::report(dev_status, GDN_DEV_TIMEOUT);
}

}  // namespace

extern "C" gdn_status_t gdn_selftest_wait_timeout(int* dev_status, unsigned long long limit_ns,
                                                  int arrive_first, unsigned long long* waited_ns,
                                                  void* stream) {
  if (!dev_status) return GDN_ERR_NULL;
  if (limit_ns == 0 || limit_ns > 100000000ull) return GDN_ERR_SHAPE;   // (0, 100 ms]
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status, limit_ns,
                                                                        arrive_first, waited_ns);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
