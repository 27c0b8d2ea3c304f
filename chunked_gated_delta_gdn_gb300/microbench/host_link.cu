// host_link.cu -- what the host link carries: 2 GiB of pinned host memory copied to and from
// the device by the copy engines on 1, 2, 4 and 8 streams, by a kernel reading or writing the
// mapped host memory, and by copies in both directions at once.  The end-to-end figures of the
// bench move every step's inputs and outputs over this link.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o host_link host_link.cu && ./host_link
#include <cstdio>
#include <cuda_runtime.h>
#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("err %s at %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

__global__ void copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) dst[i] = src[i];
}

int main() {
  const size_t bytes = (size_t)2 << 30;   // 2 GiB
  void* h = nullptr; void* d = nullptr;
  CK(cudaHostAlloc(&h, bytes, cudaHostAllocMapped));
  CK(cudaMalloc(&d, bytes));
  memset(h, 1, bytes);
  CK(cudaMemset(d, 0, bytes));
  void* hd = nullptr;
  CK(cudaHostGetDevicePointer(&hd, h, 0));
  cudaStream_t st[8];
  for (int i = 0; i < 8; ++i) CK(cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
  int sms = 0; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  for (int dir = 0; dir < 2; ++dir) {   // 0: h2d, 1: d2h
    for (int ns : {1, 2, 4, 8}) {
      float best = 1e9f;
      for (int rep = 0; rep < 4; ++rep) {
        CK(cudaDeviceSynchronize());
        CK(cudaEventRecord(e0, 0));
        for (int i = 0; i < ns; ++i) CK(cudaStreamWaitEvent(st[i], e0, 0));
        const size_t part = bytes / ns;
        for (int i = 0; i < ns; ++i) {
          char* hp = (char*)h + i * part; char* dp = (char*)d + i * part;
          if (dir == 0) CK(cudaMemcpyAsync(dp, hp, part, cudaMemcpyHostToDevice, st[i]));
          else CK(cudaMemcpyAsync(hp, dp, part, cudaMemcpyDeviceToHost, st[i]));
        }
        for (int i = 0; i < ns; ++i) { cudaEvent_t ev; CK(cudaEventCreate(&ev)); CK(cudaEventRecord(ev, st[i])); CK(cudaStreamWaitEvent(0, ev, 0)); CK(cudaEventDestroy(ev)); }
        CK(cudaEventRecord(e1, 0));
        CK(cudaEventSynchronize(e1));
        float ms = 0; CK(cudaEventElapsedTime(&ms, e0, e1));
        if (rep > 0 && ms < best) best = ms;
      }
      printf("%s copy engines, %d stream(s): %.1f GB/s\n", dir ? "d2h" : "h2d", ns, bytes / (best * 1e-3) / 1e9);
    }
    for (int blocks : {sms, 2 * sms, 4 * sms}) {
      float best = 1e9f;
      for (int rep = 0; rep < 4; ++rep) {
        CK(cudaDeviceSynchronize());
        CK(cudaEventRecord(e0, 0));
        if (dir == 0) copy_kernel<<<blocks, 512>>>((const uint4*)hd, (uint4*)d, bytes / 16);
        else copy_kernel<<<blocks, 512>>>((const uint4*)d, (uint4*)hd, bytes / 16);
        CK(cudaGetLastError());
        CK(cudaEventRecord(e1, 0));
        CK(cudaEventSynchronize(e1));
        float ms = 0; CK(cudaEventElapsedTime(&ms, e0, e1));
        if (rep > 0 && ms < best) best = ms;
      }
      printf("%s kernel on mapped host memory, %d CTAs x 512: %.1f GB/s\n", dir ? "d2h" : "h2d", blocks, bytes / (best * 1e-3) / 1e9);
    }
  }
  // both directions at once: copy engines (h2d on stream 0, d2h on stream 1) on separate halves
  {
    const size_t half = bytes / 2;
    float best = 1e9f;
    for (int rep = 0; rep < 4; ++rep) {
      CK(cudaDeviceSynchronize());
      CK(cudaEventRecord(e0, 0));
      CK(cudaStreamWaitEvent(st[0], e0, 0)); CK(cudaStreamWaitEvent(st[1], e0, 0));
      CK(cudaMemcpyAsync(d, h, half, cudaMemcpyHostToDevice, st[0]));
      CK(cudaMemcpyAsync((char*)h + half, (char*)d + half, half, cudaMemcpyDeviceToHost, st[1]));
      for (int i = 0; i < 2; ++i) { cudaEvent_t ev; CK(cudaEventCreate(&ev)); CK(cudaEventRecord(ev, st[i])); CK(cudaStreamWaitEvent(0, ev, 0)); CK(cudaEventDestroy(ev)); }
      CK(cudaEventRecord(e1, 0));
      CK(cudaEventSynchronize(e1));
      float ms = 0; CK(cudaEventElapsedTime(&ms, e0, e1));
      if (rep > 0 && ms < best) best = ms;
    }
    printf("h2d + d2h at once (1 GiB each): %.1f GB/s combined\n", bytes / (best * 1e-3) / 1e9);
  }
  CK(cudaFreeHost(h)); CK(cudaFree(d));
  return 0;
}
