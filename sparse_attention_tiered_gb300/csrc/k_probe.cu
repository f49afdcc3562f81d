// Host-link probe: the rate at which the SMs stream pinned host memory with 16-byte
// zero-copy loads (the retrievers' access path). The SPIN pages measure their
// systems against an ideal envelope that assumes retrieval at the link's peak
// (m.x-techcon.com SPIN article, section "理想与现实的差距", Figure 1); this gives the
// link's peak for reads issued by the GPU itself, next to copy-engine copies.
#include "../../include/spin.h"
#include "spin_internal.cuh"

namespace spin {

void set_global_error(const char* msg);

namespace {

// Written only when the folded words hit a key, so the loads cannot be dropped.
__device__ uint32_t g_probe_sink;

__global__ void __launch_bounds__(512) host_read_kernel(const uint4* __restrict__ src, int64_t nvec) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < nvec; i += 8 * stride) {
    uint4 r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) r[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= r[u].x ^ r[u].y ^ r[u].z ^ r[u].w;
  }
  for (; i < nvec; i += stride) {
    const uint4 r = __ldcs(src + i);
    acc ^= r.x ^ r.y ^ r.z ^ r.w;
  }
  if (acc == 0x9E3779B9u) g_probe_sink = acc;
}

}  // namespace
}  // namespace spin

extern "C" int spin_measure_host_read(const void* host, int64_t bytes, int32_t ctas_per_sm, double* gbs,
                                      spin_stream_t stream) {
  using namespace spin;
  if (!host || !gbs || bytes < 16 || (reinterpret_cast<uintptr_t>(host) & 15) || ctas_per_sm < 1 || ctas_per_sm > 4) {
    set_global_error("spin_measure_host_read: need a 16-byte aligned host buffer of >= 16 bytes, gbs != NULL and "
                     "1 <= ctas_per_sm <= 4");
    return SPIN_ERR_INVALID;
  }
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, host) != cudaSuccess || pa.type != cudaMemoryTypeHost || !pa.devicePointer) {
    cudaGetLastError();
    set_global_error("spin_measure_host_read: the buffer is not pinned host memory mapped for the device");
    return SPIN_ERR_INVALID;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    set_global_error("spin_measure_host_read: no usable CUDA device");
    return SPIN_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    if (e0) cudaEventDestroy(e0);
    set_global_error("spin_measure_host_read: creating events failed");
    return SPIN_ERR_CUDA;
  }
  const uint4* src = static_cast<const uint4*>(pa.devicePointer);
  const int64_t nvec = bytes / 16;
  const unsigned grid = (unsigned)(sms * ctas_per_sm);
  host_read_kernel<<<grid, 512, 0, st>>>(src, nvec);  // first pass: address translations
  cudaEventRecord(e0, st);
  host_read_kernel<<<grid, 512, 0, st>>>(src, nvec);
  cudaEventRecord(e1, st);
  cudaError_t e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess || ms <= 0.f) {
    cudaGetLastError();
    set_global_error("spin_measure_host_read: the timed read failed");
    return SPIN_ERR_CUDA;
  }
  *gbs = (double)(nvec * 16) / (ms * 1e-3) / 1e9;
  return SPIN_OK;
}
