// Index + Offload: partition summaries and page-format copy into pinned host memory.
//
// SPIN splits prefill-time work into Index (the algorithm organises the KV of a
// head into partitions and produces a summary per partition) and Offload (the
// system places the partitions in CPU memory): m.x-techcon.com SPIN article,
// section "Spin的核心设计" 1 (统一的分区抽象) and Figure 3; gist.science/pt,
// section 2A. The pages do not fix the summary; this library uses the mean key
// of the partition's valid tokens, in fp32.
#include "spin_internal.cuh"

namespace spin {

namespace {

constexpr int kOffloadThreads = 256;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// One CTA per (partition in chunk, kv head). k, v: [kv_heads][head_stride tokens][128],
// starting at absolute token tok0; ntok_total = the request's token count.
__global__ void __launch_bounds__(kOffloadThreads)
summarize_offload_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t head_stride,
                         int64_t tok0, int64_t ntok_total, float* __restrict__ summ_unit0,
                         uint16_t* __restrict__ host_unit0, int64_t unit_pages) {
  __shared__ __align__(16) uint16_t ks[kPart * kD];
  const int h = blockIdx.y;
  const int64_t p = tok0 / kPart + blockIdx.x;
  const int64_t row0 = p * kPart;                       // absolute first token of the partition
  const int64_t rem = ntok_total - row0;
  const int valid = rem < kPart ? (int)rem : kPart;
  const uint16_t* ksrc = k + ((int64_t)h * head_stride + (row0 - tok0)) * kD;
  const uint16_t* vsrc = v + ((int64_t)h * head_stride + (row0 - tok0)) * kD;
  uint4* page = reinterpret_cast<uint4*>(host_unit0 + ((int64_t)h * unit_pages + p) * kPageElems);

  // K half: stage in shared memory (for the summary) and write to the host page.
  constexpr int kVecPerHalf = kPart * kD / 8;          // 1024 x 16 B
  for (int i = threadIdx.x; i < kVecPerHalf; i += kOffloadThreads) {
    const int r = i / (kD / 8);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < valid) val = reinterpret_cast<const uint4*>(ksrc)[i];
    reinterpret_cast<uint4*>(ks)[i] = val;
    page[i] = val;
  }
  // V half: straight copy.
  for (int i = threadIdx.x; i < kVecPerHalf; i += kOffloadThreads) {
    const int r = i / (kD / 8);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < valid) val = reinterpret_cast<const uint4*>(vsrc)[i];
    page[kVecPerHalf + i] = val;
  }
  __syncthreads();
  if (threadIdx.x < kD) {
    float s = 0.f;
    for (int r = 0; r < valid; ++r) s += bf16_bits_to_float(ks[r * kD + threadIdx.x]);
    summ_unit0[((int64_t)h * unit_pages + p) * kD + threadIdx.x] = s / (float)valid;
  }
}

}  // namespace

cudaError_t launch_summarize_offload(const uint16_t* k, const uint16_t* v, int64_t head_stride, int32_t kv_heads,
                                     int64_t tok0, int64_t ntok_chunk, int64_t ntok_total, float* summ_unit0,
                                     uint16_t* host_unit0, int64_t unit_pages, cudaStream_t st) {
  if (ntok_chunk <= 0) return cudaSuccess;
  const int64_t parts = (ntok_chunk + kPart - 1) / kPart;
  dim3 grid((unsigned)parts, (unsigned)kv_heads);
  summarize_offload_kernel<<<grid, kOffloadThreads, 0, st>>>(k, v, head_stride, tok0, ntok_total, summ_unit0,
                                                              host_unit0, unit_pages);
  return cudaGetLastError();
}

}  // namespace spin
