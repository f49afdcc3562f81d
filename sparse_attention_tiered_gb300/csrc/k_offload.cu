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

// KV append, one CTA per request of the layer. The new token of every KV head goes
// into row tail_n[b] of the unit's tail page (HBM, after the page pool). When the
// tail holds 64 tokens it becomes partition P = P_b[b]: its fp32 mean key (same
// arithmetic as summarize_offload_kernel) goes to the summaries, the page to the
// pinned host store, the tail page is cleared and the request's counts advance.
constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
append_kernel(LayerArgs a, const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
              int32_t* P_b, int32_t* ntok_b, int32_t* tail_n, float* __restrict__ summ, uint16_t* host_store) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int tn = tail_n[b];
  const int P = P_b[b];
  const bool full = tn + 1 == kPart;
  if (tn < 0 || tn >= kPart || (full && (P < 0 || P >= a.pstride_b[b]))) {  // the host never lets this happen
    if (tid == 0) atomicOr(a.err, kErrIndex);
    return;
  }
  const int64_t u0 = a.pool_slots + a.unit_base + (int64_t)b * a.Hkv;  // pool page of head 0's tail
  constexpr int kRowVec = kD / 8;                                       // 16-byte vectors per row
  for (int i = tid; i < a.Hkv * 2 * kRowVec; i += kAppendThreads) {
    const int h = i / (2 * kRowVec), half = (i / kRowVec) & 1, c = i % kRowVec;
    const uint4* src = reinterpret_cast<const uint4*>((half ? v_new : k_new) + ((int64_t)b * a.Hkv + h) * kD);
    uint4* dst = reinterpret_cast<uint4*>(a.pool + (u0 + h) * kPageElems + half * kPart * kD + (int64_t)tn * kD);
    dst[c] = src[c];
  }
  if (!full) {
    if (tid == 0) tail_n[b] = tn + 1;
    return;
  }
  __syncthreads();  // the new rows are visible to the whole CTA
  for (int i = tid; i < a.Hkv * kD; i += kAppendThreads) {
    const int h = i / kD, d = i % kD;
    const uint16_t* K = a.pool + (u0 + h) * kPageElems;
    float s = 0.f;
    for (int r = 0; r < kPart; ++r) s += bf16_bits_to_float(K[r * kD + d]);
    summ[host_page_index(a, b, h, P) * kD + d] = s / (float)kPart;
  }
  constexpr int kPageVec = kPageElems / 8;
  for (int i = tid; i < a.Hkv * kPageVec; i += kAppendThreads) {
    const int h = i / kPageVec, c = i % kPageVec;
    const uint4* src = reinterpret_cast<const uint4*>(a.pool + (u0 + h) * kPageElems);
    reinterpret_cast<uint4*>(host_store + host_page_index(a, b, h, P) * kPageElems)[c] = src[c];
  }
  __syncthreads();  // every read of the tail pages is done
  for (int i = tid; i < a.Hkv * kPageVec; i += kAppendThreads)
    reinterpret_cast<uint4*>(a.pool + (u0 + i / kPageVec) * kPageElems)[i % kPageVec] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    P_b[b] = P + 1;
    ntok_b[b] = (P + 1) * kPart;
    tail_n[b] = 0;
    atomicAdd(&a.stats[kStatFlushes], 1ull);
  }
}

__global__ void set_request_kernel(int32_t* P_b, int32_t* ntok_b, int32_t* tail_n, int32_t P, int32_t ntok,
                                   int32_t tail) {
  *P_b = P;
  *ntok_b = ntok;
  if (tail_n) *tail_n = tail;
}

// Variable partitions: one CTA per (partition, kv head). Partition p of head h holds the
// tokens order[h][starts[h][p]] .. order[h][starts[h][p+1] - 1] (1 to 64 of them, checked
// on the host); they go into the partition's page from row 0 in that order, zero padded,
// and its summary is their fp32 mean key, summed in row order as summarize_offload_kernel
// sums a block. k, v: [kv_heads][n_tokens][128].
__global__ void __launch_bounds__(kOffloadThreads)
gather_offload_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t n_tokens,
                      const int32_t* __restrict__ order, const int32_t* __restrict__ starts, int32_t n_parts,
                      float* __restrict__ summ_unit0, uint16_t* __restrict__ host_unit0, int64_t unit_pages,
                      uint8_t* __restrict__ valid_unit0) {
  __shared__ __align__(16) uint16_t ks[kPart * kD];
  __shared__ int32_t rows[kPart];
  const int p = blockIdx.x, h = blockIdx.y;
  const int32_t* st = starts + (int64_t)h * (n_parts + 1);
  const int j0 = st[p];
  const int cnt = st[p + 1] - j0;
  if (threadIdx.x < kPart) rows[threadIdx.x] = threadIdx.x < cnt ? order[(int64_t)h * n_tokens + j0 + threadIdx.x] : 0;
  __syncthreads();
  const uint16_t* kh = k + (int64_t)h * n_tokens * kD;
  const uint16_t* vh = v + (int64_t)h * n_tokens * kD;
  uint4* page = reinterpret_cast<uint4*>(host_unit0 + ((int64_t)h * unit_pages + p) * kPageElems);
  constexpr int kRowVec = kD / 8;                      // 16-byte vectors per row
  constexpr int kVecPerHalf = kPart * kRowVec;
  for (int i = threadIdx.x; i < kVecPerHalf; i += kOffloadThreads) {
    const int r = i / kRowVec, c = i % kRowVec;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < cnt) val = reinterpret_cast<const uint4*>(kh + (int64_t)rows[r] * kD)[c];
    reinterpret_cast<uint4*>(ks)[i] = val;
    page[i] = val;
  }
  for (int i = threadIdx.x; i < kVecPerHalf; i += kOffloadThreads) {
    const int r = i / kRowVec, c = i % kRowVec;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < cnt) val = reinterpret_cast<const uint4*>(vh + (int64_t)rows[r] * kD)[c];
    page[kVecPerHalf + i] = val;
  }
  __syncthreads();
  if (threadIdx.x < kD) {
    float s = 0.f;
    for (int r = 0; r < cnt; ++r) s += bf16_bits_to_float(ks[r * kD + threadIdx.x]);
    summ_unit0[((int64_t)h * unit_pages + p) * kD + threadIdx.x] = s / (float)cnt;
  }
  if (threadIdx.x == 0) valid_unit0[(int64_t)h * unit_pages + p] = (uint8_t)cnt;
}

// Read pass over the pinned host store: one 4-byte load every `stride` bytes.
// The first GPU read of a host page pays for translating its address, and those
// translations resolve at a limited rate (on GB300 machines, 45-100 GB/s of random
// 32 KiB pages read for the first time, against 200-210 GB/s once translated).
// Paying that once, in one dense pass, keeps it out of the decode steps' retrieval.
// The loaded words are summed and the sum is stored only when it equals `key`, so
// the loads cannot be dropped as dead code; the store almost never happens and
// goes to a scratch word nobody reads.
__global__ void warm_store_kernel(const uint8_t* __restrict__ store, int64_t n_reads, int64_t stride,
                                  uint32_t* __restrict__ sink, uint32_t key) {
  uint32_t acc = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_reads; i += (int64_t)gridDim.x * blockDim.x)
    acc += __ldcg(reinterpret_cast<const uint32_t*>(store + i * stride));
  if (acc == key) *sink = acc;
}

}  // namespace

cudaError_t launch_append(const LayerArgs& a, const uint16_t* k_new, const uint16_t* v_new, int32_t* P_b,
                          int32_t* ntok_b, int32_t* tail_n, cudaStream_t st) {
  append_kernel<<<a.B, kAppendThreads, 0, st>>>(a, k_new, v_new, P_b, ntok_b, tail_n, const_cast<float*>(a.summ),
                                               const_cast<uint16_t*>(a.host_store));
  return cudaGetLastError();
}

cudaError_t launch_set_request(int32_t* P_b, int32_t* ntok_b, int32_t* tail_n, int32_t P, int32_t ntok,
                               int32_t tail, cudaStream_t st) {
  set_request_kernel<<<1, 1, 0, st>>>(P_b, ntok_b, tail_n, P, ntok, tail);
  return cudaGetLastError();
}

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

cudaError_t launch_warm_store(const void* store, int64_t bytes, int64_t stride, uint32_t* sink, int sm_count,
                              cudaStream_t st) {
  if (!store || !sink || bytes <= 0 || stride <= 0) return cudaSuccess;
  const int64_t n_reads = bytes / stride;  // every read ends inside the store
  warm_store_kernel<<<(sm_count > 0 ? sm_count : 1) * 4, 256, 0, st>>>(static_cast<const uint8_t*>(store), n_reads,
                                                                        stride, sink, 0x9E3779B9u);
  return cudaGetLastError();
}

cudaError_t launch_gather_offload(const uint16_t* k, const uint16_t* v, int64_t n_tokens, int32_t kv_heads,
                                  const int32_t* order, const int32_t* starts, int32_t n_parts, float* summ_unit0,
                                  uint16_t* host_unit0, int64_t unit_pages, uint8_t* valid_unit0, cudaStream_t st) {
  if (n_tokens <= 0 || n_parts <= 0) return cudaSuccess;
  dim3 grid((unsigned)n_parts, (unsigned)kv_heads);
  gather_offload_kernel<<<grid, kOffloadThreads, 0, st>>>(k, v, n_tokens, order, starts, n_parts, summ_unit0,
                                                           host_unit0, unit_pages, valid_unit0);
  return cudaGetLastError();
}

}  // namespace spin
