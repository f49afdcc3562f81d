// spin_select_noalloc: the Select step (fp32 scores + per-unit top-k) for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running while a CUDA graph is being
// captured, allocators that own every byte of the device (a serving engine's
// memory pool), or embedded hosts that forbid run-time allocation. Every other
// entry point of this library needs a context whose buffers spin_create
// allocates. This one takes only caller-owned inputs and outputs; the fp32 score
// array it needs between its two kernels lives in a fixed static device array
// (kNoAllocMaxScores floats = 4 MiB), which every GPU that loads the library
// holds until the process exits.
//
// The arithmetic matches the decode step's Select exactly (same summation
// order, same radix top-k and tie rule), so its result equals the selection a
// decode step makes for the same summaries and queries.
#include <mutex>

#include "../../include/spin.h"
#include "spin_internal.cuh"

namespace spin {

void set_global_error(const char* msg);

namespace {

constexpr int64_t kNoAllocMaxScores = SPIN_NOALLOC_MAX_SCORES;
constexpr int kNoAllocMaxParts = 32768;
constexpr int kMaxDevices = 64;

// The scratch: one score per (unit, partition) of the current call. Every call
// overwrites the entries it reads before reading them, so nothing has to be
// cleared between calls; calls that overlap on the GPU share it and race.
static __device__ __align__(256) float g_noalloc_scores[SPIN_NOALLOC_MAX_SCORES];

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

constexpr int kScoreThreads = 256;
constexpr int kScorePerWarp = 8;
constexpr int kScoreChunk = (kScoreThreads / 32) * kScorePerWarp;

// grid (units, ceil(P / 64)); summ [units][P][128] fp32, q [units][G][128] bf16.
__global__ void __launch_bounds__(kScoreThreads)
noalloc_score_kernel(const float* __restrict__ summ, const uint16_t* __restrict__ q, int P, int G,
                     float* __restrict__ scores) {
  const int u = blockIdx.x;
  const int p_base = blockIdx.y * kScoreChunk;
  __shared__ __align__(16) float qs[kD];
  if (threadIdx.x < kD) {
    const uint16_t* qq = q + (int64_t)u * G * kD + threadIdx.x;
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += bf16f(qq[g * kD]);
    qs[threadIdx.x] = s;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float4 qv = reinterpret_cast<const float4*>(qs)[lane];
  const float4* su = reinterpret_cast<const float4*>(summ + (int64_t)u * P * kD);
  const int p0 = p_base + warp * kScorePerWarp;
  float4 sv[kScorePerWarp];
#pragma unroll
  for (int i = 0; i < kScorePerWarp; ++i) {
    const int p = p0 + i;
    sv[i] = p < P ? __ldg(su + (int64_t)p * (kD / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float d[kScorePerWarp];
#pragma unroll
  for (int i = 0; i < kScorePerWarp; ++i) {
    float x = sv[i].x * qv.x;
    x = fmaf(sv[i].y, qv.y, x);
    x = fmaf(sv[i].z, qv.z, x);
    x = fmaf(sv[i].w, qv.w, x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    d[i] = x;
  }
  if (lane < kScorePerWarp) {
    float x = d[0];
#pragma unroll
    for (int i = 1; i < kScorePerWarp; ++i) x = (lane == i) ? d[i] : x;
    const int p = p0 + lane;
    if (p < P) scores[(int64_t)u * P + p] = (x == 0.f) ? 0.f : x;
  }
}

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;

// One CTA per unit: radix select of the k-th largest key, then compaction in
// ascending partition order with equal keys taken from the lowest index up.
__global__ void __launch_bounds__(kTopkThreads)
noalloc_topk_kernel(const float* __restrict__ scores, int P, int k, int32_t* __restrict__ sel) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* whist = reinterpret_cast<uint32_t*>(smem_raw);   // [kTopkWarps][256]
  uint32_t* keys = whist + kTopkWarps * 256;                   // [P]
  __shared__ int s_bin, s_above;
  __shared__ int s_wgt[kTopkWarps], s_weq[kTopkWarps], s_wpos[kTopkWarps], s_wtake[kTopkWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x;
  const int keff = P < k ? P : k;
  for (int p = tid; p < P; p += kTopkThreads) keys[p] = float_key(scores[(int64_t)u * P + p]);
  uint32_t prefix = 0, mask = 0;
  int krem = keff;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) whist[i] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += kTopkThreads) {
      const uint32_t key = keys[p];
      if ((key & mask) == prefix) atomicAdd(&whist[warp * 256 + ((key >> shift) & 255u)], 1u);
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t s = 0;
      for (int w = 0; w < kTopkWarps; ++w) s += whist[w * 256 + tid];
      whist[tid] = s;
    }
    __syncthreads();
    if (warp == 0) {
      int c[8], lsum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = (int)whist[255 - 8 * lane - i];
        lsum += c[i];
      }
      int incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - lsum;
      const uint32_t hitm = __ballot_sync(0xffffffffu, excl < krem && incl >= krem);
      if (lane == __ffs(hitm) - 1) {
        int above = excl;
        for (int i = 0; i < 8; ++i) {
          if (above + c[i] >= krem) {
            s_bin = 255 - 8 * lane - i;
            s_above = above;
            break;
          }
          above += c[i];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s_bin << shift;
    mask |= 0xFFu << shift;
    krem -= s_above;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int chunk = ((P + kTopkThreads - 1) / kTopkThreads) * 32;
  const int wb = warp * chunk, we = min(P, wb + chunk);
  int gt = 0, eq = 0;
  for (int base = wb; base < we; base += 32) {
    const int p = base + lane;
    const uint32_t key = p < we ? keys[p] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, p < we && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, p < we && key == T));
  }
  if (lane == 0) {
    s_wgt[warp] = gt;
    s_weq[warp] = eq;
  }
  __syncthreads();
  if (tid == 0) {
    int eq_before = 0, pos = 0;
    for (int w = 0; w < kTopkWarps; ++w) {
      const int take = max(0, min(krem - eq_before, s_weq[w]));
      s_wpos[w] = pos;
      s_wtake[w] = take;
      pos += s_wgt[w] + take;
      eq_before += s_weq[w];
    }
  }
  __syncthreads();
  int32_t* out = sel + (int64_t)u * k;
  int pos = s_wpos[warp], eq_left = s_wtake[warp];
  for (int base = wb; base < we; base += 32) {
    const int p = base + lane;
    const uint32_t key = p < we ? keys[p] : 0u;
    const bool isgt = p < we && key > T;
    const bool iseq = p < we && key == T;
    const uint32_t meq = __ballot_sync(0xffffffffu, iseq);
    const bool take = isgt || (iseq && __popc(meq & lanemask_lt()) < eq_left);
    const uint32_t msel = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(msel & lanemask_lt())] = p;
    pos += __popc(msel);
    eq_left -= min(eq_left, __popc(meq));
  }
  for (int j = keff + tid; j < k; j += kTopkThreads) out[j] = -1;
}

struct DeviceScratch {
  bool ready = false;
  float* scores = nullptr;  // device address of g_noalloc_scores on that device
};
DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Once per device, with that device current: the device address of the static
// scratch (the host-side symbol is only a stand-in) and the top-k kernel's
// shared-memory limit.
int scratch_for_current_device(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    set_global_error("spin_select_noalloc: no usable current CUDA device");
    return SPIN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  DeviceScratch& s = g_scratch[dev];
  if (!s.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scores);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_global_error("spin_select_noalloc: cudaGetSymbolAddress of the static score scratch failed");
      return SPIN_ERR_CUDA;
    }
    const int smem = (int)(sizeof(uint32_t) * (kTopkWarps * 256 + kNoAllocMaxParts));
    e = cudaFuncSetAttribute(noalloc_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_global_error("spin_select_noalloc: configuring the top-k kernel failed");
      return SPIN_ERR_CUDA;
    }
    s.scores = static_cast<float*>(p);
    s.ready = true;
  }
  *out = s.scores;
  return SPIN_OK;
}

}  // namespace
}  // namespace spin

extern "C" int spin_select_noalloc(const float* summ, const uint16_t* q, int32_t units, int32_t parts, int32_t group,
                                   int32_t topk, int32_t* sel, spin_stream_t stream) {
  using namespace spin;
  if (!summ || !q || !sel) {
    set_global_error("spin_select_noalloc: summ, q and sel must be non-NULL device pointers");
    return SPIN_ERR_INVALID;
  }
  if (units < 1 || parts < 1 || group < 1 || group > kMaxGroup || topk < 1 || topk > kMaxTopk) {
    set_global_error("spin_select_noalloc: need units >= 1, parts >= 1, 1 <= group <= 16, 1 <= topk <= 512");
    return SPIN_ERR_INVALID;
  }
  if (parts > kNoAllocMaxParts || (int64_t)units * parts > kNoAllocMaxScores) {
    set_global_error("spin_select_noalloc: units * parts exceeds the static scratch of SPIN_NOALLOC_MAX_SCORES "
                     "scores (or parts > 32768)");
    return SPIN_ERR_INVALID;
  }
  if ((reinterpret_cast<uintptr_t>(summ) & 15) || (reinterpret_cast<uintptr_t>(q) & 1) ||
      (reinterpret_cast<uintptr_t>(sel) & 3)) {
    set_global_error("spin_select_noalloc: summ must be 16-byte, q 2-byte and sel 4-byte aligned");
    return SPIN_ERR_INVALID;
  }
  float* scores = nullptr;
  int rc = scratch_for_current_device(&scores);
  if (rc != SPIN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dim3 g1((unsigned)units, (unsigned)((parts + kScoreChunk - 1) / kScoreChunk));
  noalloc_score_kernel<<<g1, kScoreThreads, 0, st>>>(summ, q, parts, group, scores);
  const size_t smem = sizeof(uint32_t) * (kTopkWarps * 256 + (size_t)parts);
  noalloc_topk_kernel<<<(unsigned)units, kTopkThreads, smem, st>>>(scores, parts, topk, sel);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error("spin_select_noalloc: kernel launch failed");
    return SPIN_ERR_CUDA;
  }
  return SPIN_OK;
}
