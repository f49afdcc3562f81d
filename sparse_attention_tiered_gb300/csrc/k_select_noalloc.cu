// spin_select_noalloc: the Select step (fp32 scores + per-unit top-k) for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running while a CUDA graph is being
// captured, allocators that own every byte of the device (a serving engine's
// memory pool), or embedded hosts that forbid run-time allocation. Every other
// entry point of this library needs a context whose buffers spin_create
// allocates. This one takes only caller-owned inputs and outputs; the fp32 score
// array it needs between its two kernels lives in a fixed static device array
// (kNoAllocMaxScores floats = 4 MiB), which every CUDA context that loads this
// module holds until it is destroyed.
//
// The scores and the top-k are the decode step's own device code (select_dev.cuh:
// same summation order, same radix select and tie rule), so the result equals the
// selection a decode step makes for the same summaries and queries.
#include "../../include/spin.h"
#include "select_dev.cuh"
#include "spin_internal.cuh"

namespace spin {

void set_global_error(const char* msg);

namespace {

constexpr int64_t kNoAllocMaxScores = SPIN_NOALLOC_MAX_SCORES;
constexpr int kNoAllocMaxParts = 32768;

// The scratch: one score per (unit, partition) of the current call. Every call
// overwrites the entries it reads before reading them, so nothing has to be
// cleared between calls; calls that overlap on the GPU share it and race.
static __device__ __align__(256) float g_noalloc_scores[SPIN_NOALLOC_MAX_SCORES];

constexpr int kScoreWarps = 8;
constexpr int kScoreRows = kScoreWarps * sel::kRowsPerBatch;  // partitions per CTA

// grid (units, ceil(P / kScoreRows)); summ [units][P][128] fp32, q [units][G][128] bf16.
__global__ void __launch_bounds__(kScoreWarps * 32)
noalloc_score_kernel(const float* __restrict__ summ, const uint16_t* __restrict__ q, int P, int G,
                     float* __restrict__ scores) {
  const int u = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = blockIdx.y * kScoreRows + warp * sel::kRowsPerBatch;
  if (p0 >= P) return;
  const int n = min(sel::kRowsPerBatch, P - p0);
  float4 sv[sel::kRowsPerBatch];
  sel::load_rows(sv, reinterpret_cast<const float4*>(summ + ((int64_t)u * P + p0) * kD), n, lane);
  const float4 qv = sel::qsum_lane(q + (int64_t)u * G * kD, G, lane);
  const float x = sel::score_batch(sv, qv, lane);
  if (lane < n) scores[(int64_t)u * P + p0 + lane] = x;
}

constexpr int kTopkThreads = 512;

// Shared memory of the top-k kernel for P partitions: group scalars, keys [P], histograms,
// candidates (units wider than the wide-unit threshold).
__host__ __device__ inline size_t topk_smem_layout(int P, uint8_t* base, sel::GroupScalars** gs, uint32_t** keys,
                                                   uint32_t** whist, uint32_t** cand) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += sel::align16(bytes);
    return p;
  };
  uint8_t* g = take(sizeof(sel::GroupScalars));
  uint8_t* k = take(sizeof(uint32_t) * (size_t)P);
  uint8_t* w = take(sizeof(uint32_t) * (kTopkThreads / 32) * 256);
  const int cc = sel::cand_capacity(kTopkThreads, P);
  uint8_t* c = take(sizeof(uint32_t) * (size_t)(cc > 0 ? cc : 1));
  if (base) {
    *gs = (sel::GroupScalars*)g;
    *keys = (uint32_t*)k;
    *whist = (uint32_t*)w;
    *cand = (uint32_t*)c;
  }
  return off;
}

// One CTA per unit: the decode step's group top-k over the unit's keys; sel [units][k].
__global__ void __launch_bounds__(kTopkThreads)
noalloc_topk_kernel(const float* __restrict__ scores, int P, int k, int32_t* __restrict__ sel_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  sel::GroupScalars* gs;
  uint32_t *keys, *whist, *cand;
  topk_smem_layout(P, smem_raw, &gs, &keys, &whist, &cand);
  const int tid = threadIdx.x;
  const int u = blockIdx.x;
  const int keff = P < k ? P : k;
  for (int p = tid; p < P; p += kTopkThreads) keys[p] = sel::float_key(scores[(int64_t)u * P + p]);
  __syncthreads();
  int32_t* out = sel_out + (int64_t)u * k;
  __shared__ int32_t s_sel[kMaxTopk];
  const bool ok = sel::group_topk<kTopkThreads>(keys, P, keff, whist, cand, sel::cand_capacity(kTopkThreads, P), gs,
                                                1, tid, s_sel);
  for (int j = tid; j < k; j += kTopkThreads) out[j] = (ok && j < keff) ? s_sel[j] : -1;
}

size_t topk_smem_bytes(int P) { return topk_smem_layout(P, nullptr, nullptr, nullptr, nullptr, nullptr); }

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
  if ((reinterpret_cast<uintptr_t>(summ) & 15) || (reinterpret_cast<uintptr_t>(q) & 7) ||
      (reinterpret_cast<uintptr_t>(sel) & 3)) {
    set_global_error("spin_select_noalloc: summ must be 16-byte, q 8-byte and sel 4-byte aligned");
    return SPIN_ERR_INVALID;
  }
  // An error left by earlier, unrelated work would be reported as this call's launch
  // failure; report it as what it is and launch nothing.
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error("spin_select_noalloc: a CUDA error from earlier work was pending; nothing was launched");
    return SPIN_ERR_CUDA;
  }
  // The device address of the static scratch in the current context (the host-side
  // symbol is only a stand-in for it). Looked up on every call, so the address always
  // belongs to the context the kernels run in; the first lookup in a context loads this
  // module, which reserves the array.
  void* scratch = nullptr;
  e = cudaGetSymbolAddress(&scratch, g_noalloc_scores);
  if (e != cudaSuccess || !scratch) {
    cudaGetLastError();
    set_global_error("spin_select_noalloc: cudaGetSymbolAddress of the static score scratch failed");
    return SPIN_ERR_CUDA;
  }
  const size_t smem = topk_smem_bytes(parts);
  e = cudaFuncSetAttribute(noalloc_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_global_error("spin_select_noalloc: configuring the top-k kernel failed");
    return SPIN_ERR_CUDA;
  }
  float* scores = static_cast<float*>(scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dim3 g1((unsigned)units, (unsigned)((parts + kScoreRows - 1) / kScoreRows));
  noalloc_score_kernel<<<g1, kScoreWarps * 32, 0, st>>>(summ, q, parts, group, scores);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error("spin_select_noalloc: launching the score kernel failed; the top-k kernel was not launched");
    return SPIN_ERR_CUDA;
  }
  noalloc_topk_kernel<<<(unsigned)units, kTopkThreads, smem, st>>>(scores, parts, topk, sel);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error("spin_select_noalloc: launching the top-k kernel failed");
    return SPIN_ERR_CUDA;
  }
  return SPIN_OK;
}
