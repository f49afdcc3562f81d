// Host runtime and C ABI of the SPIN sparse-decode library (see include/spin.h).
//
// Owns the memory tiers and metadata of the method (m.x-techcon.com SPIN article,
// section "Spin的核心设计" 2 and 3, Figures 5 and 6; gist.science/pt section 2B-C):
//   * pinned, device-mapped host page store: every page of every unit (Offload);
//   * HBM page pool: cap = buf_mult * k pages per unit (mandatory + buffer pages);
//   * two-level page table: a static directory [units][ceil(Pmax/64)] whose
//     entries point to 64-entry segments drawn on demand from one shared pool;
//   * per-page state: slot -> partition, last-use step (bucketed-LRU timestamps);
//   * fp32 partition summaries in HBM;
//   * with variable partitions (max_partitions > 0), one token count per host page.
// A decode step of one layer is one cooperative kernel on the caller's stream
// (score -> select + manage -> retrieve + attention -> combine); the first step after
// an offload call adds one read pass over the host store before it. A KV append (spin_append_kv, tail mode) is a kernel of its own that the
// caller enqueues before the step.
#include <cuda.h>
#include <cuda_runtime.h>

#include <sys/mman.h>
#include <unistd.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/spin.h"
#include "spin_internal.cuh"

using namespace spin;

namespace {

thread_local std::string g_create_error;

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct LayerBuf {
  float* scores = nullptr;
  int32_t* sel = nullptr;
  int32_t* sel_slot = nullptr;
  uint8_t* sel_hit = nullptr;
  int32_t* keff = nullptr;
  int32_t* unit_info = nullptr;
  int64_t* miss_src = nullptr;
  int64_t* miss_dst = nullptr;
  int32_t* miss_att = nullptr;
  int32_t* miss_valid = nullptr;
  int32_t* ready = nullptr;
  uint32_t* ready_cnt = nullptr;
  int32_t* miss_tag = nullptr;
  int32_t* unit_rows = nullptr;
  int32_t* unit_ready = nullptr;
  int32_t* hist12 = nullptr;
  int32_t* att_slot = nullptr;
  int32_t* att_valid = nullptr;
  int32_t* n_hit = nullptr;
  int32_t* counters = nullptr;
  float* partials = nullptr;
  uint16_t* q_stage = nullptr;  // for the host-buffer entry point
  float* out_stage = nullptr;
  LayerArgs args{};
};

constexpr int kNumStages = 5;  // score, manage, pages (retrieval + attention), combine, whole kernel
constexpr int kPipeGroupFirst = 128;  // threads of a manager group the pipelined kernel tries first
constexpr int kTimelineCalls = 4096;  // stage-stamp records of timed calls between two synchronisations

// One timed call: CUDA events around the kernel and the slot of its stage stamps.
struct TimedCall {
  cudaEvent_t ev[2];
  int rec;
};

}  // namespace

struct spin_ctx {
  // configuration
  int device = 0;
  uint32_t flags = 0;
  int B = 0, L = 0, Hq = 0, Hkv = 0, G = 0, k = 0, cap = 0, D = 0, P_max = 0, ppt = 1, n_chunks = 1;
  int sm_count = 0;
  int retr_warps = 2;  // retriever warps per CTA from the start of the retrieval phase
  int retr_late = 4;   // retriever warps that join after the CTA's resident pages are issued
  int mgr_gs = 512;    // threads of one manager group
  int pipe = 0;        // 1: the pipelined decode-step kernel
  int retr_split = 0;  // miss-list entries of a step copied in kRetrChunks pieces (the first ones)
  int store_warm = 1;          // read passes over the host store after it is written
  bool store_cold = false;     // the store was written since its last read pass
  int64_t warm_stride = 32768; // bytes between the read pass's loads: the host page size, at most 32 KiB
  std::vector<int64_t> ctx_len;
  std::vector<int32_t> P_b, ntok_b;  // fixed mode: partitions and tokens of each request
  std::vector<int32_t> pstride_b;    // host-store pages per KV head of each request (its partition capacity)
  std::vector<int64_t> poff_b;
  // tail mode (append_tokens > 0): per-(layer, request) complete partitions and tail tokens,
  // mirrored on the host (every append adds exactly one token, so the host knows them)
  bool tail_mode = false;
  // variable partitions (max_partitions > 0): every request has room for max_partitions per KV
  // head; part_valid holds each page's token count; the grouping is staged in HBM
  bool part_mode = false;
  int32_t max_partitions = 0;
  uint8_t* d_part_valid = nullptr;
  int32_t* d_gorder = nullptr;   // [Hkv][max ctx_len]
  int32_t* d_gstarts = nullptr;  // [Hkv][max_partitions + 1]
  uint16_t *d_gk = nullptr, *d_gv = nullptr;  // host-source staging, [Hkv][max ctx_len][128]
  int64_t append_tokens = 0, appended = 0;
  int ka = 0;  // attention entries per unit
  std::vector<int32_t> P_lb, tail_lb;
  int64_t pages_per_layer = 0, units = 0, S = 0;
  // memory
  std::vector<void*> dev_allocs;
  uint16_t* h_store = nullptr;  // pinned host page store
  size_t h_store_map_len = 0;   // > 0: h_store is a registered anonymous mapping of this length
  uint16_t* d_store = nullptr;  // its device-usable address
  uint16_t* d_pool = nullptr;
  float* d_summ = nullptr;
  int32_t *d_P_lb = nullptr, *d_ntok_lb = nullptr, *d_tail_lb = nullptr;  // [L][B]
  int32_t* d_pstride_b = nullptr;
  int32_t* d_budget_b = nullptr;  // [B] resident budget per unit of each request
  int64_t* d_poff_b = nullptr;
  int32_t *d_dir = nullptr, *d_seg = nullptr, *d_seg_live = nullptr;
  int32_t* h_seg = nullptr;  // tier split: the segment entries in pinned host memory (d_seg maps it)
  uint32_t* d_bitmap = nullptr;
  int32_t *d_slot_part = nullptr, *d_last_use = nullptr;
  unsigned long long* d_stats = nullptr;
  uint32_t* d_err = nullptr;
  uint32_t* d_warm_sink = nullptr;  // the read pass's sink word (written only if a sum hits its key)
  uint16_t *d_stage_k = nullptr, *d_stage_v = nullptr;
  int64_t stage_tokens = 0;
  std::vector<LayerBuf> layers;
  CUtensorMap tmap{};
  std::vector<uint8_t> offloaded;  // [L][B]
  int64_t steps_host = 0;
  std::vector<int64_t> layer_steps;  // decode steps enqueued per layer (the kernel's step counter)
  uint32_t sticky = 0;
  std::string msg;
  // stage timing
  std::vector<TimedCall> pending;
  std::vector<cudaEvent_t> spare_events;
  unsigned long long* d_timeline = nullptr;  // [kTimelineCalls][kTlSlots]
  int next_rec = 0;
  double ms[kNumStages] = {0, 0, 0, 0, 0};
  int64_t timed_calls = 0;
  int64_t bytes_meta = 0, bytes_flat = 0, bytes_pool = 0, bytes_store = 0, bytes_summ = 0;
  int64_t P_logical = 0;  // partitions per unit of the logical capacity (max_context)
};

namespace {

int fail(spin_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) c->msg = buf;
  else g_create_error = buf;
  return code;
}

int cuda_fail(spin_ctx* c, cudaError_t e, const char* what) {
  cudaGetLastError();
  return fail(c, e == cudaErrorMemoryAllocation ? SPIN_ERR_OOM : SPIN_ERR_CUDA, "%s: %s", what,
              cudaGetErrorString(e));
}

#define SPIN_CUDA(c, call, what)                  \
  do {                                            \
    cudaError_t e_ = (call);                      \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, what); \
  } while (0)

template <typename T>
cudaError_t dalloc(spin_ctx* c, T** p, size_t count) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, std::max<size_t>(count, 1) * sizeof(T));
  if (e != cudaSuccess) return e;
  c->dev_allocs.push_back(v);
  *p = static_cast<T*>(v);
  return cudaSuccess;
}

void free_all(spin_ctx* c) {
  for (void* p : c->dev_allocs) cudaFree(p);
  c->dev_allocs.clear();
  if (c->h_store) {
    if (c->h_store_map_len) {
      cudaHostUnregister(c->h_store);
      munmap(c->h_store, c->h_store_map_len);
    } else {
      cudaFreeHost(c->h_store);
    }
  }
  c->h_store = nullptr;
  c->h_store_map_len = 0;
  if (c->h_seg) cudaFreeHost(c->h_seg);
  c->h_seg = nullptr;
  for (auto& t : c->pending)
    for (auto e : t.ev) cudaEventDestroy(e);
  c->pending.clear();
  for (auto e : c->spare_events) cudaEventDestroy(e);
  c->spare_events.clear();
}

// Size of a transparent huge page (PMD size); 2 MiB when the kernel does not say.
size_t thp_bytes() {
  size_t v = 0;
  if (FILE* f = fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    unsigned long long x = 0;
    if (fscanf(f, "%llu", &x) == 1) v = (size_t)x;
    fclose(f);
  }
  return (v >= 4096 && (v & (v - 1)) == 0 && v <= ((size_t)1 << 30)) ? v : ((size_t)2 << 20);
}

// Pinned, device-mapped host memory from an anonymous mapping aligned to the huge-page
// size and advised to use transparent huge pages, then registered with CUDA (large host
// pages mean few address translations for the GPU's random page reads). nullptr when
// any step fails.
void* alloc_host_hugepages(size_t bytes, size_t* map_len) {
  const size_t hp = thp_bytes();
  const size_t len = (bytes + hp - 1) / hp * hp;
  void* m = mmap(nullptr, len + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (m == MAP_FAILED) return nullptr;
  const uintptr_t base = reinterpret_cast<uintptr_t>(m);
  const uintptr_t aligned = (base + hp - 1) / hp * hp;
  if (aligned > base) munmap(m, aligned - base);                       // leading remainder
  const size_t tail = (base + len + hp) - (aligned + len);
  if (tail) munmap(reinterpret_cast<void*>(aligned + len), tail);      // trailing remainder
  void* p = reinterpret_cast<void*>(aligned);
  (void)madvise(p, len, MADV_HUGEPAGE);  // advisory: no effect where huge pages are off
  if (cudaHostRegister(p, len, cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess) {
    cudaGetLastError();
    munmap(p, len);
    return nullptr;
  }
  *map_len = len;
  return p;
}

int check_device_error(spin_ctx* c) {
  if (!c->sticky) {
    uint32_t e = 0;
    if (cudaMemcpy(&e, c->d_err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess)
      return cuda_fail(c, cudaGetLastError(), "reading the device error word");
    c->sticky = e;
  }
  if (c->sticky & kErrCapacity)
    return fail(c, SPIN_ERR_CAPACITY, "the shared second-level segment pool ran out (device error 0x%x)", c->sticky);
  if (c->sticky & kErrTimeout)
    return fail(c, SPIN_ERR_TIMEOUT, "a bounded device wait ran out (device error 0x%x)", c->sticky);
  if (c->sticky) return fail(c, SPIN_ERR_CUDA, "device invariant check failed (error word 0x%x)", c->sticky);
  return SPIN_OK;
}

int sync_ctx(spin_ctx* c) {
  SPIN_CUDA(c, cudaDeviceSynchronize(), "synchronising the device");
  // fold finished stage timings
  if (!c->pending.empty()) {
    std::vector<unsigned long long> tl((size_t)kTimelineCalls * kTlSlots);
    SPIN_CUDA(c, cudaMemcpy(tl.data(), c->d_timeline, tl.size() * 8, cudaMemcpyDeviceToHost), "reading stage stamps");
    for (auto& t : c->pending) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, t.ev[0], t.ev[1]) == cudaSuccess) c->ms[4] += ms;
      const unsigned long long* r = tl.data() + (size_t)t.rec * kTlSlots;
      const unsigned long long t0 = ~r[kTlStart];
      auto seg = [&](unsigned long long from, unsigned long long to) {
        return (to > from && from != 0) ? (double)(to - from) * 1e-6 : 0.0;
      };
      // consecutive stamps of the critical path: scoring done, last unit published,
      // last page attended, last combine done
      const unsigned long long s1 = r[kTlScored], s2 = std::max(r[kTlManaged], s1), s3 = std::max(r[kTlPages], s2),
                               s4 = std::max(r[kTlEnd], s3);
      c->ms[0] += seg(t0, s1);
      c->ms[1] += seg(s1, s2);
      c->ms[2] += seg(s2, s3);
      c->ms[3] += seg(s3, s4);
      for (auto e : t.ev) c->spare_events.push_back(e);
    }
    c->pending.clear();
    SPIN_CUDA(c, cudaMemset(c->d_timeline, 0, (size_t)kTimelineCalls * kTlSlots * 8), "clearing stage stamps");
    c->next_rec = 0;
  }
  return check_device_error(c);
}

int encode_tensor_map(spin_ctx* c) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return fail(c, SPIN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t slots = (uint64_t)c->units * (uint64_t)c->cap + (c->tail_mode ? (uint64_t)c->units : 0u);
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)(slots * 128)};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = reinterpret_cast<EncodeTiledFn>(fn)(&c->tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->d_pool, dims,
                                                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(c, SPIN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SPIN_OK;
}

int get_event(spin_ctx* c, cudaEvent_t* e) {
  if (!c->spare_events.empty()) {
    *e = c->spare_events.back();
    c->spare_events.pop_back();
    return SPIN_OK;
  }
  SPIN_CUDA(c, cudaEventCreate(e), "creating a timing event");
  return SPIN_OK;
}

int validate(const spin_config* cfg) {
  if (!cfg) return fail(nullptr, SPIN_ERR_INVALID, "cfg is NULL");
  if (cfg->batch < 1 || cfg->layers < 1 || cfg->kv_heads < 1 || cfg->q_heads < 1)
    return fail(nullptr, SPIN_ERR_INVALID, "batch, layers, q_heads and kv_heads must be >= 1");
  if (cfg->batch > 16384) return fail(nullptr, SPIN_ERR_INVALID, "batch must be <= 16384");
  if (cfg->q_heads % cfg->kv_heads != 0 || cfg->q_heads / cfg->kv_heads > kMaxGroup)
    return fail(nullptr, SPIN_ERR_INVALID, "q_heads must be a multiple of kv_heads with a group of at most %d",
                kMaxGroup);
  if (cfg->head_dim != kD) return fail(nullptr, SPIN_ERR_INVALID, "head_dim must be %d", kD);
  if (cfg->part_tokens != kPart) return fail(nullptr, SPIN_ERR_INVALID, "part_tokens must be %d", kPart);
  if (cfg->seg_entries != 0 && cfg->seg_entries != kSeg)
    return fail(nullptr, SPIN_ERR_INVALID, "seg_entries must be 0 or %d", kSeg);
  if (cfg->topk < 1 || cfg->topk > kMaxTopk) return fail(nullptr, SPIN_ERR_INVALID, "topk must be in [1, %d]", kMaxTopk);
  if (cfg->buf_mult < 1 || (int64_t)cfg->buf_mult * cfg->topk > 8192)
    return fail(nullptr, SPIN_ERR_INVALID, "buf_mult must be >= 1 with buf_mult * topk <= 8192");
  if (!cfg->ctx_len) return fail(nullptr, SPIN_ERR_INVALID, "ctx_len is NULL");
  if (cfg->append_tokens < 0) return fail(nullptr, SPIN_ERR_INVALID, "append_tokens must be >= 0");
  for (int b = 0; b < cfg->batch; ++b) {
    if (cfg->ctx_len[b] < 0 || cfg->ctx_len[b] + cfg->append_tokens > (int64_t)32768 * kPart)
      return fail(nullptr, SPIN_ERR_INVALID, "ctx_len[%d] + append_tokens = %lld outside [0, %d]", b,
                  (long long)(cfg->ctx_len[b] + cfg->append_tokens), 32768 * kPart);
  }
  if (cfg->max_partitions < 0 || cfg->max_partitions > (1 << 20))
    return fail(nullptr, SPIN_ERR_INVALID, "max_partitions must be in [0, 2^20]");
  if (cfg->max_partitions > 0) {
    if (cfg->append_tokens > 0)
      return fail(nullptr, SPIN_ERR_INVALID, "variable partitions (max_partitions > 0) need append_tokens == 0");
    for (int b = 0; b < cfg->batch; ++b)
      if ((cfg->ctx_len[b] + kPart - 1) / kPart > cfg->max_partitions)
        return fail(nullptr, SPIN_ERR_INVALID, "ctx_len[%d] = %lld needs more than max_partitions = %d partitions", b,
                    (long long)cfg->ctx_len[b], cfg->max_partitions);
  }
  if (cfg->seg_pool_segments < 0) return fail(nullptr, SPIN_ERR_INVALID, "seg_pool_segments must be >= 0");
  if (cfg->max_context < 0 || cfg->max_context > (int64_t)32768 * kPart)
    return fail(nullptr, SPIN_ERR_INVALID, "max_context must be in [0, %d]", 32768 * kPart);
  for (int b = 0; cfg->max_context > 0 && b < cfg->batch; ++b)
    if (cfg->ctx_len[b] + cfg->append_tokens > cfg->max_context)
      return fail(nullptr, SPIN_ERR_INVALID, "ctx_len[%d] + append_tokens = %lld exceeds max_context = %lld", b,
                  (long long)(cfg->ctx_len[b] + cfg->append_tokens), (long long)cfg->max_context);
  const int64_t units = (int64_t)cfg->batch * cfg->layers * cfg->kv_heads;
  if (units * ((int64_t)cfg->buf_mult * cfg->topk + 1) >= (int64_t)1 << 24)
    return fail(nullptr, SPIN_ERR_INVALID, "units * (capacity + 1) must stay below 2^24 pages");
  return SPIN_OK;
}

LayerArgs make_args(spin_ctx* c, int l) {
  LayerArgs a{};
  LayerBuf& lb = c->layers[l];
  a.layer = l;
  a.B = c->B;
  a.Hq = c->Hq;
  a.Hkv = c->Hkv;
  a.G = c->G;
  a.k = c->k;
  a.cap = c->cap;
  a.D = c->D;
  a.P_max = c->P_max;
  a.n_chunks = c->n_chunks;
  a.ppt = c->ppt;
  a.S = (int32_t)c->S;
  a.retr_warps = c->retr_warps;
  a.retr_late = c->retr_late;
  a.mgr_gs = c->mgr_gs;
  a.pipe = c->pipe;
  a.retr_split = c->retr_split;
  a.ka = c->ka;
  a.P_b = c->d_P_lb + (int64_t)l * c->B;
  a.ntok_b = c->d_ntok_lb + (int64_t)l * c->B;
  a.tail_n = c->tail_mode ? c->d_tail_lb + (int64_t)l * c->B : nullptr;
  a.part_valid = c->d_part_valid;
  a.pstride_b = c->d_pstride_b;
  a.budget_b = c->d_budget_b;
  a.poff_b = c->d_poff_b;
  a.layer_page_base = (int64_t)l * c->pages_per_layer;
  a.unit_base = (int64_t)l * c->B * c->Hkv;
  a.host_pages = c->pages_per_layer * c->L;
  a.pool_slots = c->units * c->cap;
  a.summ = c->d_summ;
  a.host_store = c->d_store;
  a.pool = c->d_pool;
  a.dir = c->d_dir;
  a.seg = c->d_seg;
  a.seg_live = c->d_seg_live;
  a.seg_bitmap = c->d_bitmap;
  a.slot_part = c->d_slot_part;
  a.last_use = c->d_last_use;
  a.scores = lb.scores;
  a.sel = lb.sel;
  a.sel_slot = lb.sel_slot;
  a.sel_hit = lb.sel_hit;
  a.keff = lb.keff;
  a.unit_info = lb.unit_info;
  a.miss_src = lb.miss_src;
  a.miss_dst = lb.miss_dst;
  a.miss_att = lb.miss_att;
  a.miss_valid = lb.miss_valid;
  a.ready = lb.ready;
  a.ready_cnt = lb.ready_cnt;
  a.miss_tag = lb.miss_tag;
  a.unit_rows = lb.unit_rows;
  a.unit_ready = lb.unit_ready;
  a.hist12 = lb.hist12;
  a.att_slot = lb.att_slot;
  a.att_valid = lb.att_valid;
  a.n_hit = lb.n_hit;
  a.counters = lb.counters;
  a.partials = lb.partials;
  a.stats = c->d_stats;
  a.timeline = nullptr;
  a.err = c->d_err;
  return a;
}

int create_impl(const spin_config* cfg, spin_ctx* c) {
  c->device = cfg->device;
  c->flags = cfg->flags;
  c->B = cfg->batch;
  c->L = cfg->layers;
  c->Hq = cfg->q_heads;
  c->Hkv = cfg->kv_heads;
  c->G = c->Hq / c->Hkv;
  c->k = cfg->topk;
  c->cap = cfg->buf_mult * cfg->topk;
  c->ctx_len.assign(cfg->ctx_len, cfg->ctx_len + c->B);
  c->append_tokens = cfg->append_tokens;
  c->tail_mode = cfg->append_tokens > 0;
  c->part_mode = cfg->max_partitions > 0;
  c->max_partitions = cfg->max_partitions;
  c->ka = c->k + (c->tail_mode ? 1 : 0);
  c->P_b.resize(c->B);
  c->ntok_b.resize(c->B);
  c->pstride_b.resize(c->B);
  c->poff_b.resize(c->B);
  int64_t poff = 0;
  c->P_max = 0;
  int64_t auto_S = 0;
  for (int b = 0; b < c->B; ++b) {
    c->ntok_b[b] = (int32_t)c->ctx_len[b];
    c->P_b[b] = (int32_t)((c->ctx_len[b] + kPart - 1) / kPart);
    // tail mode: room for every partition the request can reach
    c->pstride_b[b] = c->tail_mode   ? (int32_t)((c->ctx_len[b] + c->append_tokens + kPart - 1) / kPart)
                      : c->part_mode ? c->max_partitions
                                     : c->P_b[b];
    c->poff_b[b] = poff;
    poff += c->pstride_b[b];
    c->P_max = std::max(c->P_max, c->pstride_b[b]);
    const int64_t Du = (c->pstride_b[b] + kSeg - 1) / kSeg;
    auto_S += std::min<int64_t>(Du, c->cap) * c->Hkv * c->L;
  }
  c->P_lb.assign((size_t)c->L * c->B, 0);
  c->tail_lb.assign((size_t)c->L * c->B, 0);
  for (int l = 0; l < c->L && !c->tail_mode && !c->part_mode; ++l)
    for (int b = 0; b < c->B; ++b) c->P_lb[(size_t)l * c->B + b] = c->P_b[b];
  // the logical capacity in partitions per unit: the static directory covers it, and the flat
  // worst-case table spin_stats reports is sized for it
  c->P_logical = std::max<int64_t>(c->P_max, (cfg->max_context + kPart - 1) / kPart);
  c->D = (int)std::max<int64_t>(1, (c->P_logical + kSeg - 1) / kSeg);
  c->pages_per_layer = poff * c->Hkv;
  c->units = (int64_t)c->B * c->L * c->Hkv;
  c->S = cfg->seg_pool_segments > 0 ? cfg->seg_pool_segments : std::max<int64_t>(auto_S, 1);
  if (c->S >= (int64_t)1 << 30) return fail(nullptr, SPIN_ERR_INVALID, "seg_pool_segments too large");

  // Test hook: report a failed pinned allocation before touching the device.
  if (c->flags & SPIN_FLAG_TEST_FAIL_PINNED)
    return fail(nullptr, SPIN_ERR_OOM, "pinned host allocation failed (injected by SPIN_FLAG_TEST_FAIL_PINNED)");

  cudaError_t e = cudaSetDevice(c->device);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "selecting the CUDA device");
  int major = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, c->device);
  cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
  if (major < 10) return fail(nullptr, SPIN_ERR_CUDA, "device %d is not a Blackwell GPU (sm_%d)", c->device, major);

  // pinned host page store (mapped: kernels read it directly)
  const int64_t total_pages = c->pages_per_layer * c->L;
  c->bytes_store = total_pages * kPageBytes;
  if (total_pages > 0) {
    void* h = nullptr;
    if (c->flags & SPIN_FLAG_HOST_HUGEPAGES) h = alloc_host_hugepages((size_t)c->bytes_store, &c->h_store_map_len);
    if (!h) {
      c->h_store_map_len = 0;
      e = cudaHostAlloc(&h, (size_t)c->bytes_store, cudaHostAllocMapped | cudaHostAllocPortable);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(nullptr, SPIN_ERR_OOM, "pinned host allocation of %lld bytes failed: %s",
                    (long long)c->bytes_store, cudaGetErrorString(e));
      }
    }
    c->h_store = static_cast<uint16_t*>(h);
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, h, 0);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "mapping the host page store");
    c->d_store = static_cast<uint16_t*>(d);
  }

  // HBM
  const int64_t slots = c->units * c->cap;
  const int64_t tail_pages = c->tail_mode ? c->units : 0;  // one tail page per unit, after the pool slots
  c->bytes_pool = (slots + tail_pages) * kPageBytes;
  c->bytes_summ = total_pages * kD * 4;
#define ALLOC(ptr, n, what) \
  if ((e = dalloc(c, &(ptr), (size_t)(n))) != cudaSuccess) return cuda_fail(nullptr, e, what)
  ALLOC(c->d_pool, (slots + tail_pages) * kPageElems, "allocating the HBM page pool");
  ALLOC(c->d_summ, total_pages * kD, "allocating the summaries");
  if (c->part_mode) {
    ALLOC(c->d_part_valid, total_pages, "allocating the partition sizes");
    SPIN_CUDA(nullptr, cudaMemset(c->d_part_valid, 0, (size_t)std::max<int64_t>(total_pages, 1)),
              "initialising the partition sizes");
  }
  ALLOC(c->d_P_lb, (int64_t)c->L * c->B, "allocating request tables");
  ALLOC(c->d_ntok_lb, (int64_t)c->L * c->B, "allocating request tables");
  ALLOC(c->d_tail_lb, (int64_t)c->L * c->B, "allocating request tables");
  ALLOC(c->d_pstride_b, c->B, "allocating request tables");
  ALLOC(c->d_budget_b, c->B, "allocating request tables");
  ALLOC(c->d_poff_b, c->B, "allocating request tables");
  ALLOC(c->d_dir, c->units * c->D, "allocating the directory");
  if (c->flags & SPIN_FLAG_TIER_SPLIT) {
    // Tier split: the capacity-heavy second-level entries go to host memory, read and
    // written by the manager kernel with plain loads and stores over the host link; the
    // directory, live counts and allocation bitmap (touched by atomics) stay in HBM.
    void* hs = nullptr;
    e = cudaHostAlloc(&hs, (size_t)c->S * kSeg * 4, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(nullptr, SPIN_ERR_OOM, "pinned allocation of the segment pool failed: %s", cudaGetErrorString(e));
    }
    c->h_seg = static_cast<int32_t*>(hs);
    memset(c->h_seg, 0xff, (size_t)c->S * kSeg * 4);
    void* ds = nullptr;
    if ((e = cudaHostGetDevicePointer(&ds, hs, 0)) != cudaSuccess) return cuda_fail(nullptr, e, "mapping the segment pool");
    c->d_seg = static_cast<int32_t*>(ds);
  } else {
    ALLOC(c->d_seg, c->S * kSeg, "allocating the segment pool");
  }
  ALLOC(c->d_seg_live, c->S, "allocating the segment pool");
  const int64_t nwords = (c->S + 31) / 32;
  ALLOC(c->d_bitmap, nwords, "allocating the segment bitmap");
  ALLOC(c->d_slot_part, slots, "allocating the page state");
  ALLOC(c->d_last_use, slots, "allocating the page state");
  ALLOC(c->d_stats, 8, "allocating counters");
  ALLOC(c->d_err, 1, "allocating counters");
  ALLOC(c->d_warm_sink, 1, "allocating counters");
  c->bytes_meta = (c->units * c->D + (c->h_seg ? 0 : c->S * kSeg) + c->S + nwords + 2 * slots) * 4;
  c->bytes_flat = (c->units * c->P_logical + 2 * slots) * 4;

  {
    // fixed mode: every layer holds the request's partitions; tail mode and variable
    // partitions: nothing until offload
    std::vector<int32_t> ntok_lb((size_t)c->L * c->B, 0);
    for (int l = 0; l < c->L && !c->tail_mode && !c->part_mode; ++l)
      for (int b = 0; b < c->B; ++b) ntok_lb[(size_t)l * c->B + b] = c->ntok_b[b];
    const size_t n = (size_t)c->L * c->B * 4;
    SPIN_CUDA(nullptr, cudaMemcpy(c->d_P_lb, c->P_lb.data(), n, cudaMemcpyHostToDevice), "uploading tables");
    SPIN_CUDA(nullptr, cudaMemcpy(c->d_ntok_lb, ntok_lb.data(), n, cudaMemcpyHostToDevice), "uploading tables");
    SPIN_CUDA(nullptr, cudaMemset(c->d_tail_lb, 0, n), "uploading tables");
  }
  SPIN_CUDA(nullptr, cudaMemcpy(c->d_pstride_b, c->pstride_b.data(), 4 * c->B, cudaMemcpyHostToDevice),
            "uploading tables");
  {
    const std::vector<int32_t> budget(c->B, c->cap);
    SPIN_CUDA(nullptr, cudaMemcpy(c->d_budget_b, budget.data(), 4 * c->B, cudaMemcpyHostToDevice),
              "uploading tables");
  }
  SPIN_CUDA(nullptr, cudaMemcpy(c->d_poff_b, c->poff_b.data(), 8 * c->B, cudaMemcpyHostToDevice), "uploading tables");
  if (tail_pages)
    SPIN_CUDA(nullptr, cudaMemset(c->d_pool + slots * kPageElems, 0, (size_t)tail_pages * kPageBytes),
              "clearing the tail pages");
  SPIN_CUDA(nullptr, cudaMemset(c->d_dir, 0xff, (size_t)c->units * c->D * 4), "initialising the directory");
  if (!c->h_seg)
    SPIN_CUDA(nullptr, cudaMemset(c->d_seg, 0xff, (size_t)c->S * kSeg * 4), "initialising the segment pool");
  SPIN_CUDA(nullptr, cudaMemset(c->d_seg_live, 0, (size_t)c->S * 4), "initialising the segment pool");
  {
    std::vector<uint32_t> bm(nwords, 0u);
    if (c->S % 32) bm[nwords - 1] = ~((1u << (c->S % 32)) - 1u);  // bits past S are never free
    SPIN_CUDA(nullptr, cudaMemcpy(c->d_bitmap, bm.data(), nwords * 4, cudaMemcpyHostToDevice), "initialising the bitmap");
  }
  SPIN_CUDA(nullptr, cudaMemset(c->d_slot_part, 0xff, (size_t)slots * 4), "initialising the page state");
  SPIN_CUDA(nullptr, cudaMemset(c->d_last_use, 0, (size_t)slots * 4), "initialising the page state");
  SPIN_CUDA(nullptr, cudaMemset(c->d_stats, 0, 8 * 8), "initialising counters");
  SPIN_CUDA(nullptr, cudaMemset(c->d_err, 0, 4), "initialising counters");

  // retriever warps: two from the start, the rest (four in the one-tile kernel, two in the
  // two-tile kernel) once the CTA's resident pages are issued
  c->retr_warps = 2;
  c->retr_late = c->G <= 8 ? 4 : 2;
  {
    const long pg = sysconf(_SC_PAGESIZE);
    c->warm_stride = pg >= 4096 ? std::min<int64_t>(pg, kPageBytes) : 4096;
  }
  if (c->flags & SPIN_FLAG_TEST_NO_RETRIEVE) c->retr_warps = c->retr_late = 0;
  // the first entries of a step's miss list are split in kRetrChunks pieces, about one piece
  // per retriever warp of the grid that loads from the start: a step with few misses gets
  // its pages in about one host-link round trip each instead of kRetrChunks
  c->retr_split = (int)std::min<int64_t>((int64_t)c->B * c->Hkv * c->k,
                                         (int64_t)std::max(1, c->sm_count) * c->retr_warps / kRetrChunks);

  // attention work split: pages per task, about one task per consumer group when pages
  // are few (each task costs a merge and a partial to combine), at most 8
  const int64_t pages_layer = (int64_t)c->B * c->Hkv * c->k;
  const int64_t groups = (int64_t)std::max(1, c->sm_count) * (c->G <= 8 ? 2 : 1);
  c->ppt = (int)std::max<int64_t>(1, std::min<int64_t>(8, (pages_layer + groups - 1) / groups));
  c->n_chunks = (c->ka + c->ppt - 1) / c->ppt;

  // manager groups: one warp per unit for small units, four warps for mid-size ones, all
  // the CTA's warps for units too wide for a group of four (or whose shared memory does
  // not fit four times in the ring's bytes)
  {
    LayerArgs probe{};
    probe.G = c->G;
    probe.P_max = c->P_max;
    probe.cap = c->cap;
    probe.k = c->k;
    probe.D = c->D;
    const int threads = step_threads(c->G), full = step_full_group(c->G);
    auto fits = [&](int gs) { return (size_t)(threads / gs) * mgr_group_bytes(gs, probe) <= step_ring_bytes(); };
    int gs = c->P_max > 4096 ? full : (c->P_max <= 128 && c->cap <= 1024 && c->k <= 256) ? 32 : 128;
    if (gs == 32 && !fits(32)) gs = 128;
    if (gs == 128 && !fits(128)) gs = full;
    c->mgr_gs = gs;
    probe.mgr_gs = gs;
    probe.B = c->B;
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    // the pipelined kernel (scoring, manager groups and retrieval at once, a 4-stage ring) for
    // units of at most 4096 partitions and groups of at most 8 query heads, when its shared
    // memory fits; otherwise the phased kernel. Its four manager warps form one group of 128
    // threads or four groups of one warp.
    if (c->G <= 8 && c->P_max <= 4096 && c->B <= 8192 && !(c->flags & SPIN_FLAG_PHASED)) {
      const int order[2] = {kPipeGroupFirst, kPipeGroupFirst == 32 ? 128 : 32};
      for (int gs_p : order) {
        LayerArgs pp = probe;
        pp.pipe = 1;
        pp.mgr_gs = gs_p;
        if (step_smem_bytes(pp) <= (size_t)optin) {
          c->pipe = 1;
          c->mgr_gs = gs_p;
          probe = pp;
          break;
        }
      }
    }
    if (step_smem_bytes(probe) > (size_t)optin)
      return fail(nullptr, SPIN_ERR_INVALID,
                  "the page manager of one unit needs %zu bytes of shared memory (max %d): reduce the longest "
                  "context, topk or buf_mult",
                  step_smem_bytes(probe), optin);
  }
  if (c->flags & SPIN_FLAG_STAGE_TIMING) {
    ALLOC(c->d_timeline, (int64_t)kTimelineCalls * kTlSlots, "allocating stage stamps");
    SPIN_CUDA(nullptr, cudaMemset(c->d_timeline, 0, (size_t)kTimelineCalls * kTlSlots * 8), "clearing stage stamps");
  }

  const int64_t Ul = (int64_t)c->B * c->Hkv;
  c->layers.resize(c->L);
  for (int l = 0; l < c->L; ++l) {
    LayerBuf& lb = c->layers[l];
    // two buffers (step parity); +4: the wide top-k reads a unit's scores four at a time, up to
    // 3 past its last partition
    ALLOC(lb.scores, 2 * Ul * std::max(1, c->P_max) + 4, "allocating layer scratch");
    SPIN_CUDA(nullptr, launch_fill_u32(reinterpret_cast<uint32_t*>(lb.scores), kScoreEmpty,
                                       2 * Ul * std::max(1, c->P_max) + 4, 0), "initialising layer scratch");
    ALLOC(lb.sel, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.sel_slot, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.sel_hit, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.keff, Ul, "allocating layer scratch");
    ALLOC(lb.unit_info, Ul * 8, "allocating layer scratch");
    ALLOC(lb.miss_src, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.miss_dst, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.att_slot, Ul * c->ka, "allocating layer scratch");
    ALLOC(lb.att_valid, Ul * c->ka, "allocating layer scratch");
    ALLOC(lb.n_hit, Ul, "allocating layer scratch");
    ALLOC(lb.miss_att, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.miss_valid, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.ready, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.ready_cnt, c->retr_split > 0 ? c->retr_split : 1, "allocating layer scratch");
    ALLOC(lb.miss_tag, Ul * c->k, "allocating layer scratch");
    ALLOC(lb.unit_rows, Ul, "allocating layer scratch");
    ALLOC(lb.unit_ready, Ul, "allocating layer scratch");
    if (c->P_max > 4096 && c->mgr_gs >= 256) {  // wide units: top-12-bit key counts filled while scoring
      ALLOC(lb.hist12, Ul * 4096, "allocating layer scratch");
      SPIN_CUDA(nullptr, cudaMemset(lb.hist12, 0, Ul * 4096 * 4), "initialising layer scratch");
    }
    ALLOC(lb.counters, kNumCtr, "allocating layer scratch");
    ALLOC(lb.partials, Ul * (c->n_chunks + c->ka) * c->G * kPartialStride, "allocating layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.n_hit, 0, Ul * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.ready, 0, Ul * c->k * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.ready_cnt, 0, (c->retr_split > 0 ? c->retr_split : 1) * 4),
              "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.miss_tag, 0, Ul * c->k * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.unit_rows, 0, Ul * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.unit_ready, 0, Ul * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.counters, 0, kNumCtr * 4), "initialising layer counters");
    SPIN_CUDA(nullptr, cudaMemset(lb.keff, 0, Ul * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.sel, 0xff, Ul * c->k * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.sel_slot, 0xff, Ul * c->k * 4), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.sel_hit, 0, Ul * c->k), "initialising layer scratch");
    SPIN_CUDA(nullptr, cudaMemset(lb.unit_info, 0, Ul * 8 * 4), "initialising layer scratch");
    lb.args = make_args(c, l);
  }
#undef ALLOC
  c->offloaded.assign((size_t)c->L * c->B, 0);
  c->layer_steps.assign(c->L, 0);

  int rc = encode_tensor_map(c);
  if (rc != SPIN_OK) {
    g_create_error = c->msg;
    return rc;
  }
  SPIN_CUDA(nullptr, step_configure(c->layers[0].args), "configuring the decode-step kernel");
  SPIN_CUDA(nullptr, cudaDeviceSynchronize(), "finishing context set-up");
  return SPIN_OK;
}

// Enqueue one layer's step on `st`: one cooperative kernel (score -> select + manage ->
// retrieve + attention -> combine).
// q: the queries in HBM the attention stages; q_src: the queries the scores read (q, or a
// device-usable address of pinned host memory whose rows the unit managers copy into q).
int enqueue_step(spin_ctx* c, int layer, const uint16_t* q, const uint16_t* q_src, float* out, cudaStream_t st) {
  LayerBuf& lb = c->layers[layer];
  LayerArgs a = lb.args;
  a.q = q;
  a.q_src = q_src;
  a.out = out;
  // stage timing: CUDA events around the kernel and a record of in-kernel stage stamps
  // (up to kTimelineCalls timed calls between two synchronising calls)
  const bool timed = (c->flags & SPIN_FLAG_STAGE_TIMING) != 0 && c->next_rec < kTimelineCalls;
  TimedCall tc{};
  if (timed) {
    for (auto& e : tc.ev) {
      int rc = get_event(c, &e);
      if (rc) return rc;
    }
    tc.rec = c->next_rec++;
    a.timeline = c->d_timeline + (size_t)tc.rec * kTlSlots;
  }
  for (int i = 0; c->store_cold && i < c->store_warm; ++i) {
    // after the store is (re)written, before the first retrieval can touch it
    SPIN_CUDA(c, launch_warm_store(c->d_store, c->bytes_store, c->warm_stride, c->d_warm_sink, c->sm_count, st),
              "launching the host-store read pass");
  }
  c->store_cold = false;
  if (timed) cudaEventRecord(tc.ev[0], st);
  SPIN_CUDA(c, launch_decode_step(a, &c->tmap, c->sm_count, st), "launching the decode step");
  if (timed) {
    cudaEventRecord(tc.ev[1], st);
    c->pending.push_back(tc);
    c->timed_calls += 1;
  }
  c->steps_host += 1;
  c->layer_steps[layer] += 1;
  return SPIN_OK;
}

// The device-usable address of pinned, device-mapped host memory at p when it is
// `align`-byte aligned; nullptr for pageable or unaligned memory.
const void* mapped_host(const void* p, uintptr_t align) {
  if (reinterpret_cast<uintptr_t>(p) & (align - 1)) return nullptr;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (pa.type != cudaMemoryTypeHost || !pa.devicePointer) return nullptr;
  if (reinterpret_cast<uintptr_t>(pa.devicePointer) & (align - 1)) return nullptr;
  return pa.devicePointer;
}

int check_layer(spin_ctx* c, int layer) {
  if (layer < 0 || layer >= c->L) return fail(c, SPIN_ERR_INVALID, "layer %d outside [0, %d)", layer, c->L);
  for (int b = 0; b < c->B; ++b)
    if (!c->offloaded[(size_t)layer * c->B + b])
      return fail(c, SPIN_ERR_STATE, "request %d of layer %d has not been offloaded", b, layer);
  if (c->sticky) return check_device_error(c);
  return SPIN_OK;
}

}  // namespace

namespace spin {
// Message for spin_last_error(NULL) from entry points that have no context.
void set_global_error(const char* msg) { g_create_error = msg; }
}  // namespace spin

extern "C" {

int spin_create(const spin_config* cfg, spin_ctx** out) {
  if (!out) return fail(nullptr, SPIN_ERR_INVALID, "out is NULL");
  *out = nullptr;
  int rc = validate(cfg);
  if (rc) return rc;
  spin_ctx* c = new (std::nothrow) spin_ctx();
  if (!c) return fail(nullptr, SPIN_ERR_OOM, "host allocation of the context failed");
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) {
    cudaGetLastError();
    prev = -1;
  }
  rc = create_impl(cfg, c);
  if (prev >= 0) cudaSetDevice(prev);
  if (rc != SPIN_OK) {
    free_all(c);
    delete c;
    return rc;
  }
  *out = c;
  return SPIN_OK;
}

int spin_index_offload(spin_ctx* c, int32_t b, int32_t layer, const uint16_t* k, const uint16_t* v,
                       int64_t n_tokens, int32_t src_is_host, spin_stream_t stream) {
  if (!c) return fail(nullptr, SPIN_ERR_INVALID, "ctx is NULL");
  if (b < 0 || b >= c->B || layer < 0 || layer >= c->L)
    return fail(c, SPIN_ERR_INVALID, "request %d / layer %d out of range", b, layer);
  if (c->part_mode)
    return fail(c, SPIN_ERR_STATE, "a context with max_partitions > 0 takes spin_index_offload_parts");
  if (n_tokens != c->ctx_len[b])
    return fail(c, SPIN_ERR_INVALID, "n_tokens %lld differs from ctx_len[%d] = %lld", (long long)n_tokens, b,
                (long long)c->ctx_len[b]);
  if (n_tokens > 0 && (!k || !v)) return fail(c, SPIN_ERR_INVALID, "k or v is NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return fail(c, SPIN_ERR_INVALID, "k and v must be 16-byte aligned");
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t P = c->pstride_b[b];  // host-store pages per KV head of the request
  const int64_t page0 = (int64_t)layer * c->pages_per_layer + (int64_t)c->Hkv * c->poff_b[b];
  float* summ0 = c->d_summ + page0 * kD;
  uint16_t* host0 = c->d_store + page0 * kPageElems;
  // Tail mode: only the complete partitions are indexed and offloaded; the remaining
  // n % 64 tokens go into the units' tail pages in HBM.
  const int64_t n_part_tok = c->tail_mode ? n_tokens / kPart * kPart : n_tokens;
  const int64_t rem = n_tokens - n_part_tok;
  if (c->tail_mode) {
    const size_t lb = (size_t)layer * c->B + b;
    const int64_t unit0 = ((int64_t)layer * c->B + b) * c->Hkv;
    uint16_t* tail0 = c->d_pool + (c->units * c->cap + unit0) * kPageElems;
    SPIN_CUDA(c, cudaMemsetAsync(tail0, 0, (size_t)c->Hkv * kPageBytes, st), "clearing the tail pages");
    if (rem > 0) {
      for (int half = 0; half < 2; ++half)
        SPIN_CUDA(c,
                  cudaMemcpy2DAsync(tail0 + half * kPart * kD, kPageBytes, (half ? v : k) + n_part_tok * kD,
                                    (size_t)n_tokens * kD * 2, (size_t)rem * kD * 2, (size_t)c->Hkv,
                                    cudaMemcpyDefault, st),
                  "copying the tail tokens");
    }
    const int32_t Pc = (int32_t)(n_part_tok / kPart);
    SPIN_CUDA(c,
              launch_set_request(c->d_P_lb + lb, c->d_ntok_lb + lb, c->d_tail_lb + lb, Pc, Pc * kPart, (int32_t)rem,
                                 st),
              "setting the request state");
    c->P_lb[lb] = Pc;
    c->tail_lb[lb] = (int32_t)rem;
  }
  if (n_part_tok > 0) {
    if (!src_is_host) {
      SPIN_CUDA(c,
                launch_summarize_offload(k, v, n_tokens, c->Hkv, 0, n_part_tok, n_part_tok, summ0, host0, P, st),
                "launching summarize/offload");
    } else {
      // stage through HBM in chunks of whole partitions
      const int64_t chunk_tok = 256 * kPart;
      if (!c->d_stage_k) {
        cudaError_t e;
        if ((e = dalloc(c, &c->d_stage_k, (size_t)c->Hkv * chunk_tok * kD)) != cudaSuccess)
          return cuda_fail(c, e, "allocating the offload staging buffer");
        if ((e = dalloc(c, &c->d_stage_v, (size_t)c->Hkv * chunk_tok * kD)) != cudaSuccess)
          return cuda_fail(c, e, "allocating the offload staging buffer");
        c->stage_tokens = chunk_tok;
      }
      for (int64_t t0 = 0; t0 < n_part_tok; t0 += chunk_tok) {
        const int64_t nt = std::min(chunk_tok, n_part_tok - t0);
        SPIN_CUDA(c,
                  cudaMemcpy2DAsync(c->d_stage_k, (size_t)nt * kD * 2, k + t0 * kD, (size_t)n_tokens * kD * 2,
                                    (size_t)nt * kD * 2, (size_t)c->Hkv, cudaMemcpyHostToDevice, st),
                  "copying K to the staging buffer");
        SPIN_CUDA(c,
                  cudaMemcpy2DAsync(c->d_stage_v, (size_t)nt * kD * 2, v + t0 * kD, (size_t)n_tokens * kD * 2,
                                    (size_t)nt * kD * 2, (size_t)c->Hkv, cudaMemcpyHostToDevice, st),
                  "copying V to the staging buffer");
        SPIN_CUDA(c,
                  launch_summarize_offload(c->d_stage_k, c->d_stage_v, nt, c->Hkv, t0, nt, n_part_tok, summ0, host0,
                                           P, st),
                  "launching summarize/offload");
      }
    }
  }
  c->offloaded[(size_t)layer * c->B + b] = 1;
  if (n_part_tok > 0) c->store_cold = true;
  return SPIN_OK;
}

int spin_index_offload_parts(spin_ctx* c, int32_t b, int32_t layer, const uint16_t* k, const uint16_t* v,
                             int64_t n_tokens, const int32_t* order, const int32_t* starts, int32_t n_parts,
                             int32_t src_is_host, spin_stream_t stream) {
  if (!c) return fail(nullptr, SPIN_ERR_INVALID, "ctx is NULL");
  if (!c->part_mode)
    return fail(c, SPIN_ERR_STATE, "spin_index_offload_parts needs a context created with max_partitions > 0");
  if (b < 0 || b >= c->B || layer < 0 || layer >= c->L)
    return fail(c, SPIN_ERR_INVALID, "request %d / layer %d out of range", b, layer);
  if (n_tokens != c->ctx_len[b])
    return fail(c, SPIN_ERR_INVALID, "n_tokens %lld differs from ctx_len[%d] = %lld", (long long)n_tokens, b,
                (long long)c->ctx_len[b]);
  if (n_tokens == 0 ? n_parts != 0 : (n_parts < 1 || n_parts > c->max_partitions))
    return fail(c, SPIN_ERR_INVALID, "n_parts = %d outside [1, max_partitions = %d] (0 for an empty request)",
                n_parts, c->max_partitions);
  if (n_tokens > 0 && (!k || !v || !order || !starts)) return fail(c, SPIN_ERR_INVALID, "k, v, order or starts is NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return fail(c, SPIN_ERR_INVALID, "k and v must be 16-byte aligned");
  // the grouping: per head, partitions of 1..64 tokens that cover a permutation of the tokens
  if (n_tokens > 0) {
    std::vector<uint8_t> seen((size_t)n_tokens);
    for (int h = 0; h < c->Hkv; ++h) {
      const int32_t* st = starts + (int64_t)h * (n_parts + 1);
      const int32_t* od = order + (int64_t)h * n_tokens;
      if (st[0] != 0 || st[n_parts] != n_tokens)
        return fail(c, SPIN_ERR_INVALID, "head %d: starts must run from 0 to n_tokens", h);
      for (int p = 0; p < n_parts; ++p) {
        const int64_t m = (int64_t)st[p + 1] - st[p];
        if (m < 1 || m > kPart)
          return fail(c, SPIN_ERR_INVALID, "head %d partition %d holds %lld tokens (1..%d allowed)", h, p, (long long)m,
                      kPart);
      }
      std::fill(seen.begin(), seen.end(), 0);
      for (int64_t j = 0; j < n_tokens; ++j) {
        const int32_t t = od[j];
        if (t < 0 || t >= n_tokens || seen[t])
          return fail(c, SPIN_ERR_INVALID, "head %d: order is not a permutation of the request's tokens", h);
        seen[t] = 1;
      }
    }
  }
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t P = c->pstride_b[b];  // = max_partitions: host-store pages per KV head of the request
  const int64_t page0 = (int64_t)layer * c->pages_per_layer + (int64_t)c->Hkv * c->poff_b[b];
  if (n_tokens > 0) {
    int64_t max_ctx = 0;
    for (int64_t n : c->ctx_len) max_ctx = std::max(max_ctx, n);
    cudaError_t e;
    if (!c->d_gorder) {
      if ((e = dalloc(c, &c->d_gorder, (size_t)c->Hkv * max_ctx)) != cudaSuccess)
        return cuda_fail(c, e, "allocating the grouping buffer");
      if ((e = dalloc(c, &c->d_gstarts, (size_t)c->Hkv * (c->max_partitions + 1))) != cudaSuccess)
        return cuda_fail(c, e, "allocating the grouping buffer");
    }
    SPIN_CUDA(c, cudaMemcpyAsync(c->d_gorder, order, (size_t)c->Hkv * n_tokens * 4, cudaMemcpyHostToDevice, st),
              "copying the token order");
    SPIN_CUDA(c,
              cudaMemcpyAsync(c->d_gstarts, starts, (size_t)c->Hkv * (n_parts + 1) * 4, cudaMemcpyHostToDevice, st),
              "copying the partition starts");
    const uint16_t *ks = k, *vs = v;
    if (src_is_host) {
      if (!c->d_gk) {
        if ((e = dalloc(c, &c->d_gk, (size_t)c->Hkv * max_ctx * kD)) != cudaSuccess)
          return cuda_fail(c, e, "allocating the offload staging buffer");
        if ((e = dalloc(c, &c->d_gv, (size_t)c->Hkv * max_ctx * kD)) != cudaSuccess)
          return cuda_fail(c, e, "allocating the offload staging buffer");
      }
      const size_t bytes = (size_t)c->Hkv * n_tokens * kD * 2;
      SPIN_CUDA(c, cudaMemcpyAsync(c->d_gk, k, bytes, cudaMemcpyHostToDevice, st), "copying K to the staging buffer");
      SPIN_CUDA(c, cudaMemcpyAsync(c->d_gv, v, bytes, cudaMemcpyHostToDevice, st), "copying V to the staging buffer");
      ks = c->d_gk;
      vs = c->d_gv;
    }
    SPIN_CUDA(c,
              launch_gather_offload(ks, vs, n_tokens, c->Hkv, c->d_gorder, c->d_gstarts, n_parts,
                                    c->d_summ + page0 * kD, c->d_store + page0 * kPageElems, P,
                                    c->d_part_valid + page0, st),
              "launching gather/offload");
  }
  const size_t lb = (size_t)layer * c->B + b;
  SPIN_CUDA(c,
            launch_set_request(c->d_P_lb + lb, c->d_ntok_lb + lb, nullptr, n_parts, (int32_t)n_tokens, 0, st),
            "setting the request state");
  SPIN_CUDA(c, cudaStreamSynchronize(st), "finishing the offload");
  c->P_lb[lb] = n_parts;
  c->offloaded[lb] = 1;
  if (n_tokens > 0) c->store_cold = true;
  return SPIN_OK;
}

int spin_append_kv(spin_ctx* c, int32_t layer, const uint16_t* k_new, const uint16_t* v_new, spin_stream_t stream) {
  if (!c) return fail(nullptr, SPIN_ERR_INVALID, "ctx is NULL");
  if (!c->tail_mode) return fail(c, SPIN_ERR_STATE, "spin_append_kv needs a context created with append_tokens > 0");
  if (!k_new || !v_new) return fail(c, SPIN_ERR_INVALID, "k_new or v_new is NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return fail(c, SPIN_ERR_INVALID, "k_new and v_new must be 16-byte aligned");
  int rc = check_layer(c, layer);
  if (rc) return rc;
  for (int b = 0; b < c->B; ++b) {
    const size_t lb = (size_t)layer * c->B + b;
    const int64_t have = (int64_t)c->P_lb[lb] * kPart + c->tail_lb[lb];
    if (have + 1 > c->ctx_len[b] + c->append_tokens)
      return fail(c, SPIN_ERR_CAPACITY, "request %d of layer %d would exceed ctx_len + append_tokens = %lld tokens", b,
                  layer, (long long)(c->ctx_len[b] + c->append_tokens));
  }
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  const size_t l0 = (size_t)layer * c->B;
  SPIN_CUDA(c,
            launch_append(c->layers[layer].args, k_new, v_new, c->d_P_lb + l0, c->d_ntok_lb + l0, c->d_tail_lb + l0,
                          static_cast<cudaStream_t>(stream)),
            "launching append");
  for (int b = 0; b < c->B; ++b) {
    if (++c->tail_lb[l0 + b] == kPart) {
      c->tail_lb[l0 + b] = 0;
      c->P_lb[l0 + b] += 1;
    }
  }
  c->appended += c->B;
  return SPIN_OK;
}

int spin_set_buffer(spin_ctx* c, int32_t b, int32_t pages, spin_stream_t stream) {
  if (!c) return fail(nullptr, SPIN_ERR_INVALID, "ctx is NULL");
  if (b < 0 || b >= c->B) return fail(c, SPIN_ERR_INVALID, "request %d outside [0, %d)", b, c->B);
  if (pages < c->k || pages > c->cap)
    return fail(c, SPIN_ERR_INVALID, "buffer of %d pages outside [topk, buf_mult * topk] = [%d, %d]", pages, c->k,
                c->cap);
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  SPIN_CUDA(c, launch_set_int(c->d_budget_b + b, pages, static_cast<cudaStream_t>(stream)), "setting the budget");
  return SPIN_OK;
}

int spin_decode_step(spin_ctx* c, int32_t layer, const uint16_t* q, float* out, spin_stream_t stream) {
  if (!c) return fail(nullptr, SPIN_ERR_INVALID, "ctx is NULL");
  if (!q || !out) return fail(c, SPIN_ERR_INVALID, "q or out is NULL");
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return fail(c, SPIN_ERR_INVALID, "q and out must be 16-byte aligned");
  int rc = check_layer(c, layer);
  if (rc) return rc;
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  return enqueue_step(c, layer, q, q, out, static_cast<cudaStream_t>(stream));
}

int spin_decode_step_host(spin_ctx* c, int32_t layer, const uint16_t* q_host, float* out_host, spin_stream_t stream) {
  if (!c) return fail(nullptr, SPIN_ERR_INVALID, "ctx is NULL");
  if (!q_host || !out_host) return fail(c, SPIN_ERR_INVALID, "q_host or out_host is NULL");
  int rc = check_layer(c, layer);
  if (rc) return rc;
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  LayerBuf& lb = c->layers[layer];
  const size_t nq = (size_t)c->B * c->Hq * kD;
  if (!lb.q_stage) {
    cudaError_t e;
    if ((e = dalloc(c, &lb.q_stage, nq)) != cudaSuccess) return cuda_fail(c, e, "allocating the query buffer");
    if ((e = dalloc(c, &lb.out_stage, nq)) != cudaSuccess) return cuda_fail(c, e, "allocating the output buffer");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Pinned, device-mapped buffers are used in place: the kernel first copies q over the host
  // link into HBM (idle warps, one release count), and the combine writes out into host
  // memory. A copy-engine transfer between two steps costs 11-17 us on
  // GB300 whatever its size; the zero-copy reads and writes cost a few. Pageable or
  // unaligned buffers go through HBM with cudaMemcpyAsync.
  const uint16_t* q_dev_src = static_cast<const uint16_t*>(mapped_host(q_host, 8));
  float* out_dev = static_cast<float*>(const_cast<void*>(mapped_host(out_host, 16)));
  if (!q_dev_src)
    SPIN_CUDA(c, cudaMemcpyAsync(lb.q_stage, q_host, nq * 2, cudaMemcpyHostToDevice, st), "copying q to the device");
  rc = enqueue_step(c, layer, lb.q_stage, q_dev_src ? q_dev_src : lb.q_stage, out_dev ? out_dev : lb.out_stage, st);
  if (rc) return rc;
  if (!out_dev)
    SPIN_CUDA(c, cudaMemcpyAsync(out_host, lb.out_stage, nq * 4, cudaMemcpyDeviceToHost, st), "copying out to the host");
  return SPIN_OK;
}

int spin_stats(spin_ctx* c, spin_stats_t* out) {
  if (!c || !out) return fail(c, SPIN_ERR_INVALID, "ctx or out is NULL");
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  int rc = sync_ctx(c);
  unsigned long long st[8] = {0};
  int32_t live = 0;
  if (cudaMemcpy(st, c->d_stats, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_fail(c, cudaGetLastError(), "reading counters");
  {
    // live segments = set bits of the bitmap that are real segments
    const int64_t nwords = (c->S + 31) / 32;
    std::vector<uint32_t> bm(nwords);
    if (cudaMemcpy(bm.data(), c->d_bitmap, nwords * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      return cuda_fail(c, cudaGetLastError(), "reading the segment bitmap");
    if (c->S % 32) bm[nwords - 1] &= (1u << (c->S % 32)) - 1u;
    for (auto w : bm) live += __builtin_popcount(w);
  }
  memset(out, 0, sizeof(*out));
  out->steps = c->steps_host;
  out->hits = (int64_t)st[kStatHits];
  out->misses = (int64_t)st[kStatMisses];
  out->evictions = (int64_t)st[kStatEvictions];
  out->lru_rounds = (int64_t)st[kStatLruRounds];
  out->retrieved_bytes = out->misses * kPageBytes;
  out->selected_bytes = (int64_t)st[kStatSelected] * kPageBytes;
  out->live_segments = live;
  out->pool_segments = c->S;
  out->metadata_bytes = c->bytes_meta;
  out->flat_table_bytes = c->bytes_flat;
  out->hbm_pool_bytes = c->bytes_pool;
  out->host_store_bytes = c->bytes_store;
  out->summary_bytes = c->bytes_summ;
  out->timed_calls = c->timed_calls;
  out->ms_score = c->ms[0];
  out->ms_manage = c->ms[1];
  out->ms_pages = c->ms[2];
  out->ms_combine = c->ms[3];
  out->ms_kernel = c->ms[4];
  out->device_error = c->sticky;
  out->appended_tokens = c->appended;
  out->tail_flushes = (int64_t)st[kStatFlushes];
  return rc;
}

int spin_debug_export(spin_ctx* c, int32_t layer, spin_state_view* v) {
  if (!c || !v) return fail(c, SPIN_ERR_INVALID, "ctx or view is NULL");
  if (layer < 0 || layer >= c->L) return fail(c, SPIN_ERR_INVALID, "layer %d out of range", layer);
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  int rc = sync_ctx(c);
  LayerBuf& lb = c->layers[layer];
  const int64_t Ul = (int64_t)c->B * c->Hkv;
  const int64_t u0 = (int64_t)layer * Ul;
#define D2H(dst, src, bytes)                                                                \
  if (dst) {                                                                                \
    if (cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)                 \
      return cuda_fail(c, cudaGetLastError(), "copying debug state");                       \
  }
  D2H(v->keff, lb.keff, Ul * 4);
  D2H(v->sel, lb.sel, Ul * c->k * 4);
  D2H(v->sel_slot, lb.sel_slot, Ul * c->k * 4);
  D2H(v->sel_hit, lb.sel_hit, Ul * c->k);
  D2H(v->slot_part, c->d_slot_part + u0 * c->cap, Ul * c->cap * 4);
  D2H(v->last_use, c->d_last_use + u0 * c->cap, Ul * c->cap * 4);
  D2H(v->unit_info, lb.unit_info, Ul * 8 * 4);
  // the last step's buffer: step t writes buffer t & 1
  D2H(v->scores, lb.scores + (size_t)((c->layer_steps[layer] + 1) & 1) * Ul * c->P_max, Ul * c->P_max * 4);
  if (v->resolve || v->live_segs) {
    int32_t *dres = nullptr, *dlive = nullptr;
    if (cudaMalloc(&dres, std::max<int64_t>(1, Ul * c->P_max) * 4) != cudaSuccess ||
        cudaMalloc(&dlive, Ul * 4) != cudaSuccess) {
      cudaFree(dres);
      return cuda_fail(c, cudaGetLastError(), "allocating debug buffers");
    }
    cudaError_t e = launch_resolve_all(lb.args, dres, dlive, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess && v->resolve) e = cudaMemcpy(v->resolve, dres, Ul * c->P_max * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v->live_segs) e = cudaMemcpy(v->live_segs, dlive, Ul * 4, cudaMemcpyDeviceToHost);
    cudaFree(dres);
    cudaFree(dlive);
    if (e != cudaSuccess) return cuda_fail(c, e, "resolving the page table");
  }
#undef D2H
  return rc;
}

int spin_debug_read_page(spin_ctx* c, int32_t layer, int32_t b, int32_t h, int32_t slot, uint16_t* dst) {
  if (!c || !dst) return fail(c, SPIN_ERR_INVALID, "ctx or dst is NULL");
  const int slot_end = c->cap + (c->tail_mode ? 1 : 0);  // slot == cap: the unit's tail page
  if (layer < 0 || layer >= c->L || b < 0 || b >= c->B || h < 0 || h >= c->Hkv || slot < 0 || slot >= slot_end)
    return fail(c, SPIN_ERR_INVALID, "page coordinates out of range");
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  int rc = sync_ctx(c);
  const int64_t unit = ((int64_t)layer * c->B + b) * c->Hkv + h;
  const int64_t page = slot == c->cap ? c->units * c->cap + unit : unit * c->cap + slot;
  SPIN_CUDA(c, cudaMemcpy(dst, c->d_pool + page * kPageElems, kPageBytes, cudaMemcpyDeviceToHost), "copying a page");
  return rc;
}

int spin_debug_summaries(spin_ctx* c, int32_t layer, int32_t b, int32_t h, float* dst) {
  if (!c || !dst) return fail(c, SPIN_ERR_INVALID, "ctx or dst is NULL");
  if (layer < 0 || layer >= c->L || b < 0 || b >= c->B || h < 0 || h >= c->Hkv)
    return fail(c, SPIN_ERR_INVALID, "unit coordinates out of range");
  DeviceGuard g(c->device);
  if (!g.ok) return fail(c, SPIN_ERR_CUDA, "cannot select device %d", c->device);
  int rc = sync_ctx(c);
  const int64_t page0 =
      (int64_t)layer * c->pages_per_layer + (int64_t)c->Hkv * c->poff_b[b] + (int64_t)h * c->pstride_b[b];
  const int32_t P = c->P_lb[(size_t)layer * c->B + b];
  if (P > 0)
    SPIN_CUDA(c, cudaMemcpy(dst, c->d_summ + page0 * kD, (size_t)P * kD * 4, cudaMemcpyDeviceToHost),
              "copying summaries");
  return rc;
}

void spin_destroy(spin_ctx* c) {
  if (!c) return;
  {
    DeviceGuard g(c->device);
    cudaDeviceSynchronize();
    free_all(c);
  }
  delete c;
}

const char* spin_last_error(const spin_ctx* c) { return c ? c->msg.c_str() : g_create_error.c_str(); }

}  // extern "C"
