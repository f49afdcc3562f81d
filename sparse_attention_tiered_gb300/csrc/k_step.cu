// One decode step of one layer in one persistent kernel: Select (scores, per-KV-head
// top-k), the page manager (two-level resolve, bump, bucketed LRU, slot assignment),
// Retrieve (host -> HBM page copies), paged split-KV decode attention and combine.
//
// Select picks the critical partitions for the query, Retrieve brings the missing
// ones from CPU memory into HBM pages and Attention is exact softmax attention over
// the tokens of the selected partitions only (m.x-techcon.com SPIN article, section
// "Spin的核心设计" 1 and Figure 3, 2 and Figure 5 steps 1-4, 3 and Figure 6;
// gist.science/pt section 2A-2C). The pages give no kernel design; everything below
// is this library's.
//
// The kernel is cooperative (every CTA is resident, one per SM). With zero-copy
// queries (pinned host memory) every warp first copies a few units' query rows into
// HBM and counts them with one release; scorers and producers acquire that count. Its
// work, per CTA:
//   A. scoring: fp32 scores of 8-row batches of partition summaries, written to this
//      step's score buffer (two buffers, alternating by step);
//   B. managing: groups of GS threads claim units in order; once a unit's scores are
//      all in, a group runs its top-k and the page manager, reserves the unit's entries
//      in the step's miss list, writes them, the attention order and the page state
//      with plain stores, and publishes them with one release fence followed by the
//      entries' tags and the unit's ready flag;
//   C. retrieval and attention:
//      * retriever warps walk the miss list as entries appear (host page -> HBM slot,
//        16-byte zero-copy loads over the host link); the first entries of a step are
//        copied in four pieces by four warps; a page's (last piece's) lane 0 raises its
//        ready flag with one release, the warp barrier ordering its lanes' stores;
//      * two consumer groups of four warps take alternate stages of a shared-memory
//        ring guarded by mbarriers, so two pages are in the math at once;
//      * each consumer group has a producer warp that stages its pages through TMA:
//        first resident pages (hits) in tasks of up to `ppt` pages of one unit (after
//        the unit's ready flag), then retrieved pages in miss-list order, each after
//        an acquire of its ready flag.
// Two variants. Pipelined (PIPE): A, B and C run at once in different warps of every
// CTA; scoring batches are dealt round-robin in unit-major order so units complete one
// after another, and a manager group starts on a unit when no slot of its score row
// still holds the empty-slot sentinel (and sets the unit's slots of the other buffer
// back to it). Phased: A over contiguous row ranges (a unit's row counter, added with a
// release as a warp leaves the unit; wide units also count their keys' top 12 bits),
// then B in the CTA's manager groups overlaying the ring, then C.
// So retrieval starts as soon as the first units are managed, the attention over the
// hits (HBM bound) hides under the retrieval (host-link bound) and each retrieved page
// is attended as soon as it lands (and from L2). When every CTA is done with its
// pages (an arrival counter), every consumer warp combines (unit, query head) pairs.
// Memory ordering uses as few GPU-scope ordering points as the protocol needs: a fence
// waits for the thread's earlier accesses, which on an SM with host-link loads queued
// takes many microseconds; polls end with one acquire load.
//
// Attention data layout. A page (32 KiB) holds K[64][128] then V[64][128] bf16.
// A TMA tensor map views the whole HBM pool as a 2-D bf16 tensor of 128 columns
// and (slots * 128) rows; a page is loaded as four 64x64 boxes (K left/right, V
// left/right) with the 128-byte swizzle, so ldmatrix reads are bank-conflict
// free. The first page of a task also brings the unit's G query rows (bulk copy).
//
// Consumer math. Every consumer warp handles 16 of the 64 tokens of each page for
// all G query heads of the unit, with tokens as the M dimension:
//   S^T[16 tokens][8 heads] = K Q^T        mma.m16n8k16 bf16 -> fp32 (heads padded to 8)
//   online softmax per head in fp32 (base-2 exponent, scale log2(e)/sqrt(128))
//   O^T[128][8 heads] += V^T P             P transposed in registers (movmatrix) and
//                                          split into bf16 hi + lo parts, two mma each
// At the end of a task the group's four warps merge (m, l, O) in the stage of the
// task's last page and write one partial (m, l, acc[128]) per query head; the
// combine computes out_g = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
//
// Every wait (scored rows, unit and miss-list flags, mbarriers, page flags, the
// arrival counter) is bounded in time; a wait that runs out sets the device error
// word, after which every other wait gives up at once, stops issuing work and drains
// the copies already issued.
#include "select_dev.cuh"
#include "spin_internal.cuh"

namespace spin {

namespace {

constexpr int kStages = 6;    // ring stages (stage i belongs to consumer group i % groups)
constexpr int kStagesPipe = 4;  // the pipelined kernel's ring: the manager group's shared memory sits beside it
constexpr int kCWarps = 4;    // consumer warps of one group: 16 tokens of a page each
constexpr int kMaxGroups = 2;
// Stage i of the ring belongs to consumer group i % groups for good: the stage count is a
// multiple of the group count, so each stage's barriers see one group's uses only, in order,
// and a parity wait is never more than one phase away from the barrier's current phase.
static_assert(kStages % kMaxGroups == 0 && kStagesPipe % kMaxGroups == 0, "stages must split evenly between groups");
// Roles per CTA. One 8-head tile (NT = 1, at most 128 registers a thread): two
// consumer groups that take alternate ring stages, so two pages are in the math at
// once, each fed by its own producer warp, and six retriever warps (two saturate the
// host link alone). Two tiles (G > 8, 168 registers): one group, one producer, four
// retrievers. Threads x registers stay within 64 K.
template <int NT>
struct Roles {
  static constexpr int kGroups = NT == 1 ? 2 : 1;
  static constexpr int kConsumers = kCWarps * kGroups;
  static constexpr int kRWarps = NT == 1 ? 6 : 4;
  static constexpr int kThreads = (kGroups + kConsumers + kRWarps) * 32;
};
constexpr int kQBytes = kMaxGroup * kD * 2;            // query rows of one unit (<= 16 heads)
constexpr int kStageBytes = kPageBytes + kQBytes;       // 36 KiB, a multiple of 1024
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kMergeRow = kD + 4;                       // padded row of the merge buffer
constexpr int kMergeFloats = 16 * kMergeRow + 32;       // O[16 heads][128+4], m[16], l[16]
static_assert(kCWarps * kMergeFloats * 4 <= kStageBytes, "a task's merge must fit in its last page's stage");
constexpr float kScaleLog2 = 0.12751743074173449f;      // log2(e) / sqrt(128)
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s

struct StageMeta {
  int part, ul, valid, first, last;  // partial slot of the task, unit, valid tokens, first / last page of the task
};

// Dynamic shared memory: a header (barriers, stage descriptors, flags) then, 1024-byte
// aligned, the region that holds the manager groups in phase B and the ring in phase C.
struct StepSmem {
  uint64_t* full;     // [kStages]
  uint64_t* empty;    // [kStages]
  uint64_t* mrg;      // [groups][2]: written, read
  StageMeta* meta;    // [kStages]
  int* abort_flag;
  int* hits_done;     // set once every producer of this CTA has issued its resident-page tasks
  int* hits_groups;   // producers past their resident pages
  int* tl_count;      // [2] stage timing: scoring warps done, combining warps done
  uint8_t* region;    // ring (kStages x kStageBytes) / manager groups
};

constexpr size_t kHeaderBytes = 1024;

__host__ __device__ inline void step_smem_layout(StepSmem* s, uint8_t* base) {
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = (off + align - 1) & ~(align - 1);
    uint8_t* p = base + off;
    off += bytes;
    return p;
  };
  s->full = (uint64_t*)take(sizeof(uint64_t) * kStages, 8);
  s->empty = (uint64_t*)take(sizeof(uint64_t) * kStages, 8);
  s->mrg = (uint64_t*)take(sizeof(uint64_t) * 2 * kMaxGroups, 8);
  s->meta = (StageMeta*)take(sizeof(StageMeta) * kStages, 16);
  s->abort_flag = (int*)take(sizeof(int), 4);
  s->hits_done = (int*)take(sizeof(int), 4);
  s->hits_groups = (int*)take(sizeof(int), 4);
  s->tl_count = (int*)take(sizeof(int) * 2, 4);
  s->region = base + kHeaderBytes;
}
static_assert(sizeof(uint64_t) * (2 * kStages + 2 * kMaxGroups) + sizeof(StageMeta) * kStages + 64 <= kHeaderBytes,
              "header overflow");

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until the phase with the given parity has completed; false after kWaitNs.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *p reaches `want` (== when exact, else >=), bounded by kWaitNs, or (err != nullptr)
// until another wait has run out (the timeout bit of the error word). Polls with relaxed loads and a short
// sleep, then one acquire fence: acquire loads and fences in a tight loop hold up the SM's
// other memory traffic (the retrievers' host loads).
__device__ __noinline__ bool wait_flag(const int* p, int want, bool exact, const uint32_t* err) {
  auto hit = [&](int v) { return exact ? v == want : v >= want; };
  bool ok = hit(ld_relaxed(p));
  if (!ok) {
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30) && !ok; ++it) {
      __nanosleep(128);
      ok = hit(ld_relaxed(p));
      if (!ok && (it & 63u) == 0 &&
          (globaltimer_ns() - t0 > kWaitNs || (err != nullptr && (ld_relaxed_u32(err) & kErrTimeout))))
        break;
    }
  }
  if (ok) (void)ld_acquire(p);  // an acquire load, not a fence: nothing earlier to wait for
  return ok;
}

// Zero-copy queries: staging warp sw of nsw copies the query rows of units sw, sw + nsw, ...
// from host memory into q (HBM), one 256-byte row per warp access, and counts them in
// kCtrQStaged with one release (the warp barrier orders every lane's stores before it).
__device__ __noinline__ void stage_queries(const LayerArgs& a, int sw, int nsw, int lane) {
  const int U = a.B * a.Hkv;
  int done = 0;
  for (int u = sw; u < U; u += nsw) {
    const int64_t q0 = ((int64_t)(u / a.Hkv) * a.Hq + (int64_t)(u % a.Hkv) * a.G) * kD;
    const uint2* src = reinterpret_cast<const uint2*>(a.q_src + q0);
    uint2* dst = reinterpret_cast<uint2*>(const_cast<uint16_t*>(a.q) + q0);
    for (int g0 = 0; g0 < a.G; g0 += 4) {
      uint2 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (g0 + i < a.G) v[i] = src[(g0 + i) * (kD / 4) + lane];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (g0 + i < a.G) dst[(g0 + i) * (kD / 4) + lane] = v[i];
    }
    ++done;
  }
  __syncwarp();
  if (lane == 0 && done) red_release_add(a.counters + kCtrQStaged, done);
}

// Zero-copy queries: returns once every unit's rows are in q (bounded; a wait that runs
// out sets the time-out bit, and the step's results are not used).
__device__ __forceinline__ void await_queries(const LayerArgs& a, int lane) {
  if (a.q_src == a.q) return;
  int ok = 1;
  if (lane == 0) ok = wait_flag(a.counters + kCtrQStaged, a.B * a.Hkv, false, a.err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
  __syncwarp();
  (void)ld_acquire(a.counters + kCtrQStaged);
}

// State of miss-list entry m of this step: 1 = written (its fields may be read after an
// acquire), 0 = past the end of the step's final list, -1 = the bounded wait ran out.
// The list is final once every unit of the layer is managed.
__device__ __noinline__ int miss_entry(const LayerArgs& a, int m, int tag, int U, int kmax) {
  if (m >= kmax) return 0;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (ld_relaxed(a.miss_tag + m) == tag) return 1;
    if (ld_relaxed(a.counters + kCtrManaged) >= U) {
      (void)ld_acquire(a.counters + kCtrManaged);
      if (m >= ld_relaxed(a.counters + kCtrMiss)) return 0;
      continue;  // every entry below the final count is published before its unit: the tag is there
    }
    if ((it & 63u) == 63u && (globaltimer_ns() - t0 > kWaitNs || (ld_relaxed_u32(a.err) & kErrTimeout))) return -1;
    __nanosleep(64);
  }
  return -1;
}

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo_f(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Byte offset of 16-byte chunk `cd` (0..15) of row `r` (0..63) of a page half,
// as written by TMA with the 128-byte swizzle into two 8 KiB 64x64 boxes.
__device__ __forceinline__ uint32_t swz(int r, int cd) {
  return (uint32_t)((cd >> 3) * 8192 + r * 128 + (((cd & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------
// Combine of one (unit, query head): out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c
// over the unit's partials (its hit tasks and its retrieved pages), by one warp, four
// columns per lane, in one online pass: 16 partials at a time, their (m, l) and
// accumulator rows all loaded before use, folded into a running maximum.
// ---------------------------------------------------------------------------
__device__ void combine_head(const LayerArgs& a, int ul, int g, int lane) {
  constexpr int kBatch = 16;
  const int b = ul / a.Hkv, h = ul - b * a.Hkv;
  const int has_tail = (a.tail_n != nullptr && a.tail_n[b] > 0) ? 1 : 0;
  const int keff = __ldcg(a.keff + ul) + has_tail, nh = __ldcg(a.n_hit + ul);  // attended; resident (tail incl.)
  const int nc = (nh + a.ppt - 1) / a.ppt;
  const int U = a.B * a.Hkv;
  const int n = nc + (keff - nh);
  float4* out = reinterpret_cast<float4*>(a.out + ((int64_t)b * a.Hq + (int64_t)h * a.G + g) * kD);
  // partial slots: hit tasks ul * n_chunks + c (c < nc), retrieved pages U * n_chunks + ul * ka + j (nh <= j < keff)
  auto part_ptr = [&](int i) -> const float* {
    const int64_t slot =
        i < nc ? (int64_t)ul * a.n_chunks + i : (int64_t)U * a.n_chunks + (int64_t)ul * a.ka + nh + (i - nc);
    return a.partials + (slot * a.G + g) * kPartialStride;
  };
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < n; i0 += kBatch) {
    float m_l = -INFINITY, l_l = 0.f;  // lane u < kBatch: partial i0 + u
    if (lane < kBatch && i0 + lane < n) {
      const float* pp = part_ptr(i0 + lane);
      m_l = __ldcg(pp);
      l_l = __ldcg(pp + 1);
    }
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      v[u] = (i0 + u < n) ? __ldcg(reinterpret_cast<const float4*>(part_ptr(i0 + u) + 4) + lane)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    float Mc = m_l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o));
    const float Mn = fmaxf(M, Mc);
    if (Mn == -INFINITY) continue;  // nothing attended so far
    const float al = exp2f(M - Mn);  // M = -inf gives 0
    const float sc_l = exp2f(m_l - Mn);  // lanes without a partial: m = -inf gives 0
    float ls = sc_l * l_l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    L = fmaf(L, al, ls);
    acc.x *= al;
    acc.y *= al;
    acc.z *= al;
    acc.w *= al;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const float sc = __shfl_sync(0xffffffffu, sc_l, u);
      acc.x = fmaf(sc, v[u].x, acc.x);
      acc.y = fmaf(sc, v[u].y, acc.y);
      acc.z = fmaf(sc, v[u].z, acc.z);
      acc.w = fmaf(sc, v[u].w, acc.w);
    }
    M = Mn;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  out[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// Combine of one (unit, query head) by the nw consumer warps of a CTA (named barrier
// `bar`), for units with many partials: warp w folds partials w, w + nw, ... (their loads
// all in flight at once) into (M_w, L_w, acc_w), the warps' results meet in shared memory
// `red` and are folded again: out = sum_w 2^(M_w - M) acc_w / sum_w 2^(M_w - M) L_w.
__device__ void combine_head_cta(const LayerArgs& a, int ul, int g, int w, int nw, int lane, float* red, int bar) {
  const int b = ul / a.Hkv, h = ul - b * a.Hkv;
  const int has_tail = (a.tail_n != nullptr && a.tail_n[b] > 0) ? 1 : 0;
  const int keff = __ldcg(a.keff + ul) + has_tail, nh = __ldcg(a.n_hit + ul);
  const int nc = (nh + a.ppt - 1) / a.ppt;
  const int U = a.B * a.Hkv;
  const int n = nc + (keff - nh);
  auto part_ptr = [&](int i) -> const float* {
    const int64_t slot =
        i < nc ? (int64_t)ul * a.n_chunks + i : (int64_t)U * a.n_chunks + (int64_t)ul * a.ka + nh + (i - nc);
    return a.partials + (slot * a.G + g) * kPartialStride;
  };
  constexpr int kMaxPer = 8;
  float Mw = -INFINITY, Lw = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = w; i0 < n; i0 += kMaxPer * nw) {
    float m[kMaxPer], l[kMaxPer];
    float4 v[kMaxPer];
#pragma unroll
    for (int u = 0; u < kMaxPer; ++u) {
      const int i = i0 + u * nw;
      if (i < n) {
        const float* pp = part_ptr(i);
        m[u] = __ldcg(pp);
        l[u] = __ldcg(pp + 1);
        v[u] = __ldcg(reinterpret_cast<const float4*>(pp + 4) + lane);
      } else {
        m[u] = -INFINITY;
        l[u] = 0.f;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mn = Mw;
#pragma unroll
    for (int u = 0; u < kMaxPer; ++u) Mn = fmaxf(Mn, m[u]);
    if (Mn != -INFINITY) {
      const float al = exp2f(Mw - Mn);  // Mw = -inf gives 0
      Lw *= al;
      acc.x *= al;
      acc.y *= al;
      acc.z *= al;
      acc.w *= al;
#pragma unroll
      for (int u = 0; u < kMaxPer; ++u) {
        const float sc = exp2f(m[u] - Mn);  // padding entries: m = -inf gives 0
        Lw = fmaf(sc, l[u], Lw);
        acc.x = fmaf(sc, v[u].x, acc.x);
        acc.y = fmaf(sc, v[u].y, acc.y);
        acc.z = fmaf(sc, v[u].z, acc.z);
        acc.w = fmaf(sc, v[u].w, acc.w);
      }
      Mw = Mn;
    }
  }
  float* rw = red + w * (kD + 4);
  reinterpret_cast<float4*>(rw + 4)[lane] = acc;
  if (lane == 0) {
    rw[0] = Mw;
    rw[1] = Lw;
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nw * 32) : "memory");
  if (w == 0) {
    float M = -INFINITY;
    for (int ww = 0; ww < nw; ++ww) M = fmaxf(M, red[ww * (kD + 4)]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int ww = 0; ww < nw; ++ww) {
        const float* r = red + ww * (kD + 4);
        const float sc = exp2f(r[0] - M);
        L = fmaf(sc, r[1], L);
        const float4 x = reinterpret_cast<const float4*>(r + 4)[lane];
        o.x = fmaf(sc, x.x, o.x);
        o.y = fmaf(sc, x.y, o.y);
        o.z = fmaf(sc, x.z, o.z);
        o.w = fmaf(sc, x.w, o.w);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    reinterpret_cast<float4*>(a.out + ((int64_t)b * a.Hq + (int64_t)h * a.G + g) * kD)[lane] =
        make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nw * 32) : "memory");
}

// ---------------------------------------------------------------------------
// The decode-step kernel. NT = number of 8-head tiles (G <= 8 * NT); GS = threads of
// one manager group in phase B.
// ---------------------------------------------------------------------------
template <int NT, int GS, bool PIPE>
__global__ void __launch_bounds__(Roles<NT>::kThreads, 1)
decode_step_kernel(const __grid_constant__ CUtensorMap tmap, LayerArgs a, int n_hit_tasks) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  StepSmem sm;
  step_smem_layout(&sm, base);
  constexpr int kThreads = Roles<NT>::kThreads;
  constexpr int kSt = PIPE ? kStagesPipe : kStages;  // ring stages
  static_assert(kSt % Roles<NT>::kGroups == 0, "each ring stage must belong to one consumer group");
  constexpr int NG = Roles<NT>::kGroups, NC = Roles<NT>::kConsumers;
  constexpr int kWarps = kThreads / 32;
  constexpr uint32_t kAll = 0xffffffffu;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = a.counters[kCtrStep];
  const int tag = t + 1;  // flag value of this step (flags are never reset)
  const int U = a.B * a.Hkv;
  const int kmax = U * a.k;  // miss-list capacity
  float* sc_cur = a.scores + (int64_t)(t & 1) * U * a.P_max;  // this step's score buffer
  unsigned long long* tl = a.timeline;

  if (tid == 0) {
    if (tl) atomicMax(tl + 0, ~globaltimer_ns());
    for (int s = 0; s < kSt; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kCWarps);  // the four warps of the stage's group
    }
    for (int m = 0; m < 2 * NG; ++m) mbar_init(smem_u32(&sm.mrg[m]), kCWarps);
    *sm.abort_flag = 0;
    *sm.hits_done = 0;
    *sm.hits_groups = 0;
    sm.tl_count[0] = sm.tl_count[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  if constexpr (PIPE) {
    // ------------------------------ A + B, pipelined ------------------------------
    // Warps 0 .. NC+NG-1 (consumers and producers) score batches of up to 8 partitions
    // of one unit, batch j of the layer (unit-major order) going to scoring warp
    // j mod (grid x (NC+NG)), so units complete in order across the grid; each then
    // takes its phase-C role. Warps NC+NG .. NC+NG+3 form manager groups (one of four
    // warps, or four of one) that claim units in order as soon as they are complete
    // (no slot of the unit's score row still empty), then join the retrievers; the
    // remaining retriever warps start on the miss list at once.
    constexpr int kMgrWarps = 4;
    constexpr int kMgrGroups = kMgrWarps * 32 / GS;
    const size_t gbytes = sel::mgr_smem_layout(GS, a.P_max, a.cap, a.k, a.D, nullptr, nullptr);
    uint8_t* mreg = sm.region + (size_t)kSt * kStageBytes;
    int* s_pre = reinterpret_cast<int*>(mreg + kMgrGroups * gbytes);  // [B + 1] batches before request b
    // zero-copy queries: every warp of the grid copies at most a few units' rows first
    if (a.q_src != a.q)
      stage_queries(a, (int)blockIdx.x * kWarps + warp, (int)gridDim.x * kWarps, lane);
    if (warp == 0) {
      int run = 0;
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        const int v = b < a.B ? a.Hkv * ((a.P_b[b] + sel::kRowsPerBatch - 1) / sel::kRowsPerBatch) : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kAll, x, o);
          if (lane >= o) x += y;
        }
        if (b < a.B) s_pre[b] = run + x - v;
        run += __shfl_sync(kAll, x, 31);
      }
      if (lane == 0) s_pre[a.B] = run;
    }
    __syncthreads();
    float* sc_next = a.scores + (int64_t)((t + 1) & 1) * U * a.P_max;
    if (warp < NC + NG) {
      const int nbatch = s_pre[a.B];
      const int SWp = (int)gridDim.x * (NC + NG);
      // request, head, first partition and row count of batch jj
      auto locate = [&](int jj, int& b, int& h, int& p0, int& n) {
        int lo = 0, hi = a.B;  // the largest b with s_pre[b] <= jj
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_pre[mid] <= jj) lo = mid;
          else hi = mid;
        }
        b = lo;
        const int Pb = a.P_b[b];
        const int nb = (Pb + sel::kRowsPerBatch - 1) / sel::kRowsPerBatch;
        const int off = jj - s_pre[b];
        h = off / nb;
        p0 = (off - h * nb) * sel::kRowsPerBatch;
        n = min(sel::kRowsPerBatch, Pb - p0);
      };
      int j = (int)blockIdx.x * (NC + NG) + warp;
      if (j < nbatch) {
        int b, h, p0, n;
        locate(j, b, h, p0, n);
        float4 cur[sel::kRowsPerBatch], nxt[sel::kRowsPerBatch];
        sel::load_rows(cur, reinterpret_cast<const float4*>(a.summ + host_page_index(a, b, h, p0) * kD), n, lane);
        await_queries(a, lane);
        float4 qv = sel::qsum_lane(a.q + ((int64_t)b * a.Hq + (int64_t)h * a.G) * kD, a.G, lane, a.q_src != a.q);
        for (;;) {
          const int j2 = j + SWp;
          const bool more = j2 < nbatch;
          int b2 = 0, h2 = 0, p2 = 0, n2 = 0;
          if (more) {
            locate(j2, b2, h2, p2, n2);
            sel::load_rows(nxt, reinterpret_cast<const float4*>(a.summ + host_page_index(a, b2, h2, p2) * kD), n2, lane);
          }
          const float x = sel::score_batch(cur, qv, lane);
          if (lane < n) sc_cur[(int64_t)(b * a.Hkv + h) * a.P_max + p0 + lane] = x;
          if (!more) break;
          if (b2 != b || h2 != h) qv = sel::qsum_lane(a.q + ((int64_t)b2 * a.Hq + (int64_t)h2 * a.G) * kD, a.G, lane, a.q_src != a.q);
          j = j2;
          b = b2;
          h = h2;
          p0 = p2;
          n = n2;
#pragma unroll
          for (int i = 0; i < sel::kRowsPerBatch; ++i) cur[i] = nxt[i];
        }
      }
      // stage timing: the CTA's last scoring warp stamps (one global atomic per CTA)
      if (tl && lane == 0 && atomicAdd(sm.tl_count, 1) == NC + NG - 1) atomicMax(tl + kTlScored, globaltimer_ns());
    } else if (warp < NC + NG + kMgrWarps) {
      const int grp = (tid - (NC + NG) * 32) / GS, gt = tid - (NC + NG) * 32 - grp * GS;
      const int bar = 1 + grp;
      sel::MgrSmem ms;
      sel::mgr_smem_layout(GS, a.P_max, a.cap, a.k, a.D, &ms, mreg + grp * gbytes);
      for (;;) {
        if (gt == 0) ms.gs->unit = atomicAdd(&a.counters[kCtrManage], 1);
        sel::gsync<GS>(bar);
        const int ul = ms.gs->unit;
        sel::gsync<GS>(bar);
        if (ul >= U) break;
        // wait until no slot of the unit's score row is empty (bounded)
        const int P = a.P_b[ul / a.Hkv];
        const float* sc = sc_cur + (int64_t)ul * a.P_max;
        const unsigned long long t0 = globaltimer_ns();
        bool ok = true;
        for (uint32_t it = 0;; ++it) {
          bool empty = false;
          for (int p = gt; p < P; p += GS) empty |= __float_as_uint(__ldcg(sc + p)) == kScoreEmpty;
          const bool any = __any_sync(kAll, empty);
          if (gt == 0) ms.gs->ok = 0;
          sel::gsync<GS>(bar);
          if (any && lane == 0) atomicOr(&ms.gs->ok, 1);
          if (gt == 0 && (it & 15u) == 15u &&
              (globaltimer_ns() - t0 > kWaitNs || (ld_relaxed_u32(a.err) & kErrTimeout)))
            atomicOr(&ms.gs->ok, 2);
          sel::gsync<GS>(bar);
          const int st = ms.gs->ok;
          sel::gsync<GS>(bar);
          if (st == 0) break;
          if (st & 2) {
            ok = false;
            break;
          }
          __nanosleep(200);
        }
        if (!ok) {
          if (gt == 0) {
            atomicOr(a.err, kErrTimeout);
            // publish the unit with nothing selected, so nobody waits for it
            a.keff[ul] = 0;
            a.n_hit[ul] = 0;
            sel::publish_unit(a, ul, tag);
          }
          continue;
        }
        sel::manage_unit<GS>(a, ul, t, tag, ms, bar, gt, sc, sc_next + (int64_t)ul * a.P_max);
        if (tl && gt == 0) atomicMax(tl + kTlManaged, globaltimer_ns());
      }
    }
  } else {
  // ------------------------------ A. scoring ------------------------------
  // The layer's partitions, request-major then head then partition, are split into
  // equal contiguous row ranges, one per warp of the grid. A warp scores its range in
  // batches of up to 8 rows of one unit, the next batch's loads in flight while the
  // current one is reduced; it adds its rows to a unit's counter (release) when it
  // leaves the unit. Wide units also count their keys' top 12 bits.
  {
    int64_t* s_pre = reinterpret_cast<int64_t*>(sm.region);  // [B + 1] rows before request b
    if (warp == 0) {
      int64_t run = 0;
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        const int64_t v = b < a.B ? (int64_t)a.Hkv * a.P_b[b] : 0;
        int64_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t y = __shfl_up_sync(kAll, x, o);
          if (lane >= o) x += y;
        }
        if (b < a.B) s_pre[b] = run + x - v;
        run += __shfl_sync(kAll, x, 31);
      }
      if (lane == 0) s_pre[a.B] = run;
    }
    __syncthreads();
    const int64_t R = s_pre[a.B];
    const int64_t TW = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    if (a.q_src != a.q) stage_queries(a, (int)gw, (int)TW, lane);
    int64_t r = R * gw / TW;
    const int64_t r_end = R * (gw + 1) / TW;
    if (r < r_end) {
      int lo = 0, hi = a.B;  // the request of row r: the largest b with s_pre[b] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid] <= r) lo = mid;
        else hi = mid;
      }
      int b = lo, Pb = a.P_b[b];
      const int64_t off = r - s_pre[b];
      int h = (int)(off / Pb), p = (int)(off - (int64_t)h * Pb);
      int n = (int)min((int64_t)min(sel::kRowsPerBatch, Pb - p), r_end - r);
      float4 cur[sel::kRowsPerBatch], nxt[sel::kRowsPerBatch];
      sel::load_rows(cur, reinterpret_cast<const float4*>(a.summ + host_page_index(a, b, h, p) * kD), n, lane);
      await_queries(a, lane);
      float4 qv = sel::qsum_lane(a.q + ((int64_t)b * a.Hq + (int64_t)h * a.G) * kD, a.G, lane, a.q_src != a.q);
      int counted = 0;
      for (;;) {
        // the next batch: the rest of this unit, else the start of the next non-empty unit
        const int64_t r2 = r + n;
        const bool more = r2 < r_end;
        int b2 = b, h2 = h, p2 = p + n, Pb2 = Pb, n2 = 0;
        if (more) {
          if (p2 >= Pb) {
            p2 = 0;
            if (++h2 == a.Hkv) {
              h2 = 0;
              do {
                Pb2 = a.P_b[++b2];
              } while (Pb2 == 0);
            }
          }
          n2 = (int)min((int64_t)min(sel::kRowsPerBatch, Pb2 - p2), r_end - r2);
          sel::load_rows(nxt, reinterpret_cast<const float4*>(a.summ + host_page_index(a, b2, h2, p2) * kD), n2, lane);
        }
        const int ul = b * a.Hkv + h;
        const float x = sel::score_batch(cur, qv, lane);
        if (lane < n) {
          sc_cur[(int64_t)ul * a.P_max + p + lane] = x;
          if (a.hist12) atomicAdd(a.hist12 + (int64_t)ul * sel::kHistBins + (sel::float_key(x) >> (32 - sel::kHistBits)), 1);
        }
        counted += n;
        const bool leave = !more || b2 != b || h2 != h;
        if (leave) {
          __syncwarp();
          if (lane == 0) red_release_add(a.unit_rows + ul, counted);
          counted = 0;
        }
        if (!more) break;
        if (leave) qv = sel::qsum_lane(a.q + ((int64_t)b2 * a.Hq + (int64_t)h2 * a.G) * kD, a.G, lane, a.q_src != a.q);
        r = r2;
        b = b2;
        h = h2;
        p = p2;
        Pb = Pb2;
        n = n2;
#pragma unroll
        for (int i = 0; i < sel::kRowsPerBatch; ++i) cur[i] = nxt[i];
      }
    }
  }
  __syncthreads();
  if (tl && tid == 0) atomicMax(tl + 1, globaltimer_ns());

  // ------------------------------ B. managing ------------------------------
  {
    constexpr int kGroupsB = kThreads / GS;
    const int grp = tid / GS, gt = tid - grp * GS;
    if (grp < kGroupsB) {
      sel::MgrSmem ms;
      const size_t gbytes = sel::mgr_smem_layout(GS, a.P_max, a.cap, a.k, a.D, nullptr, nullptr);
      sel::mgr_smem_layout(GS, a.P_max, a.cap, a.k, a.D, &ms, sm.region + (size_t)grp * gbytes);
      const int bar = 1 + grp;
      for (;;) {
        if (gt == 0) {
          int ul = atomicAdd(&a.counters[kCtrManage], 1);
          int ok = 1;
          if (ul < U) {
            // wait until every partition of the unit is scored
            const int P = a.P_b[ul / a.Hkv];
            ok = wait_flag(a.unit_rows + ul, P, false, a.err) ? 1 : 0;
            a.unit_rows[ul] = 0;  // every row of this step is in: ready for the next step
          }
          ms.gs->unit = ul;
          ms.gs->ok = ok;
        }
        sel::gsync<GS>(bar);
        const int ul = ms.gs->unit;
        const int ok = ms.gs->ok;
        sel::gsync<GS>(bar);
        if (ul >= U) break;
        if (!ok) {
          if (gt == 0) {
            atomicOr(a.err, kErrTimeout);
            // publish the unit with nothing selected, so nobody waits for it
            a.keff[ul] = 0;
            a.n_hit[ul] = 0;
            sel::publish_unit(a, ul, tag);
          }
          continue;
        }
        sel::manage_unit<GS>(a, ul, t, tag, ms, bar, gt, sc_cur + (int64_t)ul * a.P_max, nullptr);
        if (tl && gt == 0) atomicMax(tl + 2, globaltimer_ns());
      }
    }
  }
  // the manager groups wrote the region with generic stores; TMA writes it next
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  }
  volatile int* abort_flag = sm.abort_flag;

  // ------------------------------ C. retrieval + attention ------------------------------
  if (warp >= NC + NG) {
    // ------------------------------ retrievers ------------------------------
    // kEarly warps copy from the start; the others join once this CTA's resident pages
    // are issued (so they do not slow the HBM-bound hits).
    const int rw = warp - NC - NG;
    bool active = PIPE ? a.retr_warps > 0 : rw < a.retr_warps;
    if (!PIPE && !active && rw < a.retr_warps + a.retr_late) {
      volatile int* hd = sm.hits_done;
      const unsigned long long t0 = globaltimer_ns();
      for (uint32_t it = 1; it < (1u << 30) && !*hd; ++it) {
        __nanosleep(256);
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitNs) break;
      }
      active = *hd != 0 && !*abort_flag;
    }
    constexpr int kVec = kPageBytes / 16;  // 2048 x 16 B
    constexpr int kUnroll = 16;            // 16 x 16 B in flight per lane
    constexpr int kPieceVec = kVec / kRetrChunks;
    static_assert(kPieceVec % (32 * kUnroll) == 0 && (kRetrChunks & (kRetrChunks - 1)) == 0, "piece layout");
    const int split = a.retr_split;
    for (; active;) {
      // claim i: pieces of the first `split` entries, then whole pages (m is non-decreasing in i)
      int i = 0;
      if (lane == 0) i = atomicAdd(&a.counters[kCtrRetrieve], 1);
      i = __shfl_sync(kAll, i, 0);
      const bool piece = i < split * kRetrChunks;
      const int m = piece ? i / kRetrChunks : split + (i - split * kRetrChunks);
      const int v0 = piece ? (i % kRetrChunks) * kPieceVec : 0, v1 = piece ? v0 + kPieceVec : kVec;
      int st = 0;
      if (lane == 0) st = miss_entry(a, m, tag, U, kmax);
      st = __shfl_sync(kAll, st, 0);
      if (st == 0) break;
      if (st < 0) {
        if (lane == 0) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      __syncwarp();
      (void)ld_acquire(a.miss_tag + m);
      const int64_t sp = __ldcg(a.miss_src + m), dp = __ldcg(a.miss_dst + m);
      const bool in_range = sp >= 0 && sp < a.host_pages && dp >= 0 && dp < a.pool_slots;
      if (!in_range && lane == 0) atomicOr(a.err, kErrIndex);  // never expected: skip the copy
      const uint4* src = reinterpret_cast<const uint4*>(a.host_store + sp * kPageElems);
      uint4* dst = reinterpret_cast<uint4*>(a.pool + dp * kPageElems);
#pragma unroll 1
      for (int c = v0; in_range && c < v1; c += 32 * kUnroll) {
        uint4 r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) r[u] = __ldcs(src + c + u * 32 + lane);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) dst[c + u * 32 + lane] = r[u];
      }
      // every lane's stores are ordered before lane 0's release by the warp barrier (the
      // release is cumulative): one GPU-scope ordering point per piece, not one per lane
      __syncwarp();
      if (lane == 0) {
        // a split entry's flag goes up with its last piece: the counter grows by kRetrChunks
        // every step, so the piece that brings it to a multiple of kRetrChunks is the last
        // (its acq_rel add sees the other pieces' stores, and the release store passes them on)
        const bool last = !piece || ((atom_add_acq_rel(a.ready_cnt + m, 1u) + 1u) & (kRetrChunks - 1)) == 0;
        if (last) st_release(a.ready + m, tag);
      }
    }
  } else if (warp >= NC) {
    // ------------------------------ producers ------------------------------
    // Producer warp g feeds consumer group g: stage indices i = g, g + NG, ... use ring
    // stage i % kSt. Its stream: resident-page tasks (up to ppt pages of one unit,
    // claimed from a shared counter, after the unit's ready flag), then retrieved pages
    // (one page each, in miss-list order, once the entry is written and its page
    // published), then a sentinel.
    // The whole warp runs the loop so that nothing the issue path needs is a fresh
    // global load: tasks are claimed two ahead, the next task's page descriptors load
    // into the lanes' registers (lane j: page j) while the current task issues (if its
    // unit is managed by then; else when it becomes current), and the next retrieved
    // page's miss-list entry loads before its flag is awaited. Lane 0 alone waits on
    // the ring barriers and issues the copies.
    const int g = warp - NC;
    const uint32_t qbytes = (uint32_t)a.G * kD * 2;
    // zero-copy queries: the rows the TMA stages were copied into q with generic stores in
    // this kernel; after the acquire, one proxy fence orders them before every later bulk copy
    await_queries(a, lane);
    if (lane == 0 && a.q_src != a.q) asm volatile("fence.proxy.async.global;" ::: "memory");
    bool ok = true, done = false;
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    // Descriptors of hit task T (lane j: its page j) once the task's unit is managed;
    // `block` waits for that (bounded), else returns false when it is not managed yet.
    auto load_task = [&](int T, bool block, int& slot, int& valid, int& nhit) -> bool {
      if (T >= n_hit_tasks) return true;
      const int tu = T / a.n_chunks, j0 = (T - tu * a.n_chunks) * a.ppt;
      int r = 0;
      if (lane == 0) {
        if (block) {
          r = wait_flag(a.unit_ready + tu, tag, true, a.err) ? 1 : -1;
        } else {
          r = ld_relaxed(a.unit_ready + tu) == tag ? 1 : 0;
        }
      }
      r = __shfl_sync(kAll, r, 0);
      if (r < 0) ok = false;
      if (r <= 0) return false;
      __syncwarp();
      (void)ld_acquire(a.unit_ready + tu);
      nhit = __ldcg(a.n_hit + tu);
      const bool in = lane < a.ppt && j0 + lane < a.ka;
      slot = in ? __ldcg(a.att_slot + (int64_t)tu * a.ka + j0 + lane) : 0;
      valid = in ? __ldcg(a.att_valid + (int64_t)tu * a.ka + j0 + lane) : 0;
      return true;
    };
    int cur_task = 0, cur_ul = 0, cur_n = 0, cur_j = 0, cur_y = 0, cur_valid = 0;
    int nx_task, nx_slot = 0, nx_valid = 0, nx_nhit = 0, c2_raw = 0;
    bool nx_loaded;
    // Tasks are claimed two ahead when there are several per producer; with few tasks a
    // producer holds one claim at a time, so the tasks spread over every producer.
    const bool ahead2 = n_hit_tasks >= 4 * (int)gridDim.x * NG;
    {
      const int t0 = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
      nx_task = __shfl_sync(kAll, t0, 0);
      nx_loaded = load_task(nx_task, false, nx_slot, nx_valid, nx_nhit);
      if (ahead2) c2_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
    }
    bool in_miss = false;
    // retrieved pages: the next entry claimed and loading ahead
    int mq = 0, mq_att = 0, mq_valid = 0, mq_state = 0, m_raw = 0;
    int64_t mq_dst = 0;
    bool m_init = false;
    auto miss_advance = [&]() {
      mq = __shfl_sync(kAll, m_raw, 0);
      int st = 0;
      if (lane == 0) st = miss_entry(a, mq, tag, U, kmax);
      mq_state = __shfl_sync(kAll, st, 0);
      if (mq_state == 1) {
        __syncwarp();
        (void)ld_acquire(a.miss_tag + mq);
        mq_att = __ldcg(a.miss_att + mq);
        mq_dst = __ldcg(a.miss_dst + mq);
        mq_valid = __ldcg(a.miss_valid + mq);
      }
      m_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskMisses], 1) : 0;
    };
    auto leave_hits = [&]() {  // the last producer past its resident pages lets the late retrievers start
      if (lane == 0 && atomicAdd(sm.hits_groups, 1) == NG - 1) *((volatile int*)sm.hits_done) = 1;
    };
    int last_issue[kSt];  // lane 0: last stage index that staged a page in each ring stage
#pragma unroll
    for (int st = 0; st < kSt; ++st) last_issue[st] = -1;
    for (int i = g; ok && !done; i += NG) {
      if (__shfl_sync(kAll, *abort_flag, 0)) {
        ok = false;
        break;
      }
      int y = 0, valid = 0, part = 0, ul = 0;
      bool first = false, last_page = false, have = false;
      while (!have && !done && ok) {
        if (!in_miss) {
          if (cur_j < cur_n) {
            const int j = cur_j++;
            y = __shfl_sync(kAll, cur_y, j);
            valid = __shfl_sync(kAll, cur_valid, j);
            ul = cur_ul;
            part = cur_task;
            first = j == 0;
            last_page = j == cur_n - 1;
            have = true;
          } else {
            if (nx_task < 0) {  // one claim at a time: the next task is claimed only now
              const int tn = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
              nx_task = __shfl_sync(kAll, tn, 0);
              nx_loaded = false;
            }
            const int T = nx_task;
            if (T >= n_hit_tasks) {
              in_miss = true;
              leave_hits();
              continue;
            }
            if (!nx_loaded && !load_task(T, true, nx_slot, nx_valid, nx_nhit)) break;  // ran out of time
            const int tu = T / a.n_chunks, j0 = (T - tu * a.n_chunks) * a.ppt;
            cur_task = T;
            cur_ul = tu;
            cur_n = max(0, min(nx_nhit, j0 + a.ppt) - j0);
            cur_j = 0;
            int slot = nx_slot;
            if (a.tail_n != nullptr && slot == a.cap) {  // the unit's tail page
              cur_y = (int)((a.pool_slots + a.unit_base + tu) * 128);
            } else {
              if (slot < 0 || slot >= a.cap) {  // never expected for a page of the task: stage slot 0 and report
                if (lane < cur_n) atomicOr(a.err, kErrIndex);
                slot = 0;
              }
              cur_y = (int)(((a.unit_base + tu) * a.cap + slot) * 128);
            }
            cur_valid = nx_valid;
            if (ahead2) {
              nx_task = __shfl_sync(kAll, c2_raw, 0);  // claimed a task ago: no wait
              c2_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
              nx_loaded = load_task(nx_task, false, nx_slot, nx_valid, nx_nhit);
            } else {
              nx_task = -1;
              nx_loaded = false;
            }
          }
        } else {
          if (!m_init) {
            m_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskMisses], 1) : 0;
            miss_advance();
            m_init = true;
          }
          if (mq_state == 0) {
            done = true;
            break;
          }
          if (mq_state < 0) {
            ok = false;
            break;
          }
          int okf = 1;
          if (lane == 0) okf = wait_flag(a.ready + mq, tag, true, a.err) ? 1 : 0;
          if (!__shfl_sync(kAll, okf, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");  // TMA reads the generic stores
          int att = mq_att;
          int64_t dp = mq_dst;
          if (att < 0 || att >= U * a.ka || dp < 0 || dp >= a.pool_slots) {  // never expected
            if (lane == 0) atomicOr(a.err, kErrIndex);
            att = 0;
            dp = 0;
          }
          ul = att / a.ka;
          part = U * a.n_chunks + att;
          y = (int)(dp * 128);
          valid = mq_valid;
          first = last_page = true;
          have = true;
          miss_advance();
        }
      }
      if (!ok) break;
      const int st = i % kSt;
      const uint32_t ph = (uint32_t)(i / kSt) & 1u;
      int oke = 1;
      if (lane == 0) oke = mbar_wait(smem_u32(&sm.empty[st]), ph ^ 1u) ? 1 : 0;
      if (!__shfl_sync(kAll, oke, 0)) {
        ok = false;
        break;
      }
      if (!have) {  // the group's sentinel: no task follows
        if (lane == 0) {
          sm.meta[st].part = -1;
          mbar_arrive(smem_u32(&sm.full[st]));
        }
        break;
      }
      if (lane == 0) {
        StageMeta m;
        m.part = part;
        m.ul = ul;
        m.valid = valid;
        m.first = first;
        m.last = last_page;
        sm.meta[st] = m;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, kPageBytes + (first ? qbytes : 0u));
        const uint32_t dst = smem_u32(sm.region + (size_t)st * kStageBytes);
        tma_load_2d(dst, &tmap, fb, 0, y);
        tma_load_2d(dst + 8192, &tmap, fb, 64, y);
        tma_load_2d(dst + 16384, &tmap, fb, 0, y + 64);
        tma_load_2d(dst + 24576, &tmap, fb, 64, y + 64);
        if (first) {
          const int b = ul / a.Hkv, h = ul - b * a.Hkv;
          bulk_load(dst + kPageBytes, a.q + ((int64_t)b * a.Hq + (int64_t)h * a.G) * kD, qbytes, fb);
        }
        last_issue[st] = i;
      }
    }
    if (!in_miss) leave_hits();
    if (lane == 0 && !ok) {
      atomicOr(a.err, kErrTimeout);
      *abort_flag = 1;
      *((volatile int*)sm.hits_done) = 1;  // nobody waits for it in vain
      // drain the copies already issued before leaving (bounded)
#pragma unroll
      for (int st = 0; st < kSt; ++st)
        if (last_issue[st] >= 0) (void)mbar_wait(smem_u32(&sm.full[st]), (uint32_t)(last_issue[st] / kSt) & 1u);
    }
  } else {
    // ------------------------------ consumers ------------------------------
    const int grp = warp / kCWarps;   // consumer group: stage indices grp, grp + NG, ...
    const int w = warp % kCWarps;     // tokens 16w .. 16w+15 of every page
    const int t0 = 16 * w;
    const int mi = lane >> 3, ri = lane & 7;
    const int g4 = lane >> 2, q4 = lane & 3;
    const int tokA = t0 + ri + ((mi & 1) << 3);   // K rows feeding the A operand
    const int tokV = t0 + ri + ((mi >> 1) << 3);  // V rows feeding the transposed A operand
    const uint32_t mrg0 = smem_u32(&sm.mrg[2 * grp]), mrg1 = smem_u32(&sm.mrg[2 * grp + 1]);

    uint32_t qb[NT][8][2];
    float o[8][NT][4];
    float mrow[NT][2], lrow[NT][2];
    uint32_t mph = 0;
    int i = grp;

    for (;;) {
      const int st = i % kSt;
      const uint32_t ph = (uint32_t)(i / kSt) & 1u;
      if (!mbar_wait(smem_u32(&sm.full[st]), ph)) {
        atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      const StageMeta m = sm.meta[st];
      if (m.part < 0) break;  // the group's sentinel
      uint8_t* stage = sm.region + (size_t)st * kStageBytes;
      if (m.first) {
        // query rows of the unit, brought with the task's first page: B operand fragments
        const uint8_t* qs = stage + kPageBytes;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int head = 8 * nt + g4;
          const bool live = head < a.G;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            qb[nt][kk][0] = live ? *reinterpret_cast<const uint32_t*>(qs + head * 256 + (16 * kk + 2 * q4) * 2) : 0u;
            qb[nt][kk][1] = live ? *reinterpret_cast<const uint32_t*>(qs + head * 256 + (16 * kk + 8 + 2 * q4) * 2)
                                 : 0u;
          }
          mrow[nt][0] = mrow[nt][1] = -INFINITY;
          lrow[nt][0] = lrow[nt][1] = 0.f;
#pragma unroll
          for (int md = 0; md < 8; ++md) o[md][nt][0] = o[md][nt][1] = o[md][nt][2] = o[md][nt][3] = 0.f;
        }
      }

      // ---------------- one page: tokens t0..t0+15 ----------------
      const uint32_t kb = smem_u32(stage);
      const uint32_t vb = kb + 16384;
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t af[4];
        ldsm_x4(kb + swz(tokA, 2 * kk + (mi >> 1)), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(s[nt], af, qb[nt][kk][0], qb[nt][kk][1]);
      }
      // online softmax per head (column), over this warp's 16 tokens (rows)
      const bool v0 = (t0 + g4) < m.valid, v1 = (t0 + g4 + 8) < m.valid;
      uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x0 = v0 ? s[nt][e] * kScaleLog2 : -INFINITY;
          const float x1 = v1 ? s[nt][2 + e] * kScaleLog2 : -INFINITY;
          float mx = fmaxf(x0, x1);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(mrow[nt][e], mx);
          const float al = (mn == -INFINITY) ? 1.f : exp2f(mrow[nt][e] - mn);
          p[e] = (mn == -INFINITY) ? 0.f : exp2f(x0 - mn);
          p[2 + e] = (mn == -INFINITY) ? 0.f : exp2f(x1 - mn);
          lrow[nt][e] = fmaf(lrow[nt][e], al, p[e] + p[2 + e]);
          mrow[nt][e] = mn;
#pragma unroll
          for (int md = 0; md < 8; ++md) {
            o[md][nt][e] *= al;
            o[md][nt][2 + e] *= al;
          }
        }
        // P^T fragments (token rows, head columns) -> B operand (head rows, token columns)
        const uint32_t h0 = pack_bf16(p[0], p[1]), h1 = pack_bf16(p[2], p[3]);
        const uint32_t l0 = pack_bf16(p[0] - bf16_lo_f(h0), p[1] - bf16_hi_f(h0));
        const uint32_t l1 = pack_bf16(p[2] - bf16_lo_f(h1), p[3] - bf16_hi_f(h1));
        bh[nt][0] = movmatrix_t(h0);
        bh[nt][1] = movmatrix_t(h1);
        bl[nt][0] = movmatrix_t(l0);
        bl[nt][1] = movmatrix_t(l1);
      }
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        uint32_t af[4];
        ldsm_x4_t(vb + swz(tokV, 2 * md + (mi & 1)), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16(o[md][nt], af, bh[nt][0], bh[nt][1]);
          mma_bf16(o[md][nt], af, bl[nt][0], bl[nt][1]);
        }
      }
      if (m.last) {
        // ---- the task's last page: merge the group's four warps inside this stage ----
        __syncwarp();
        if (lane == 0) mbar_arrive(mrg0);
        if (!mbar_wait(mrg0, mph)) {  // every warp of the group is done reading the page
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        float* gmerge = reinterpret_cast<float*>(stage);
        float* mw = gmerge + w * kMergeFloats;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float l = lrow[nt][e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int hh = 8 * nt + 2 * q4 + e;
#pragma unroll
            for (int md = 0; md < 8; ++md) {
              mw[hh * kMergeRow + 16 * md + g4] = o[md][nt][e];
              mw[hh * kMergeRow + 16 * md + g4 + 8] = o[md][nt][2 + e];
            }
            if (g4 == 0) {
              mw[16 * kMergeRow + hh] = mrow[nt][e];
              mw[16 * kMergeRow + 16 + hh] = l;
            }
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(mrg1);
        if (!mbar_wait(mrg1, mph)) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        mph ^= 1u;
        const int d = w * 32 + lane;  // 0..127
        for (int g = 0; g < a.G; ++g) {
          float M = -INFINITY;
#pragma unroll
          for (int ww = 0; ww < kCWarps; ++ww) M = fmaxf(M, gmerge[ww * kMergeFloats + 16 * kMergeRow + g]);
          float L = 0.f, acc = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int ww = 0; ww < kCWarps; ++ww) {
              const float* src = gmerge + ww * kMergeFloats;
              const float sc = exp2f(src[16 * kMergeRow + g] - M);
              L = fmaf(sc, src[16 * kMergeRow + 16 + g], L);
              acc = fmaf(sc, src[g * kMergeRow + d], acc);
            }
          }
          float* part = a.partials + ((int64_t)m.part * a.G + g) * kPartialStride;
          part[4 + d] = acc;
          if (d == 0) {
            part[0] = M;
            part[1] = L;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));  // the group's four warps free the stage
      i += NG;
    }
  }

  // ---------------- all pages of all CTAs done: combine the partials ----------------
  // Every warp of the CTA (retrievers after their last claim, the producers, the
  // consumers after their last page) meets here before the CTA arrives, so block 0's
  // counter reset below cannot race with a late claim of this step.
  __syncthreads();
  if (tid == 0) {
    if (tl) atomicMax(tl + kTlPages, globaltimer_ns());
    fence_acq_rel();  // the CTA's partials (ordered before by the block barrier), then the arrival
    atomicAdd(&a.counters[kCtrArrive], 1);
    const int target = (int)gridDim.x * tag;  // the counter grows by gridDim.x every step
    // no early exit on another wait's timeout here: block 0 resets the step's counters only
    // once every CTA has stopped claiming work
    if (!wait_flag(&a.counters[kCtrArrive], target, false, nullptr)) atomicOr(a.err, kErrTimeout);
    if (blockIdx.x == 0) {  // the step's counters are no longer read by anyone
      a.counters[kCtrMiss] = 0;
      a.counters[kCtrTaskHits] = 0;
      a.counters[kCtrTaskMisses] = 0;
      a.counters[kCtrRetrieve] = 0;
      a.counters[kCtrManage] = 0;
      a.counters[kCtrManaged] = 0;
      a.counters[kCtrQStaged] = 0;
      a.counters[kCtrStep] += 1;
    }
  }
  __syncthreads();
  if (warp >= NC) return;
  const int pairs = U * a.G;
  if (pairs <= (int)gridDim.x && a.n_chunks + a.k > 16) {
    // few (unit, head) pairs with many partials each: one pair per CTA, all its consumer warps
    // (the ring is free: every CTA is past its pages)
    float* red = reinterpret_cast<float*>(sm.region);
    for (int p = blockIdx.x; p < pairs; p += gridDim.x) combine_head_cta(a, p / a.G, p % a.G, warp, NC, lane, red, 5);
  } else {
    // (unit, head) pairs spread over every consumer warp of the grid
    for (int p = blockIdx.x * NC + warp; p < pairs; p += gridDim.x * NC) combine_head(a, p / a.G, p % a.G, lane);
  }
  if (tl && lane == 0 && atomicAdd(sm.tl_count + 1, 1) == NC - 1) atomicMax(tl + kTlEnd, globaltimer_ns());
}

// ---------------------------------------------------------------------------
// Debug: resolve every partition through the two-level table; live segments per unit.
// ---------------------------------------------------------------------------
__global__ void resolve_all_kernel(LayerArgs a, int32_t* resolve, int32_t* live) {
  __shared__ int s_live;
  const int ul = blockIdx.x;
  const int b = ul / a.Hkv;
  const int P = a.P_b[b];
  const int64_t unit = a.unit_base + ul;
  if (threadIdx.x == 0) s_live = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < a.P_max; p += blockDim.x) {
    int s = -1;
    if (p < P) {
      const int sg = a.dir[unit * a.D + (p >> 6)];
      s = sg < 0 ? -1 : a.seg[(int64_t)sg * kSeg + (p & 63)];
    }
    resolve[(int64_t)ul * a.P_max + p] = s;
  }
  for (int d = threadIdx.x; d < a.D; d += blockDim.x)
    if (a.dir[unit * a.D + d] >= 0) atomicAdd(&s_live, 1);
  __syncthreads();
  if (threadIdx.x == 0) live[ul] = s_live;
}

__global__ void set_int_kernel(int32_t* p, int32_t v) { *p = v; }

__global__ void fill_u32_kernel(uint32_t* p, uint32_t v, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

template <int NT, int GS, bool PIPE = false>
const void* kernel_ptr() {
  return (const void*)decode_step_kernel<NT, GS, PIPE>;
}

// The kernel instance for a layer: NT from the group size G, GS from mgr_gs.
const void* pick_kernel(const LayerArgs& a) {
  if (a.pipe) return a.mgr_gs == 32 ? kernel_ptr<1, 32, true>() : kernel_ptr<1, 128, true>();
  if (a.G <= 8) {
    switch (a.mgr_gs) {
      case 32: return kernel_ptr<1, 32>();
      case 128: return kernel_ptr<1, 128>();
      default: return kernel_ptr<1, 512>();
    }
  }
  switch (a.mgr_gs) {
    case 32: return kernel_ptr<2, 32>();
    case 128: return kernel_ptr<2, 128>();
    default: return kernel_ptr<2, 256>();
  }
}

}  // namespace

int step_threads(int G) { return G <= 8 ? Roles<1>::kThreads : Roles<2>::kThreads; }

int step_full_group(int G) { return G <= 8 ? 512 : 256; }

size_t step_ring_bytes() { return (size_t)kRingBytes; }

// Dynamic shared memory of the decode-step kernel: header + max(ring, manager groups) +
// 1 KiB for aligning the base.
size_t step_smem_bytes(const LayerArgs& a) {
  if (a.pipe)  // header, the ring, the manager groups (128 threads in all), the batch prefix
    return kHeaderBytes + (size_t)kStagesPipe * kStageBytes +
           (size_t)(128 / a.mgr_gs) * sel::mgr_smem_layout(a.mgr_gs, a.P_max, a.cap, a.k, a.D, nullptr, nullptr) +
           4 * ((size_t)a.B + 1) + 16 + 1024;
  const int groups = step_threads(a.G) / a.mgr_gs;
  const size_t mgr = (size_t)groups * sel::mgr_smem_layout(a.mgr_gs, a.P_max, a.cap, a.k, a.D, nullptr, nullptr);
  return kHeaderBytes + (mgr > (size_t)kRingBytes ? mgr : (size_t)kRingBytes) + 1024;
}

size_t mgr_group_bytes(int gs, const LayerArgs& a) {
  return sel::mgr_smem_layout(gs, a.P_max, a.cap, a.k, a.D, nullptr, nullptr);
}

cudaError_t step_configure(const LayerArgs& a) {
  const size_t smem = step_smem_bytes(a);
  return cudaFuncSetAttribute(pick_kernel(a), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_decode_step(const LayerArgs& a, const CUtensorMap* tmap, int grid, cudaStream_t st) {
  int n_hit_tasks = a.B * a.Hkv * a.n_chunks;
  LayerArgs args = a;
  void* params[] = {const_cast<CUtensorMap*>(tmap), &args, &n_hit_tasks};
  return cudaLaunchCooperativeKernel(pick_kernel(a), dim3(grid), dim3(step_threads(a.G)), params,
                                     step_smem_bytes(a), st);
}

cudaError_t launch_set_int(int32_t* p, int32_t v, cudaStream_t st) {
  set_int_kernel<<<1, 1, 0, st>>>(p, v);
  return cudaGetLastError();
}

cudaError_t launch_fill_u32(uint32_t* p, uint32_t v, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  fill_u32_kernel<<<(unsigned)blocks, 256, 0, st>>>(p, v, n);
  return cudaGetLastError();
}

cudaError_t launch_resolve_all(const LayerArgs& a, int32_t* resolve, int32_t* live_segs, cudaStream_t st) {
  resolve_all_kernel<<<a.B * a.Hkv, 256, 0, st>>>(a, resolve, live_segs);
  return cudaGetLastError();
}

}  // namespace spin
