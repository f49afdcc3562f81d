// Retrieve (host -> HBM page copies), paged split-KV decode attention and combine.
//
// Retrieve brings the critical partitions that are not resident from CPU memory
// into their HBM pages; Attention is exact softmax attention over the tokens of
// the selected partitions only (m.x-techcon.com SPIN article, section
// "Spin的核心设计" 1 and Figure 3, 2 and Figure 5 step 4; gist.science/pt section
// 2A). The pages give no kernel design; everything below is this library's.
//
// One cooperative persistent kernel per layer step does both, one CTA per SM:
//   * retriever warps walk the step's miss list (host page -> HBM slot, 16-byte
//     zero-copy loads over the host link), and publish each copied page with a
//     release store of the step tag into its ready flag; two start at once, the
//     others join when the CTA's resident pages have all been issued;
//   * two consumer groups of four warps take alternate stages of a 6-stage
//     shared-memory ring guarded by mbarriers, so two pages are in the math at once;
//   * each group has a producer warp that stages its pages through TMA: first
//     resident pages (hits) in tasks of up to `ppt` pages of one unit, then
//     retrieved pages in miss-list order, each after an acquire of its ready flag.
//     Nothing on the issue path waits for a fresh global load: tasks are claimed
//     two ahead, the next task's page descriptors sit in the lanes' registers, and a
//     retrieved page's miss-list entry is loaded before its flag is awaited.
// So the attention over the hits (HBM bound) hides under the retrieval (host-link
// bound) and each retrieved page is attended as soon as it lands (and from L2).
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
// task's last page and write one partial (m, l, acc[128]) per query head. When
// every CTA has finished its pages (an arrival counter; all CTAs are co-resident
// under the cooperative launch), every consumer warp of the grid combines
// (unit, query head) pairs of partials into the output:
//   out_g = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
//
// Every wait (mbarrier, ready flag, arrival counter) is bounded in time; a wait
// that runs out sets the device error word, stops issuing work and drains the
// copies already issued.
#include "spin_internal.cuh"

namespace spin {

namespace {

constexpr int kStages = 6;    // ring stages (stage i belongs to consumer group i % groups)
constexpr int kCWarps = 4;    // consumer warps of one group: 16 tokens of a page each
constexpr int kMaxGroups = 2;
// Roles per CTA. One 8-head tile (NT = 1, at most 128 registers a thread): two
// consumer groups that take alternate ring stages, so two pages are in the math at
// once, each fed by its own producer warp, and six retriever warps (two saturate the
// host link alone). Two tiles (168 registers): one group, one producer, four
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
constexpr int kMergeRow = kD + 4;                       // padded row of the merge buffer
constexpr int kMergeFloats = 16 * kMergeRow + 32;       // O[16 heads][128+4], m[16], l[16]
static_assert(kCWarps * kMergeFloats * 4 <= kStageBytes, "a task's merge must fit in its last page's stage");
constexpr float kScaleLog2 = 0.12751743074173449f;      // log2(e) / sqrt(128)
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s

struct StageMeta {
  int part, ul, valid, first, last;  // partial slot of the task, unit, valid tokens, first / last page of the task
};

struct AttnSmem {
  uint8_t* ring;      // kStages x kStageBytes, 1024-aligned (a task's last stage also holds its merge)
  uint64_t* full;     // [kStages]
  uint64_t* empty;    // [kStages]
  uint64_t* mrg;      // [groups][2]: written, read
  StageMeta* meta;    // [kStages]
  int* abort_flag;
  int* hits_done;     // set once every producer of this CTA has issued its resident-page tasks
  int* hits_groups;   // producers past their resident pages
};

__host__ __device__ inline size_t attn_smem_layout(AttnSmem* s, uint8_t* base) {
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = (off + align - 1) & ~(align - 1);
    uint8_t* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  };
  uint8_t* ring = take((size_t)kStages * kStageBytes, 1024);
  uint8_t* full = take(sizeof(uint64_t) * kStages, 8);
  uint8_t* empty = take(sizeof(uint64_t) * kStages, 8);
  uint8_t* mrg = take(sizeof(uint64_t) * 2 * kMaxGroups, 8);
  uint8_t* meta = take(sizeof(StageMeta) * kStages, 16);
  uint8_t* ab = take(sizeof(int), 4);
  uint8_t* hd = take(sizeof(int), 4);
  uint8_t* hg = take(sizeof(int), 4);
  if (s) {
    s->ring = ring;
    s->full = (uint64_t*)full;
    s->empty = (uint64_t*)empty;
    s->mrg = (uint64_t*)mrg;
    s->meta = (StageMeta*)meta;
    s->abort_flag = (int*)ab;
    s->hits_done = (int*)hd;
    s->hits_groups = (int*)hg;
  }
  return off;
}

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

__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Wait until *p reaches `want` (== when exact, else >=), bounded by kWaitNs. Polls with
// relaxed loads and a short sleep, then one acquire fence: acquire loads and fences in a
// tight loop hold up the SM's other memory traffic (the retrievers' host loads).
__device__ __noinline__ bool wait_flag(const int* p, int want, bool exact) {
  auto hit = [&](int v) { return exact ? v == want : v >= want; };
  bool ok = hit(ld_relaxed(p));
  if (!ok) {
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30) && !ok; ++it) {
      __nanosleep(128);
      ok = hit(ld_relaxed(p));
      if (!ok && (it & 63u) == 0 && globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  if (ok) fence_acq_rel();
  return ok;
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
// columns per lane. The lanes fetch the (m, l) of up to 32 partials at once; the
// accumulator rows are loaded eight at a time before they are used, so a head costs
// a few round trips to L2 whatever the number of partials.
// ---------------------------------------------------------------------------
__device__ void combine_head(const LayerArgs& a, int ul, int g, int lane) {
  const int b = ul / a.Hkv, h = ul - b * a.Hkv;
  const int has_tail = (a.tail_n != nullptr && a.tail_n[b] > 0) ? 1 : 0;
  const int keff = a.keff[ul] + has_tail, nh = a.n_hit[ul];  // attended pages; resident ones (tail included)
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
  float M = -INFINITY;
  for (int i0 = 0; i0 < n; i0 += 32)
    if (i0 + lane < n) M = fmaxf(M, __ldcg(part_ptr(i0 + lane)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
    for (int i0 = 0; i0 < n; i0 += 32) {
      float sc_l = 0.f, l_l = 0.f;
      if (i0 + lane < n) {
        const float* pp = part_ptr(i0 + lane);
        sc_l = exp2f(__ldcg(pp) - M);
        l_l = __ldcg(pp + 1);
      }
      float ls = sc_l * l_l;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      L += ls;
      const int cnt = min(32, n - i0);
      for (int i1 = 0; i1 < cnt; i1 += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = (i1 + u < cnt) ? __ldcg(reinterpret_cast<const float4*>(part_ptr(i0 + i1 + u) + 4) + lane)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float sc = __shfl_sync(0xffffffffu, sc_l, (i1 + u) & 31);  // 0 past cnt: its v is 0 too
          acc.x = fmaf(sc, v[u].x, acc.x);
          acc.y = fmaf(sc, v[u].y, acc.y);
          acc.z = fmaf(sc, v[u].z, acc.z);
          acc.w = fmaf(sc, v[u].w, acc.w);
        }
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  out[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// ---------------------------------------------------------------------------
// Retrieve + attention kernel. NT = number of 8-head tiles (G <= 8 * NT).
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(Roles<NT>::kThreads, 1)
attend_retrieve_kernel(const __grid_constant__ CUtensorMap tmap, LayerArgs a, int n_hit_tasks) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  AttnSmem sm;
  attn_smem_layout(&sm, base);
  constexpr int NG = Roles<NT>::kGroups, NC = Roles<NT>::kConsumers;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_miss = a.counters[kCtrMiss];
  const int tag = a.counters[kCtrStep] + 1;  // ready-flag value of this step (flags are never reset)

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kCWarps);  // the four warps of the stage's group
    }
    for (int m = 0; m < 2 * NG; ++m) mbar_init(smem_u32(&sm.mrg[m]), kCWarps);
    *sm.abort_flag = 0;
    *sm.hits_done = 0;
    *sm.hits_groups = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort_flag = sm.abort_flag;

  if (warp >= NC + NG) {
    // ------------------------------ retrievers ------------------------------
    // retr_warps warps copy from the start; retr_late more join once this CTA's
    // resident pages are issued (so they do not slow the HBM-bound hits); the rest idle.
    const int rw = warp - NC - NG;
    bool active = rw < a.retr_warps && !a.retrieve_in_select;
    if (!active && rw < a.retr_warps + a.retr_late && !a.retrieve_in_select) {
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
    for (; active;) {
      int m = 0;
      if (lane == 0) m = atomicAdd(&a.counters[kCtrRetrieve], 1);
      m = __shfl_sync(0xffffffffu, m, 0);
      if (m >= n_miss) break;
      const int64_t sp = a.miss_src[m], dp = a.miss_dst[m];
      const bool in_range = sp >= 0 && sp < a.host_pages && dp >= 0 && dp < a.pool_slots;
      if (!in_range && lane == 0) atomicOr(a.err, kErrIndex);  // never expected: skip the copy
      const uint4* src = reinterpret_cast<const uint4*>(a.host_store + sp * kPageElems);
      uint4* dst = reinterpret_cast<uint4*>(a.pool + dp * kPageElems);
#pragma unroll 1
      for (int c = 0; in_range && c < kVec; c += 32 * kUnroll) {
        uint4 r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) r[u] = __ldcs(src + c + u * 32 + lane);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) dst[c + u * 32 + lane] = r[u];
      }
      fence_acq_rel();  // each lane's stores of the page before the flag (acq_rel: no full sc fence)
      __syncwarp();
      if (lane == 0) st_release(a.ready + m, tag);
    }
  } else if (warp >= NC) {
    // ------------------------------ producers ------------------------------
    // Producer warp g feeds consumer group g: stage indices i = g, g + NG, ... use ring
    // stage i % kStages. Its stream: resident-page tasks (up to ppt pages of one unit,
    // claimed from a shared counter), then retrieved pages (one page each, in miss-list
    // order, once its ready flag is published), then a sentinel.
    // The whole warp runs the loop so that nothing the issue path needs is a fresh
    // global load: tasks are claimed two ahead, the next task's page descriptors load
    // into the lanes' registers (lane j: page j) while the current task issues, and the
    // next retrieved page's miss-list entry loads before its flag is awaited. Lane 0
    // alone waits on the ring barriers and issues the copies.
    constexpr uint32_t kAll = 0xffffffffu;
    const int g = warp - NC;
    const uint32_t qbytes = (uint32_t)a.G * kD * 2;
    const int U = a.B * a.Hkv;
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    auto load_task = [&](int T, int& slot, int& valid, int& nhit) {
      if (T < n_hit_tasks) {
        const int tu = T / a.n_chunks, j0 = (T - tu * a.n_chunks) * a.ppt;
        nhit = a.n_hit[tu];
        const bool in = lane < a.ppt && j0 + lane < a.ka;
        slot = in ? a.att_slot[tu * a.ka + j0 + lane] : 0;
        valid = in ? a.att_valid[tu * a.ka + j0 + lane] : 0;
      }
    };
    int cur_task = 0, cur_ul = 0, cur_n = 0, cur_j = 0, cur_y = 0, cur_valid = 0;
    int nx_task, nx_slot = 0, nx_valid = 0, nx_nhit = 0, c2_raw;
    {
      const int t0 = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
      nx_task = __shfl_sync(kAll, t0, 0);
      load_task(nx_task, nx_slot, nx_valid, nx_nhit);
      c2_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
    }
    bool in_miss = false;
    // retrieved pages: the next entry claimed and loading ahead
    int mq = 0, mq_att = 0, mq_valid = 0, m_raw = 0;
    int64_t mq_dst = 0;
    bool m_init = false;
    auto miss_advance = [&]() {
      mq = __shfl_sync(kAll, m_raw, 0);
      if (mq < n_miss) {
        mq_att = a.miss_att[mq];
        mq_dst = a.miss_dst[mq];
        mq_valid = a.miss_valid[mq];
      }
      m_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskMisses], 1) : 0;
    };
    auto leave_hits = [&]() {  // the last producer past its resident pages lets the late retrievers start
      if (lane == 0 && atomicAdd(sm.hits_groups, 1) == NG - 1) *((volatile int*)sm.hits_done) = 1;
    };
    int last_issue[kStages];  // lane 0: last stage index that staged a page in each ring stage
#pragma unroll
    for (int st = 0; st < kStages; ++st) last_issue[st] = -1;
    bool ok = true, done = false;
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
            const int T = nx_task;
            if (T >= n_hit_tasks) {
              in_miss = true;
              leave_hits();
              continue;
            }
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
            nx_task = __shfl_sync(kAll, c2_raw, 0);  // claimed a task ago: no wait
            load_task(nx_task, nx_slot, nx_valid, nx_nhit);
            c2_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskHits], 1) : 0;
          }
        } else {
          if (!m_init) {
            m_raw = lane == 0 ? atomicAdd(&a.counters[kCtrTaskMisses], 1) : 0;
            miss_advance();
            m_init = true;
          }
          if (mq >= n_miss) {
            done = true;
            break;
          }
          int okf = 1;
          if (lane == 0) okf = wait_flag(a.ready + mq, tag, true) ? 1 : 0;
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
      const int st = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
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
        const uint32_t dst = smem_u32(sm.ring + (size_t)st * kStageBytes);
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
      for (int st = 0; st < kStages; ++st)
        if (last_issue[st] >= 0) (void)mbar_wait(smem_u32(&sm.full[st]), (uint32_t)(last_issue[st] / kStages) & 1u);
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
      const int st = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      if (!mbar_wait(smem_u32(&sm.full[st]), ph)) {
        atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      const StageMeta m = sm.meta[st];
      if (m.part < 0) break;  // the group's sentinel
      uint8_t* stage = sm.ring + (size_t)st * kStageBytes;
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
  // Every warp of the CTA (retrievers after their last claim, the producer, the
  // consumers after their last page) meets here before the CTA arrives, so block 0's
  // counter reset below cannot race with a late claim of this step.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(&a.counters[kCtrArrive], 1);
    const int target = (int)gridDim.x * tag;  // the counter grows by gridDim.x every step
    if (!wait_flag(&a.counters[kCtrArrive], target, false)) atomicOr(a.err, kErrTimeout);
    if (blockIdx.x == 0) {  // the step's counters are no longer read by anyone
      a.counters[kCtrMiss] = 0;
      a.counters[kCtrTaskHits] = 0;
      a.counters[kCtrTaskMisses] = 0;
      a.counters[kCtrRetrieve] = 0;
      a.counters[kCtrStep] += 1;
    }
  }
  __syncthreads();
  if (warp >= NC) return;
  // (unit, head) pairs spread over every consumer warp of the grid
  const int pairs = a.B * a.Hkv * a.G;
  for (int p = blockIdx.x * NC + warp; p < pairs; p += gridDim.x * NC) combine_head(a, p / a.G, p % a.G, lane);
}

}  // namespace

size_t attention_smem_bytes() { return attn_smem_layout(nullptr, nullptr) + 1024; }

cudaError_t attention_configure() {
  const int kMaxShared = 100;  // cudaSharedmemCarveoutMaxShared
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attend_retrieve_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attention_smem_bytes())) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attend_retrieve_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attention_smem_bytes())) != cudaSuccess)
    return e;
  (void)kMaxShared;
  return cudaSuccess;
}

cudaError_t launch_attend_retrieve(const LayerArgs& a, const CUtensorMap* tmap, int grid, cudaStream_t st) {
  int n_hit_tasks = a.B * a.Hkv * a.n_chunks;
  LayerArgs args = a;
  void* params[] = {const_cast<CUtensorMap*>(tmap), &args, &n_hit_tasks};
  if (a.G <= 8)
    return cudaLaunchCooperativeKernel((const void*)attend_retrieve_kernel<1>, dim3(grid),
                                       dim3(Roles<1>::kThreads), params, attention_smem_bytes(), st);
  return cudaLaunchCooperativeKernel((const void*)attend_retrieve_kernel<2>, dim3(grid), dim3(Roles<2>::kThreads),
                                     params, attention_smem_bytes(), st);
}


}  // namespace spin
