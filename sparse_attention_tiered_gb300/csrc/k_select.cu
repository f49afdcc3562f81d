// Select (score + per-KV-head top-k) and the page manager of one decode step.
//
// Page citations (SPIN, arXiv 2604.26837):
//   [XT] m.x-techcon.com, "吞吐量提升5.66倍！微软、港中大等Spin框架如何统一稀疏注意力与分级内存…",
//        section "Spin的核心设计": 1 (分区抽象, Figure 3: Select picks the critical
//        partitions), 2 (局部性感知的KV管理: mandatory/buffer pages, bucketed LRU,
//        Figure 5 steps 1-4), 3 (分级元数据组织, Figure 6: two-level table);
//   [GS] gist.science/pt, same title, section 2A-2C.
// Rules the pages leave open and this library fixes: the score of a partition is
// the sum over the GQA group's query heads of q . summary (fp32); the k highest
// scores are taken with equal scores going to the lower partition index; the
// resident capacity of a unit is buf_mult * k pages, mandatory pages included;
// the bucket of a page is 63 - min(63, t - last_use) (0 = oldest); whole buckets
// are reclaimed from bucket 0 upward until the count covers the demand; misses in
// ascending partition order take free slots in ascending slot order; a segment
// covers 64 consecutive partitions.
#include "spin_internal.cuh"

namespace spin {

namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Order-preserving map fp32 -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---------------------------------------------------------------------------
// Scores: sc[u][p] = sum_g q_g . s_p = (sum_g q_g) . s_p, fp32.
// Grid (ceil(Pmax / 64), units of the layer); 8 warps, 8 partitions per warp,
// one 16-byte summary slice per lane (the 512-byte summary is one coalesced row).
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kScorePerWarp = 8;
constexpr int kScoreChunk = (kScoreThreads / 32) * kScorePerWarp;  // 64

__global__ void __launch_bounds__(kScoreThreads) score_kernel(LayerArgs a) {
  const int ul = blockIdx.y;
  const int b = ul / a.Hkv, h = ul % a.Hkv;
  const int P = a.P_b[b];
  const int p_base = blockIdx.x * kScoreChunk;
  if (p_base >= P) return;
  __shared__ __align__(16) float qs[kD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the summary loads do not depend on the query: issue them first
  const float4* su = reinterpret_cast<const float4*>(a.summ + host_page_index(a, b, h, 0) * kD);
  const int p0 = p_base + warp * kScorePerWarp;
  float4 sv[kScorePerWarp];
#pragma unroll
  for (int i = 0; i < kScorePerWarp; ++i) {
    const int p = p0 + i;
    sv[i] = p < P ? __ldg(su + (int64_t)p * (kD / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (threadIdx.x < kD) {
    const uint16_t* q = a.q + ((int64_t)b * a.Hq + (int64_t)h * a.G) * kD + threadIdx.x;
    float s = 0.f;
    for (int g = 0; g < a.G; ++g) s += bf16_bits_to_float(q[g * kD]);
    qs[threadIdx.x] = s;
  }
  __syncthreads();
  const float4 qv = reinterpret_cast<const float4*>(qs)[lane];
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
    if (p < P) a.scores[(int64_t)ul * a.P_max + p] = (x == 0.f) ? 0.f : x;  // -0 -> +0
  }
}

// ---------------------------------------------------------------------------
// Select + manage: one CTA per unit of the layer.
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
// Units with more partitions than this take the wide-unit paths of the top-k (512
// threads only): the radix passes after the first run on the keys of the threshold
// bin, and the compaction ranks a short list of the keys >= the threshold.
constexpr int kWideP = 4096;
constexpr int kCandMax = 8192;   // keys of the first pass's threshold bin kept for the later passes
__host__ __device__ inline int cand_capacity(int P_max) { return P_max > kWideP ? (P_max < kCandMax ? P_max : kCandMax) : 0; }
constexpr int kListMax = 1024;   // keys >= the threshold ranked in the list compaction

struct SelSmem {
  uint32_t* keys;     // [P_max]
  int32_t* sp;        // [cap] slot -> partition
  int32_t* lu;        // [cap] slot -> last use
  int32_t* flist;     // [cap] free slots ascending
  int32_t* sel;       // [k]
  int32_t* sslot;     // [k]
  int32_t* hit;       // [k]
  int32_t* mrank;     // [k] misses before j (exclusive)
  int32_t* dirs;      // [D]
  uint32_t* whist;    // [kSelWarps][256]
  uint8_t* mand;      // [cap]
  int64_t* msrc;      // [k] host page of the unit's r-th miss (copy in this kernel)
  int64_t* mdst;      // [k] pool page of the unit's r-th miss
  int32_t* midx;      // [k] miss-list entry of the unit's r-th miss, -1 = none
  uint32_t* cand;     // [cand_capacity(P_max)] (wide units) keys of the first radix pass's threshold bin
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline size_t sel_smem_layout(int P_max, int cap, int k, int D, SelSmem* s, uint8_t* base) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += align16(bytes);
    return p;
  };
  uint8_t* keys = take(sizeof(uint32_t) * (size_t)(P_max > 0 ? P_max : 1));
  uint8_t* sp = take(sizeof(int32_t) * cap);
  uint8_t* lu = take(sizeof(int32_t) * cap);
  uint8_t* fl = take(sizeof(int32_t) * cap);
  uint8_t* sel = take(sizeof(int32_t) * k);
  uint8_t* ss = take(sizeof(int32_t) * k);
  uint8_t* hit = take(sizeof(int32_t) * k);
  uint8_t* mrank = take(sizeof(int32_t) * k);
  uint8_t* dirs = take(sizeof(int32_t) * (D > 0 ? D : 1));
  uint8_t* wh = take(sizeof(uint32_t) * kSelWarps * 256);
  uint8_t* mand = take((size_t)cap);
  uint8_t* msrc = take(sizeof(int64_t) * k);
  uint8_t* mdst = take(sizeof(int64_t) * k);
  uint8_t* midx = take(sizeof(int32_t) * k);
  uint8_t* cand = take(sizeof(uint32_t) * (size_t)cand_capacity(P_max));
  if (s) {
    s->keys = (uint32_t*)keys;
    s->sp = (int32_t*)sp;
    s->lu = (int32_t*)lu;
    s->flist = (int32_t*)fl;
    s->sel = (int32_t*)sel;
    s->sslot = (int32_t*)ss;
    s->hit = (int32_t*)hit;
    s->mrank = (int32_t*)mrank;
    s->dirs = (int32_t*)dirs;
    s->whist = (uint32_t*)wh;
    s->mand = mand;
    s->msrc = (int64_t*)msrc;
    s->mdst = (int64_t*)mdst;
    s->midx = (int32_t*)midx;
    s->cand = (uint32_t*)cand;
  }
  return off;
}

// Claim a free segment of the shared pool (bitmap, lock free). -1 when exhausted.
__device__ int alloc_segment(const LayerArgs& a, uint32_t hint) {
  const int nwords = (a.S + 31) >> 5;
  for (int i = 0; i < nwords; ++i) {
    const int w = (int)((hint + (uint32_t)i) % (uint32_t)nwords);
    uint32_t bits = *((volatile uint32_t*)&a.seg_bitmap[w]);
    for (int tries = 0; tries < 33 && bits != 0xffffffffu; ++tries) {
      const int bit = __ffs(~bits) - 1;
      const uint32_t old = atomicOr(&a.seg_bitmap[w], 1u << bit);
      if (!(old & (1u << bit))) {
        __threadfence();
        return w * 32 + bit;
      }
      bits = old | (1u << bit);
    }
  }
  return -1;
}

__device__ __forceinline__ void release_segment(const LayerArgs& a, int sg) {
  __threadfence();
  atomicAnd(&a.seg_bitmap[sg >> 5], ~(1u << (sg & 31)));
}

// Barrier over the first NT threads of the CTA (one warp: __syncwarp; otherwise a
// named barrier, so the warps that left after scoring are not waited for).
template <int NT>
__device__ __forceinline__ void group_sync() {
  if constexpr (NT == 32) {
    __syncwarp();
  } else {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  }
}

// Exclusive scan of one int per thread over the first NT threads; *total = sum.
template <int NT>
__device__ int group_exclusive_scan(int v, int* total, int* wsum) {
  constexpr int kW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if constexpr (kW == 1) {
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
  } else {
    if (lane == 31) wsum[warp] = x;
    group_sync<NT>();
    if (warp == 0) {
      int w = lane < kW ? wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < kW) wsum[lane] = w;  // inclusive
    }
    group_sync<NT>();
    const int before = (warp > 0 ? wsum[warp - 1] : 0) + x - v;
    *total = wsum[kW - 1];
    group_sync<NT>();
    return before;
  }
}

// One CTA (512 threads) per unit.
// kFusedScore: the CTA computes its unit's scores itself (same arithmetic as
// score_kernel: per partition, lane l holds dims 4l..4l+3, one mul and three fma,
// then a butterfly sum) instead of reading them from the score kernel's output.
// Used when there are enough units per layer to keep HBM busy with one CTA each.
// NT: threads that run top-k and the page manager after the keys are in shared
// memory (32 = one warp with warp-level primitives only, for small units; 512 =
// the whole CTA, for large ones).
template <int NT, bool kFusedScore>
__global__ void __launch_bounds__(kSelThreads) select_manage_kernel(LayerArgs a) {
  constexpr int kW = NT / 32;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int s_bin, s_above, s_cnt_hits, s_cnt_res, s_cutoff, s_evicted;
  __shared__ int s_wgt[kSelWarps], s_weq[kSelWarps], s_wpos[kSelWarps], s_wtake[kSelWarps];
  __shared__ int s_scan[kSelWarps];
  __shared__ int s_ncand, s_nlist, s_ntaken;
  SelSmem sm;
  sel_smem_layout(a.P_max, a.cap, a.k, a.D, &sm, smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ul = blockIdx.x;
  const int b = ul / a.Hkv, h = ul % a.Hkv;
  const int P = a.P_b[b];
  const int k = a.k, cap = a.cap;
  const int keff = P < k ? P : k;
  const int64_t unit = a.unit_base + ul;
  const int t = a.counters[kCtrStep];
  // After a pool or invariant error the page state is no longer trusted: leave it as is.
  if (*((volatile uint32_t*)a.err) & (kErrCapacity | kErrInternal | kErrSelCount | kErrSegId | kErrIndex)) return;

  // ---------------- scores -> order-preserving keys ----------------
  if constexpr (kFusedScore) {
    __shared__ __align__(16) float s_qs[kD];
    constexpr int kPer = 8;  // partitions in flight per warp
    const float4* su = reinterpret_cast<const float4*>(a.summ + host_page_index(a, b, h, 0) * kD);
    float4 sv[kPer];
    int p0 = warp * kPer;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      sv[i] = (p0 + i < P) ? __ldg(su + (int64_t)(p0 + i) * (kD / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < kD) {
      const uint16_t* q = a.q + ((int64_t)b * a.Hq + (int64_t)h * a.G) * kD + tid;
      float s = 0.f;
      for (int g = 0; g < a.G; ++g) s += bf16_bits_to_float(q[g * kD]);
      s_qs[tid] = s;
    }
    __syncthreads();
    const float4 qv = reinterpret_cast<const float4*>(s_qs)[lane];
    for (; p0 < P; p0 += kSelWarps * kPer) {
      float d[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        float x = sv[i].x * qv.x;
        x = fmaf(sv[i].y, qv.y, x);
        x = fmaf(sv[i].z, qv.z, x);
        x = fmaf(sv[i].w, qv.w, x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        d[i] = x;
      }
      const int pn = p0 + kSelWarps * kPer;  // prefetch the warp's next partitions
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        sv[i] = (pn + i < P) ? __ldg(su + (int64_t)(pn + i) * (kD / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < kPer) {
        float x = d[0];
#pragma unroll
        for (int i = 1; i < kPer; ++i) x = (lane == i) ? d[i] : x;
        const int p = p0 + lane;
        if (p < P) {
          x = (x == 0.f) ? 0.f : x;  // -0 -> +0
          a.scores[(int64_t)ul * a.P_max + p] = x;
          sm.keys[p] = float_key(x);
        }
      }
    }
    __syncthreads();
  } else {
    // eight independent loads per thread before the stores: one round trip per 4096 keys
    const float* sc = a.scores + (int64_t)ul * a.P_max;
    for (int p0 = tid; p0 < P; p0 += 8 * kSelThreads) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (p0 + u * kSelThreads < P) ? sc[p0 + u * kSelThreads] : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p0 + u * kSelThreads < P) sm.keys[p0 + u * kSelThreads] = float_key(v[u]);
    }
  }

  __syncthreads();  // keys complete for every thread
  if (tid >= NT) return;

  // ---------------- top-k: radix select on order-preserving keys ----------------
  uint32_t prefix = 0, mask = 0;
  int krem = keff;
  const bool wide = NT == kSelThreads && P > kWideP;
  int ncand = -1;  // >= 0: the later passes scan sm.cand[0, ncand) instead of every key
  if (keff > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < kW * 256; i += NT) sm.whist[i] = 0;
      group_sync<NT>();
      const uint32_t* src = ncand >= 0 ? sm.cand : sm.keys;
      const int nsrc = ncand >= 0 ? ncand : P;
      for (int p = tid; p < nsrc; p += NT) {
        const uint32_t key = src[p];
        if ((key & mask) == prefix) atomicAdd(&sm.whist[warp * 256 + ((key >> shift) & 255u)], 1u);
      }
      group_sync<NT>();
      if constexpr (kW > 1) {
        for (int i = tid; i < 256; i += NT) {
          uint32_t s = 0;
          for (int w = 0; w < kW; ++w) s += sm.whist[w * 256 + i];
          sm.whist[i] = s;  // row 0 now holds the merged histogram (each thread owns its column)
        }
      }
      group_sync<NT>();
      if (warp == 0) {
        // lane l owns bins 255-8l down to 248-8l (the top bins first)
        int c[8], lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = (int)sm.whist[255 - 8 * lane - i];
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
      group_sync<NT>();
      prefix |= (uint32_t)s_bin << shift;
      mask |= 0xFFu << shift;
      krem -= s_above;
      if (pass == 0 && wide && (int)sm.whist[s_bin] <= cand_capacity(a.P_max)) {
        // keep the keys of the threshold bin (row 0 of the histogram holds its merged count)
        group_sync<NT>();
        if (tid == 0) s_ncand = 0;
        group_sync<NT>();
        for (int p = tid; p < P; p += NT) {
          const uint32_t key = sm.keys[p];
          if ((key & mask) == prefix) sm.cand[atomicAdd(&s_ncand, 1)] = key;
        }
        group_sync<NT>();
        ncand = s_ncand;
      }
      group_sync<NT>();
    }
  }
  const uint32_t T = prefix;  // the k-th largest key; krem = equal keys still to take

  // ---------------- compaction in ascending partition order ----------------
  // Wide units: the keys >= T go to a short unordered list (partition, key) in the
  // histogram scratch; each list entry is taken when its key is > T or it is one of the
  // krem equal keys with the lowest partitions, and lands at the rank of its partition
  // among the taken entries. A list that would overflow falls back to the warp scans.
  bool compacted = false;
  if (wide && keff > 0) {
    int32_t* lp = reinterpret_cast<int32_t*>(sm.whist);                // [kListMax] partition
    uint32_t* lk = sm.whist + kListMax;                                  // [kListMax] key
    int32_t* tk = reinterpret_cast<int32_t*>(sm.whist) + 2 * kListMax;  // [kListMax] taken flag
    static_assert(3 * kListMax <= kSelWarps * 256, "the list must fit in the histogram scratch");
    if (tid == 0) {
      s_nlist = 0;
      s_ntaken = 0;
    }
    group_sync<NT>();
    for (int p = tid; p < P; p += NT) {
      const uint32_t key = sm.keys[p];
      if (key >= T) {
        const int i = atomicAdd(&s_nlist, 1);
        if (i < kListMax) {
          lp[i] = p;
          lk[i] = key;
        }
      }
    }
    group_sync<NT>();
    const int n = s_nlist;
    if (n <= kListMax) {
      for (int i = tid; i < n; i += NT) {
        int taken = lk[i] > T;
        if (!taken) {  // equal key: taken when fewer than krem equal keys sit at lower partitions
          int eqb = 0;
          for (int j = 0; j < n; ++j) eqb += (lk[j] == T && lp[j] < lp[i]);
          taken = eqb < krem;
        }
        tk[i] = taken;
        if (taken) atomicAdd(&s_ntaken, 1);
      }
      group_sync<NT>();
      if (s_ntaken != keff) {  // never expected: leave the unit untouched and report
        if (tid == 0) atomicOr(a.err, kErrSelCount);
        return;
      }
      for (int i = tid; i < n; i += NT) {
        if (!tk[i]) continue;
        int pos = 0;
        for (int j = 0; j < n; ++j) pos += (tk[j] && lp[j] < lp[i]);
        if (pos < keff) sm.sel[pos] = lp[i];
      }
      compacted = true;
    }
    group_sync<NT>();
  }
  if (!compacted) {
    const int chunk = ((P + NT - 1) / NT) * 32;
    const int wb = warp * chunk, we = min(P, wb + chunk);
    int gt = 0, eq = 0;
    if (keff > 0)
      for (int base = wb; base < we; base += 32) {
        const int p = base + lane;
        const uint32_t key = p < we ? sm.keys[p] : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, p < we && key > T));
        eq += __popc(__ballot_sync(0xffffffffu, p < we && key == T));
      }
    if (lane == 0) {
      s_wgt[warp] = gt;
      s_weq[warp] = eq;
    }
    group_sync<NT>();
    if (tid == 0) {
      int eq_before = 0, pos = 0;
      for (int w = 0; w < kW; ++w) {
        const int take = max(0, min(krem - eq_before, s_weq[w]));
        s_wpos[w] = pos;
        s_wtake[w] = take;
        pos += s_wgt[w] + take;
        eq_before += s_weq[w];
      }
      s_bin = pos;  // total selected (reuses the radix scratch)
    }
    group_sync<NT>();
    if (s_bin != keff) {  // never expected: leave the unit untouched and report
      if (tid == 0) atomicOr(a.err, kErrSelCount);
      return;
    }
    int pos = s_wpos[warp], eq_left = s_wtake[warp];
    if (keff > 0)
      for (int base = wb; base < we; base += 32) {
        const int p = base + lane;
        const uint32_t key = p < we ? sm.keys[p] : 0u;
        const bool isgt = p < we && key > T;
        const bool iseq = p < we && key == T;
        const uint32_t meq = __ballot_sync(0xffffffffu, iseq);
        const bool take = isgt || (iseq && __popc(meq & lanemask_lt()) < eq_left);
        const uint32_t msel = __ballot_sync(0xffffffffu, take);
        if (take && pos + __popc(msel & lanemask_lt()) < keff) sm.sel[pos + __popc(msel & lanemask_lt())] = p;
        pos += __popc(msel);
        eq_left -= min(eq_left, __popc(meq));
      }
  }

  // ---------------- load the unit's page state ----------------
  int32_t* g_sp = a.slot_part + unit * cap;
  int32_t* g_lu = a.last_use + unit * cap;
  for (int s = tid; s < cap; s += NT) {
    sm.sp[s] = g_sp[s];
    sm.lu[s] = g_lu[s];
    sm.mand[s] = 0;
  }
  for (int d = tid; d < a.D; d += NT) sm.dirs[d] = a.dir[unit * a.D + d];
  for (int j = tid; j < k; j += NT) sm.midx[j] = -1;
  if (tid == 0) {
    s_cnt_hits = 0;
    s_cnt_res = 0;
    s_cutoff = -1;
    s_evicted = 0;
  }
  group_sync<NT>();

  // ---------------- 1. residency check through the two-level table; 2. bump ----------------
  for (int j = tid; j < keff; j += NT) {
    const int p = sm.sel[j];
    int sg = sm.dirs[p >> 6];
    if (sg >= a.S) {
      atomicOr(a.err, kErrSegId);
      sg = -1;
    }
    const int slot = sg < 0 ? -1 : a.seg[(int64_t)sg * kSeg + (p & 63)];
    if (slot >= cap) atomicOr(a.err, kErrIndex);
    sm.sslot[j] = slot;
    sm.hit[j] = slot >= 0;
    if (slot >= 0 && slot < cap) {
      sm.lu[slot] = t;
      sm.mand[slot] = 1;
      atomicAdd(&s_cnt_hits, 1);
    } else if (slot >= cap) {
      sm.sslot[j] = -1;
      sm.hit[j] = 0;
    }
  }
  {
    int res = 0;
    for (int s = tid; s < cap; s += NT) res += sm.sp[s] >= 0;
    res = __reduce_add_sync(0xffffffffu, res);
    if (lane == 0 && res) atomicAdd(&s_cnt_res, res);
  }
  group_sync<NT>();
  const int hits = s_cnt_hits;
  const int misses = keff - hits;
  // tail mode: the request's tail page is attended after the hits, before the misses
  const int has_tail = (a.tail_n != nullptr && a.tail_n[b] > 0) ? 1 : 0;
  const int resident = s_cnt_res;
  // free pages are counted against the request's budget (buffer elasticity): after a
  // shrink the demand includes the excess and the LRU reclaims down to the budget
  const int demand = misses - (a.budget_b[b] - resident);

  // ---------------- 3. bucketed LRU ----------------
  if (demand > 0) {
    uint32_t* hist = sm.whist;  // 64 bins
    for (int i = tid; i < kBuckets; i += NT) hist[i] = 0;
    group_sync<NT>();
    for (int s = tid; s < cap; s += NT) {
      if (sm.sp[s] < 0 || sm.mand[s]) continue;
      const int age = t - sm.lu[s];
      const int bucket = kBuckets - 1 - min(kBuckets - 1, age);
      atomicAdd(&hist[bucket], 1u);
    }
    group_sync<NT>();
    if (warp == 0) {
      // lane l owns buckets 2l, 2l+1 (oldest first)
      const int c0 = (int)hist[2 * lane], c1 = (int)hist[2 * lane + 1];
      const int lsum = c0 + c1;
      int incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - lsum;
      const uint32_t m = __ballot_sync(0xffffffffu, excl < demand && incl >= demand);
      if (lane == __ffs(m) - 1) s_cutoff = (excl + c0 >= demand) ? 2 * lane : 2 * lane + 1;
    }
    group_sync<NT>();
    const int cutoff = s_cutoff;
    for (int s = tid; s < cap; s += NT) {
      const int p = sm.sp[s];
      if (p < 0 || sm.mand[s]) continue;
      const int age = t - sm.lu[s];
      const int bucket = kBuckets - 1 - min(kBuckets - 1, age);
      if (bucket > cutoff) continue;
      // clear the table entry; the last page of a segment returns it to the pool
      const int sg = sm.dirs[p >> 6];
      if (sg >= a.S) {
        atomicOr(a.err, kErrSegId);
      } else if (sg >= 0) {
        a.seg[(int64_t)sg * kSeg + (p & 63)] = -1;
        __threadfence();
        if (atomicSub(&a.seg_live[sg], 1) == 1) {
          sm.dirs[p >> 6] = -1;
          release_segment(a, sg);
        }
      } else {
        atomicOr(a.err, kErrInternal);  // a resident page without a table entry
      }
      sm.sp[s] = -1;
      atomicAdd(&s_evicted, 1);
    }
    group_sync<NT>();
  }

  // ---------------- 4. assign free slots to misses, allocate segments ----------------
  // free slots in ascending order
  __shared__ int s_nfree;
  {
    int base = 0;
    for (int r = 0; r < cap; r += NT) {
      const int s = r + tid;
      const int f = (s < cap && sm.sp[s] < 0) ? 1 : 0;
      int tot;
      const int ex = group_exclusive_scan<NT>(f, &tot, s_scan);
      if (f) sm.flist[base + ex] = s;
      base += tot;
    }
    if (tid == 0) s_nfree = base;
  }
  // rank of each miss among the misses (ascending partition = ascending j)
  {
    int base = 0;
    for (int r = 0; r < keff; r += NT) {
      const int j = r + tid;
      const int m = (j < keff && !sm.hit[j]) ? 1 : 0;
      int tot;
      const int ex = group_exclusive_scan<NT>(m, &tot, s_scan);
      if (m) sm.hit[j] = -1 - (base + ex);  // encode: hit = 1, miss = -1 - rank
      if (j < keff) sm.mrank[j] = base + ex;
      base += tot;
    }
  }
  // one segment per 64-range that receives its first page
  for (int j = tid; j < keff; j += NT) {
    if (sm.hit[j] > 0) continue;
    const int r = sm.sel[j] >> 6;
    if (sm.dirs[r] >= 0) continue;
    if (atomicCAS(&sm.dirs[r], -1, -2) == -1) {
      const int sg = alloc_segment(a, (uint32_t)(unit * 2654435761u + r));
      if (sg < 0) {
        atomicOr(a.err, kErrCapacity);
        sm.dirs[r] = -3;
      } else {
        int32_t* e = a.seg + (int64_t)sg * kSeg;
        for (int i = 0; i < kSeg; ++i) e[i] = -1;
        a.seg_live[sg] = 0;
        sm.dirs[r] = sg;
      }
    }
  }
  group_sync<NT>();
  for (int j = tid; j < keff; j += NT) {
    const int code = sm.hit[j];
    if (code > 0) continue;
    const int rank = -1 - code;
    if (rank >= s_nfree) {  // cannot happen: the LRU step freed at least `demand` pages
      atomicOr(a.err, kErrInternal);
      continue;
    }
    const int s = sm.flist[rank];
    const int p = sm.sel[j];
    sm.sp[s] = p;
    sm.lu[s] = t;
    sm.sslot[j] = s;
    sm.hit[j] = 0;
    const int sg = sm.dirs[p >> 6];
    if (sg >= a.S) {
      atomicOr(a.err, kErrSegId);
    } else if (sg >= 0) {
      a.seg[(int64_t)sg * kSeg + (p & 63)] = s;
      atomicAdd(&a.seg_live[sg], 1);
    }
    const int idx = atomicAdd(&a.counters[kCtrMiss], 1);
    if (idx >= a.B * a.Hkv * k) {
      atomicOr(a.err, kErrIndex);
      continue;
    }
    const int64_t src = host_page_index(a, b, h, p), dst = unit * cap + s;
    a.miss_src[idx] = src;
    a.miss_dst[idx] = dst;
    a.miss_att[idx] = ul * a.ka + hits + has_tail + rank;  // misses follow the hits and the tail
    a.miss_valid[idx] = (a.part_valid && src >= 0 && src < a.host_pages)
                            ? (int)a.part_valid[src]
                            : ((p == P - 1) ? a.ntok_b[b] - p * kPart : kPart);
    if (src >= 0 && src < a.host_pages && dst >= 0 && dst < a.pool_slots) {
      sm.msrc[rank] = src;
      sm.mdst[rank] = dst;
      sm.midx[rank] = idx;
    } else {
      atomicOr(a.err, kErrIndex);  // never expected: the page is not copied
    }
  }
  group_sync<NT>();

  // ---------------- write back ----------------
  for (int s = tid; s < cap; s += NT) {
    g_sp[s] = sm.sp[s];
    g_lu[s] = sm.lu[s];
  }
  for (int d = tid; d < a.D; d += NT) a.dir[unit * a.D + d] = sm.dirs[d] < 0 ? -1 : sm.dirs[d];
  for (int j = tid; j < k; j += NT) {
    const bool v = j < keff;
    a.sel[(int64_t)ul * k + j] = v ? sm.sel[j] : -1;
    a.sel_slot[(int64_t)ul * k + j] = v ? sm.sslot[j] : -1;
    a.sel_hit[(int64_t)ul * k + j] = v ? (uint8_t)(sm.hit[j] > 0) : 0;
  }
  // attention order: hits (ascending partition) first, then the tail page (slot == cap),
  // then this step's misses
  {
    const int ntok = a.ntok_b[b];
    for (int j = tid; j < keff; j += NT) {
      const int p = sm.sel[j];
      const bool hit = sm.hit[j] > 0;
      const int pos = hit ? j - sm.mrank[j] : hits + has_tail + sm.mrank[j];
      a.att_slot[(int64_t)ul * a.ka + pos] = sm.sslot[j];
      const int64_t hp = host_page_index(a, b, h, p);
      a.att_valid[(int64_t)ul * a.ka + pos] = (a.part_valid && hp >= 0 && hp < a.host_pages)
                                                  ? (int)a.part_valid[hp]
                                                  : ((p == P - 1) ? ntok - p * kPart : kPart);
    }
    if (has_tail && tid == 0) {
      a.att_slot[(int64_t)ul * a.ka + hits] = cap;
      a.att_valid[(int64_t)ul * a.ka + hits] = a.tail_n[b];
    }
  }
  if (tid == 0) {
    a.n_hit[ul] = hits + has_tail;
    a.keff[ul] = keff;
    int32_t* info = a.unit_info + (int64_t)ul * 8;
    info[0] = hits;
    info[1] = misses;
    info[2] = resident;
    info[3] = demand;
    info[4] = demand > 0 ? s_cutoff : -1;
    info[5] = s_evicted;
    info[6] = t;
    info[7] = 0;
    if (hits) atomicAdd(&a.stats[kStatHits], (unsigned long long)hits);
    if (misses) atomicAdd(&a.stats[kStatMisses], (unsigned long long)misses);
    if (s_evicted) atomicAdd(&a.stats[kStatEvictions], (unsigned long long)s_evicted);
    if (demand > 0) atomicAdd(&a.stats[kStatLruRounds], 1ull);
    if (keff) atomicAdd(&a.stats[kStatSelected], (unsigned long long)keff);
  }

  // ---------------- Retrieve in this kernel (retrieve_in_select) ----------------
  // The group copies the unit's missing pages host -> HBM right after managing the
  // unit (while other units are still being selected), then publishes each page's
  // ready flag; the attend kernel then finds every page resident.
  if (a.retrieve_in_select && misses > 0) {
    group_sync<NT>();
    constexpr int kPV = kPageElems / 8;  // 16-byte vectors per page (2048)
    constexpr int kU = 8;                // vectors in flight per thread
    const int nvec = misses * kPV;
    const uint4* hs = reinterpret_cast<const uint4*>(a.host_store);
    uint4* pool = reinterpret_cast<uint4*>(a.pool);
    for (int blk = 0; blk < nvec; blk += NT * kU) {
      uint4 r[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = blk + u * NT + tid;
        if (e < nvec && sm.midx[e / kPV] >= 0) r[u] = __ldcs(hs + sm.msrc[e / kPV] * kPV + (e % kPV));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = blk + u * NT + tid;
        if (e < nvec && sm.midx[e / kPV] >= 0) pool[sm.mdst[e / kPV] * kPV + (e % kPV)] = r[u];
      }
    }
    __threadfence();
    group_sync<NT>();
    for (int r = tid; r < misses; r += NT)
      if (sm.midx[r] >= 0)
        asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(a.ready + sm.midx[r]), "r"(t + 1) : "memory");
  }
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

}  // namespace

bool select_fuses_score(const LayerArgs& a);

cudaError_t launch_score(const LayerArgs& a, cudaStream_t st) {
  if (a.P_max <= 0 || select_fuses_score(a)) return cudaSuccess;  // scored inside the select kernel
  dim3 grid((unsigned)((a.P_max + kScoreChunk - 1) / kScoreChunk), (unsigned)(a.B * a.Hkv));
  score_kernel<<<grid, kScoreThreads, 0, st>>>(a);
  return cudaGetLastError();
}

size_t select_manage_smem_bytes(const LayerArgs& a) { return sel_smem_layout(a.P_max, a.cap, a.k, a.D, nullptr, nullptr); }

template <int NT, bool F>
cudaError_t configure_one(size_t smem) {
  const int kMaxShared = 100;  // cudaSharedmemCarveoutMaxShared: no carveout switch before attention
  cudaError_t e = cudaFuncSetAttribute(select_manage_kernel<NT, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(select_manage_kernel<NT, F>, cudaFuncAttributePreferredSharedMemoryCarveout, kMaxShared);
}

cudaError_t select_manage_configure(size_t smem) {
  cudaError_t e;
  if ((e = configure_one<32, false>(smem)) != cudaSuccess) return e;
  if ((e = configure_one<32, true>(smem)) != cudaSuccess) return e;
  if ((e = configure_one<kSelThreads, false>(smem)) != cudaSuccess) return e;
  if ((e = configure_one<kSelThreads, true>(smem)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(score_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

bool select_fuses_score(const LayerArgs& a) { return a.B * a.Hkv >= 64 && a.P_max <= 4096; }
static bool select_single_warp(const LayerArgs& a) {
  if (a.select_group == 32 || a.select_group == kSelThreads) return a.select_group == 32;
  return a.P_max <= 128 && a.cap <= 1024 && a.k <= 256;  // measured: 512 threads win from P = 512 up
}

cudaError_t launch_select_manage(const LayerArgs& a, cudaStream_t st) {
  const size_t smem = select_manage_smem_bytes(a);
  const unsigned grid = (unsigned)(a.B * a.Hkv);
  const bool f = select_fuses_score(a), w = select_single_warp(a);
  if (w && f) select_manage_kernel<32, true><<<grid, kSelThreads, smem, st>>>(a);
  else if (w) select_manage_kernel<32, false><<<grid, kSelThreads, smem, st>>>(a);
  else if (f) select_manage_kernel<kSelThreads, true><<<grid, kSelThreads, smem, st>>>(a);
  else select_manage_kernel<kSelThreads, false><<<grid, kSelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

__global__ void set_int_kernel(int32_t* p, int32_t v) { *p = v; }

cudaError_t launch_set_int(int32_t* p, int32_t v, cudaStream_t st) {
  set_int_kernel<<<1, 1, 0, st>>>(p, v);
  return cudaGetLastError();
}

cudaError_t launch_resolve_all(const LayerArgs& a, int32_t* resolve, int32_t* live_segs, cudaStream_t st) {
  resolve_all_kernel<<<a.B * a.Hkv, 256, 0, st>>>(a, resolve, live_segs);
  return cudaGetLastError();
}

}  // namespace spin
