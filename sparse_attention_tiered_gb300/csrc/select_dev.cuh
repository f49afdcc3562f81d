// Device code of Select (partition scores, per-unit top-k) and of the page manager
// (two-level resolve, bump, bucketed LRU, slot assignment, table update). Included
// by the decode-step kernel and by the allocation-free Select, so both compute the
// same selection by construction.
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
#pragma once

#include "spin_internal.cuh"

namespace spin {
namespace sel {

__device__ __forceinline__ float bf16f(uint32_t h) { return __uint_as_float(h << 16); }

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
// Scores: sc_p = (sum_g q_g) . s_p in fp32. Lane l holds dimensions 4l..4l+3: the
// query sum is added in head order, the dot product is one mul and three fma per
// lane, then a butterfly sum over the warp.
// ---------------------------------------------------------------------------
constexpr int kRowsPerBatch = 8;  // partitions scored by one warp at a time (8 loads in flight per lane)

// q: the group's query rows [G][128] bf16 (8-byte aligned rows). `staged`: the rows were
// copied into place earlier in the same kernel, so they are read with coherent loads (else
// through the read-only cache).
__device__ __forceinline__ float4 qsum_lane(const uint16_t* __restrict__ q, int G, int lane, bool staged = false) {
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int g = 0; g < G; ++g) {
    const uint2* r = reinterpret_cast<const uint2*>(q + (int64_t)g * kD) + lane;
    const uint2 v = staged ? __ldcg(r) : __ldg(r);
    s.x += bf16f(v.x & 0xffffu);
    s.y += bf16f(v.x >> 16);
    s.z += bf16f(v.y & 0xffffu);
    s.w += bf16f(v.y >> 16);
  }
  return s;
}

// Loads the lane's 16-byte slices of the n <= kRowsPerBatch summary rows at su
// ([rows][128] fp32, as float4); rows past n read as zero.
__device__ __forceinline__ void load_rows(float4 (&sv)[kRowsPerBatch], const float4* __restrict__ su, int n,
                                          int lane) {
#pragma unroll
  for (int i = 0; i < kRowsPerBatch; ++i)
    sv[i] = i < n ? __ldg(su + (int64_t)i * (kD / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Scores of the rows in sv; lane i < kRowsPerBatch returns row i's score (-0 returned as +0).
__device__ __forceinline__ float score_batch(const float4 (&sv)[kRowsPerBatch], float4 qv, int lane) {
  float mine = 0.f;
#pragma unroll
  for (int i = 0; i < kRowsPerBatch; ++i) {
    float x = sv[i].x * qv.x;
    x = fmaf(sv[i].y, qv.y, x);
    x = fmaf(sv[i].z, qv.z, x);
    x = fmaf(sv[i].w, qv.w, x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    mine = (lane == i) ? x : mine;
  }
  return mine == 0.f ? 0.f : mine;
}

// Histogram of the top kHistBits key bits per wide unit, filled while scoring, so the
// top-k of a wide unit starts with those bits resolved.
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;

// ---------------------------------------------------------------------------
// Thread groups. A group is NT consecutive threads of a CTA (NT a multiple of 32);
// groups synchronise with a named barrier of their own (one warp: __syncwarp).
// ---------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ void gsync(int bar) {
  if constexpr (NT == 32) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(NT) : "memory");
  }
}

// Shared scalars of one group.
struct GroupScalars {
  int bin, above, ncand, nlist, ntaken, total, unit, ok;
  int cnt_hits, cnt_res, cutoff, evicted, nfree, pad0, pad1, pad2;
  int wgt[16], weq[16], wpos[16], wtake[16], scan[16];
};

// Exclusive scan of one int per thread over the NT threads of a group; *total = sum.
template <int NT>
__device__ int group_exclusive_scan(int v, int* total, GroupScalars* gs, int gt, int bar) {
  constexpr int kW = NT / 32;
  const int lane = gt & 31, w = gt >> 5;
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
    if (lane == 31) gs->scan[w] = x;
    gsync<NT>(bar);
    if (w == 0) {
      int s = lane < kW ? gs->scan[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      if (lane < kW) gs->scan[lane] = s;  // inclusive
    }
    gsync<NT>(bar);
    const int before = (w > 0 ? gs->scan[w - 1] : 0) + x - v;
    *total = gs->scan[kW - 1];
    gsync<NT>(bar);
    return before;
  }
}

// ---------------------------------------------------------------------------
// Top-k of one unit by one group: radix select of the k-th largest key (four 8-bit
// passes over order-preserving keys), then compaction in ascending partition order
// with equal keys taken from the lowest partition up.
// Units with more than kWideP partitions (groups of >= 256 threads only) keep the
// first pass's threshold bin in `cand` for the later passes, and rank a short list of
// the keys >= the threshold instead of scanning every key per warp.
// ---------------------------------------------------------------------------
constexpr int kWideP = 4096;
constexpr int kCandMax = 8192;
__host__ __device__ inline int cand_capacity(int nt, int P_max) {
  return (nt >= 256 && P_max > kWideP) ? (P_max < kCandMax ? P_max : kCandMax) : 0;
}
// keys >= the threshold ranked by the list compaction: three arrays in the histogram scratch
__host__ __device__ constexpr int list_max(int nt) { return (nt / 32) * 256 / 3 < 1024 ? (nt / 32) * 256 / 3 : 1024; }

// keys [P] (shared), whist [NT/32][256] and cand [cand_cap] scratch (shared), sel [keff] out (shared).
// Returns false (after a group barrier) when the selection did not come out at keff entries,
// which never happens for consistent input.
template <int NT>
__device__ bool group_topk(const uint32_t* keys, int P, int keff, uint32_t* whist, uint32_t* cand, int cand_cap,
                           GroupScalars* gs, int bar, int gt, int32_t* sel) {
  constexpr int kW = NT / 32;
  const int lane = gt & 31, w = gt >> 5;
  uint32_t prefix = 0, mask = 0;
  int krem = keff;
  const bool wide = NT >= 256 && P > kWideP && cand_cap > 0;
  int ncand = -1;  // >= 0: the later passes scan cand[0, ncand) instead of every key
  int rb = 32;     // key bits still to resolve (from the top)
  if (keff > 0) {
    for (bool first = rb == 32; rb > 0; first = false) {
      const int digit = rb >= 8 ? 8 : rb;
      const int shift = rb - digit;
      const uint32_t dmask = (1u << digit) - 1u;
      for (int i = gt; i < kW * 256; i += NT) whist[i] = 0;
      gsync<NT>(bar);
      const uint32_t* src = ncand >= 0 ? cand : keys;
      const int nsrc = ncand >= 0 ? ncand : P;
      for (int p = gt; p < nsrc; p += NT) {
        const uint32_t key = src[p];
        if ((key & mask) == prefix) atomicAdd(&whist[w * 256 + ((key >> shift) & dmask)], 1u);
      }
      gsync<NT>(bar);
      if constexpr (kW > 1) {
        for (int i = gt; i < 256; i += NT) {
          uint32_t s = 0;
          for (int ww = 0; ww < kW; ++ww) s += whist[ww * 256 + i];
          whist[i] = s;  // row 0 now holds the merged histogram (each thread owns its columns)
        }
      }
      gsync<NT>(bar);
      if (w == 0) {
        // lane l owns bins 255-8l down to 248-8l (the top bins first)
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
              gs->bin = 255 - 8 * lane - i;
              gs->above = above;
              break;
            }
            above += c[i];
          }
        }
      }
      gsync<NT>(bar);
      const int bin = gs->bin;
      prefix |= (uint32_t)bin << shift;
      mask |= dmask << shift;
      krem -= gs->above;
      if (first && wide && (int)whist[bin] <= cand_cap) {
        // keep the keys of the threshold bin (row 0 of the histogram holds its merged count)
        if (gt == 0) gs->ncand = 0;
        gsync<NT>(bar);
        for (int p = gt; p < P; p += NT) {
          const uint32_t key = keys[p];
          if ((key & mask) == prefix) cand[atomicAdd(&gs->ncand, 1)] = key;
        }
        gsync<NT>(bar);
        ncand = gs->ncand;
      }
      gsync<NT>(bar);
      rb -= digit;
    }
  }
  const uint32_t T = prefix;  // the k-th largest key; krem = equal keys still to take

  // Wide units: the keys >= T go to a short unordered list (partition, key) in the
  // histogram scratch; each list entry is taken when its key is > T or it is one of the
  // krem equal keys with the lowest partitions, and lands at the rank of its partition
  // among the taken entries. A list that would overflow falls back to the warp scans.
  bool compacted = false;
  if (wide && keff > 0) {
    constexpr int kL = list_max(NT);
    int32_t* lp = reinterpret_cast<int32_t*>(whist);                // [kL] partition
    uint32_t* lk = whist + kL;                                       // [kL] key
    int32_t* tk = reinterpret_cast<int32_t*>(whist) + 2 * kL;       // [kL] taken flag
    if (gt == 0) {
      gs->nlist = 0;
      gs->ntaken = 0;
    }
    gsync<NT>(bar);
    for (int p = gt; p < P; p += NT) {
      const uint32_t key = keys[p];
      if (key >= T) {
        const int i = atomicAdd(&gs->nlist, 1);
        if (i < kL) {
          lp[i] = p;
          lk[i] = key;
        }
      }
    }
    gsync<NT>(bar);
    const int n = gs->nlist;
    if (n <= kL) {
      for (int i = gt; i < n; i += NT) {
        int taken = lk[i] > T;
        if (!taken) {  // equal key: taken when fewer than krem equal keys sit at lower partitions
          int eqb = 0;
          for (int j = 0; j < n; ++j) eqb += (lk[j] == T && lp[j] < lp[i]);
          taken = eqb < krem;
        }
        tk[i] = taken;
        if (taken) atomicAdd(&gs->ntaken, 1);
      }
      gsync<NT>(bar);
      if (gs->ntaken != keff) {
        gsync<NT>(bar);
        return false;
      }
      for (int i = gt; i < n; i += NT) {
        if (!tk[i]) continue;
        int pos = 0;
        for (int j = 0; j < n; ++j) pos += (tk[j] && lp[j] < lp[i]);
        if (pos < keff) sel[pos] = lp[i];
      }
      compacted = true;
    }
    gsync<NT>(bar);
  }
  if (!compacted) {
    const int chunk = ((P + NT - 1) / NT) * 32;
    const int wb = w * chunk, we = min(P, wb + chunk);
    int gt_n = 0, eq_n = 0;
    if (keff > 0)
      for (int base = wb; base < we; base += 32) {
        const int p = base + lane;
        const uint32_t key = p < we ? keys[p] : 0u;
        gt_n += __popc(__ballot_sync(0xffffffffu, p < we && key > T));
        eq_n += __popc(__ballot_sync(0xffffffffu, p < we && key == T));
      }
    if (lane == 0) {
      gs->wgt[w] = gt_n;
      gs->weq[w] = eq_n;
    }
    gsync<NT>(bar);
    if (gt == 0) {
      int eq_before = 0, pos = 0;
      for (int ww = 0; ww < kW; ++ww) {
        const int take = max(0, min(krem - eq_before, gs->weq[ww]));
        gs->wpos[ww] = pos;
        gs->wtake[ww] = take;
        pos += gs->wgt[ww] + take;
        eq_before += gs->weq[ww];
      }
      gs->total = pos;
    }
    gsync<NT>(bar);
    if (gs->total != keff) {
      gsync<NT>(bar);
      return false;
    }
    int pos = gs->wpos[w], eq_left = gs->wtake[w];
    if (keff > 0)
      for (int base = wb; base < we; base += 32) {
        const int p = base + lane;
        const uint32_t key = p < we ? keys[p] : 0u;
        const bool isgt = p < we && key > T;
        const bool iseq = p < we && key == T;
        const uint32_t meq = __ballot_sync(0xffffffffu, iseq);
        const bool take = isgt || (iseq && __popc(meq & lanemask_lt()) < eq_left);
        const uint32_t msel = __ballot_sync(0xffffffffu, take);
        if (take && pos + __popc(msel & lanemask_lt()) < keff) sel[pos + __popc(msel & lanemask_lt())] = p;
        pos += __popc(msel);
        eq_left -= min(eq_left, __popc(meq));
      }
  }
  gsync<NT>(bar);
  return true;
}

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// ---------------------------------------------------------------------------
// Top-k of a wide unit from the histogram of its keys' top 12 bits (filled while
// scoring, cleared here as it is read): the threshold value b1 of those bits comes
// from the histogram, one pass over the unit's scores keeps the (partition, key)
// pairs whose top bits are >= b1, the radix resolves the low 20 bits over the pairs
// at b1 only, and the taken pairs are ranked by partition. Never loads every key into
// shared memory. Returns 1 with sel[0, keff) filled, 0 when the caller must run the
// general top-k instead (the list would not fit, or too many keys tie at the
// threshold), -1 when the selection did not come out at keff entries.
// list_p / list_k: shared scratch of lmax entries each; tmp: shared scratch of >= keff ints.
// ---------------------------------------------------------------------------
template <int NT>
__device__ int wide_topk(const float* __restrict__ sc, int P, int keff, int32_t* __restrict__ hist12,
                         int32_t* list_p, uint32_t* list_k, int lmax, int32_t* tmp, uint32_t* whist,
                         GroupScalars* gs, int bar, int gt, int32_t* sel) {
  static_assert(NT >= 256, "wide units need a group of at least 256 threads");
  constexpr int kW = NT / 32;
  constexpr int kPer = kHistBins / NT;
  constexpr int kShift = 32 - kHistBits;
  const int lane = gt & 31, w = gt >> 5;
  // The unit's scores go out with the histogram's counts when they fit eight 16-byte loads
  // a thread: one memory round trip before the list can be built.
  const int n4 = (P + 3) >> 2;
  const bool in_regs = (reinterpret_cast<uintptr_t>(sc) & 15) == 0 && n4 <= 8 * NT;
  const float4* sc4 = reinterpret_cast<const float4*>(sc);
  float4 v4[8];
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = w * 32 + u * NT + lane;
      v4[u] = i < n4 ? __ldcg(sc4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // 1. the threshold value of the top 12 bits
  // thread gt holds the kPer bins below kHistBins - kPer * gt (c[0] the highest), read and
  // cleared with 16-byte accesses
  static_assert(kPer % 4 == 0, "whole int4 runs of bins per thread");
  int c[kPer], lsum = 0;
  {
    int4* h4 = reinterpret_cast<int4*>(hist12 + kHistBins - kPer * (gt + 1));
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const int4 x = __ldcg(h4 + q);
      c[kPer - 1 - 4 * q] = x.x;
      c[kPer - 2 - 4 * q] = x.y;
      c[kPer - 3 - 4 * q] = x.z;
      c[kPer - 4 - 4 * q] = x.w;
    }
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) h4[q] = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kPer; ++i) lsum += c[i];
  }
  int tot;
  const int excl = group_exclusive_scan<NT>(lsum, &tot, gs, gt, bar);
  if (keff > 0 && excl < keff && excl + lsum >= keff) {
    int above = excl;
    for (int i = 0; i < kPer; ++i) {
      if (above + c[i] >= keff) {
        gs->bin = kHistBins - 1 - kPer * gt - i;
        gs->above = above;
        gs->total = c[i];
        break;
      }
      above += c[i];
    }
  }
  if (gt == 0) gs->nlist = 0;
  gsync<NT>(bar);
  if (keff <= 0 || tot != P || gs->above + gs->total > lmax) return 0;
  const uint32_t b1 = (uint32_t)gs->bin;
  // 2. the pairs at or above b1: each lane loads 4 consecutive scores at a time (16-byte
  // loads when the row is 16-byte aligned), eight loads in flight per lane
  auto append = [&](int p, float v) {
    const uint32_t key = float_key(v);
    const bool in = p < P && (key >> kShift) >= b1;
    const uint32_t m = __ballot_sync(0xffffffffu, in);
    int base = 0;
    if (lane == 0 && m) base = atomicAdd(&gs->nlist, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (in) {
      list_p[base + __popc(m & lanemask_lt())] = p;
      list_k[base + __popc(m & lanemask_lt())] = key;
    }
  };
  if (in_regs) {
    // each lane counts its keys at or above the threshold; one warp scan and one
    // shared-memory atomic a warp place them, and each lane writes its own
    const uint32_t kb = b1 << kShift;
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = 4 * (w * 32 + u * NT + lane);
      cnt += (p < P && float_key(v4[u].x) >= kb) + (p + 1 < P && float_key(v4[u].y) >= kb) +
             (p + 2 < P && float_key(v4[u].z) >= kb) + (p + 3 < P && float_key(v4[u].w) >= kb);
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int wtot = __shfl_sync(0xffffffffu, incl, 31);
    int base = 0;
    if (lane == 0 && wtot) base = atomicAdd(&gs->nlist, wtot);
    base = __shfl_sync(0xffffffffu, base, 0) + incl - cnt;
    if (cnt) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = 4 * (w * 32 + u * NT + lane);
        const float vv[4] = {v4[u].x, v4[u].y, v4[u].z, v4[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t key = float_key(vv[c]);
          if (p + c < P && key >= kb) {
            list_p[base] = p + c;
            list_k[base] = key;
            ++base;
          }
        }
      }
    }
  } else if ((reinterpret_cast<uintptr_t>(sc) & 15) == 0) {
    for (int i0 = w * 32; i0 < n4; i0 += 8 * NT) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * NT + lane;
        v[u] = i < n4 ? __ldcg(sc4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = 4 * (i0 + u * NT + lane);
        append(p, v[u].x);
        append(p + 1, v[u].y);
        append(p + 2, v[u].z);
        append(p + 3, v[u].w);
      }
    }
  } else {
    for (int p0 = w * 32; p0 < P; p0 += 8 * NT) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = p0 + u * NT + lane;
        v[u] = p < P ? __ldcg(sc + p) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) append(p0 + u * NT + lane, v[u]);
    }
  }
  gsync<NT>(bar);
  const int n = gs->nlist;
  // 3. radix over the pairs at b1: bits 19..0 in digits of 8, 8 and 4. One shared
  // histogram (the pairs are few), two of them alternating: warp 0 scans one while the
  // other warps clear the next, two barriers a pass.
  uint32_t prefix = b1 << kShift, mask = ~0u << kShift;
  int krem = keff - gs->above;
  uint32_t* hcur = whist;
  uint32_t* hnxt = whist + 256;
  for (int i = gt; i < 256; i += NT) hcur[i] = 0;
  gsync<NT>(bar);
  for (int rb = kShift; rb > 0;) {
    const int digit = rb >= 8 ? 8 : rb;
    const int shift = rb - digit;
    const uint32_t dmask = (1u << digit) - 1u;
    for (int i = gt; i < n; i += NT) {
      const uint32_t key = list_k[i];
      if ((key & mask) == prefix) atomicAdd(&hcur[(key >> shift) & dmask], 1u);
    }
    gsync<NT>(bar);
    if (w == 0) {
      int cc[8], ls = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cc[i] = (int)hcur[255 - 8 * lane - i];
        ls += cc[i];
      }
      int incl = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int ex = incl - ls;
      const uint32_t hitm = __ballot_sync(0xffffffffu, ex < krem && incl >= krem);
      if (lane == __ffs(hitm) - 1) {
        int above = ex;
        for (int i = 0; i < 8; ++i) {
          if (above + cc[i] >= krem) {
            gs->bin = 255 - 8 * lane - i;
            gs->above = above;
            break;
          }
          above += cc[i];
        }
      }
    } else {
      for (int i = gt - 32; i < 256; i += NT - 32) hnxt[i] = 0;
    }
    gsync<NT>(bar);
    prefix |= (uint32_t)gs->bin << shift;
    mask |= dmask << shift;
    krem -= gs->above;
    uint32_t* h = hcur;
    hcur = hnxt;
    hnxt = h;
    rb -= digit;
  }
  const uint32_t T = prefix;  // the k-th largest key; krem = equal keys still to take
  // 4. taken pairs: keys > T, then the krem equal keys with the lowest partitions (ranked
  // among the equal pairs, gathered in the histogram scratch)
  int32_t* eq_p = reinterpret_cast<int32_t*>(whist);
  constexpr int kEqMax = kW * 256;
  if (gt == 0) {
    gs->ntaken = 0;
    gs->ncand = 0;
  }
  gsync<NT>(bar);
  for (int i0 = w * 32; i0 < n; i0 += NT) {  // one shared-memory atomic per warp and kind
    const int i = i0 + lane;
    const uint32_t key = i < n ? list_k[i] : 0u;
    const bool above = i < n && key > T, equal = i < n && key == T;
    const uint32_t mg = __ballot_sync(0xffffffffu, above), me = __ballot_sync(0xffffffffu, equal);
    int bg = 0, be = 0;
    if (lane == 0) {
      if (mg) bg = atomicAdd(&gs->ntaken, __popc(mg));
      if (me) be = atomicAdd(&gs->ncand, __popc(me));
    }
    bg = __shfl_sync(0xffffffffu, bg, 0);
    be = __shfl_sync(0xffffffffu, be, 0);
    if (above) {
      const int j = bg + __popc(mg & lanemask_lt());
      if (j < keff) tmp[j] = list_p[i];
    }
    if (equal) {
      const int j = be + __popc(me & lanemask_lt());
      if (j < kEqMax) eq_p[j] = list_p[i];
    }
  }
  gsync<NT>(bar);
  const int ngt = gs->ntaken, neq = gs->ncand;
  if (neq > kEqMax || ngt + krem != keff || neq < krem) {
    gsync<NT>(bar);
    return neq > kEqMax ? 0 : -1;
  }
  for (int i = gt; i < neq; i += NT) {
    const int pi = eq_p[i];
    int r = 0;
    for (int j = 0; j < neq; ++j) r += eq_p[j] < pi;
    if (r < krem) tmp[ngt + r] = pi;
  }
  gsync<NT>(bar);
  // 5. ascending partition order
  for (int i = gt; i < keff; i += NT) {
    const int pi = tmp[i];
    int r = 0;
    for (int j = 0; j < keff; ++j) r += tmp[j] < pi;
    sel[r] = pi;
  }
  gsync<NT>(bar);
  return 1;
}

// ---------------------------------------------------------------------------
// Page manager of one unit, by one group of NT threads.
// ---------------------------------------------------------------------------
struct MgrSmem {
  uint32_t* keys;     // [P_max]
  int32_t* sp;        // [cap] slot -> partition
  int32_t* lu;        // [cap] slot -> last use
  int32_t* flist;     // [cap] free slots ascending
  int32_t* sel;       // [k]
  int32_t* sslot;     // [k]
  int32_t* hit;       // [k]
  int32_t* mrank;     // [k] misses before j (exclusive)
  int32_t* dirs;      // [D]
  uint32_t* whist;    // [NT/32][256]
  uint8_t* mand;      // [cap]
  uint32_t* cand;     // [cand_capacity(NT, P_max)]
  GroupScalars* gs;
  int cand_cap;
};

// Bytes of one manager group's shared memory (base == nullptr) or its layout at base.
__host__ __device__ inline size_t mgr_smem_layout(int nt, int P_max, int cap, int k, int D, MgrSmem* s,
                                                  uint8_t* base) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += align16(bytes);
    return p;
  };
  const int cc = cand_capacity(nt, P_max);
  uint8_t* gs = take(sizeof(GroupScalars));
  uint8_t* keys = take(sizeof(uint32_t) * (size_t)(P_max > 0 ? P_max : 1));
  uint8_t* sp = take(sizeof(int32_t) * cap);
  uint8_t* lu = take(sizeof(int32_t) * cap);
  uint8_t* fl = take(sizeof(int32_t) * cap);
  uint8_t* sl = take(sizeof(int32_t) * k);
  uint8_t* ss = take(sizeof(int32_t) * k);
  uint8_t* hit = take(sizeof(int32_t) * k);
  uint8_t* mrank = take(sizeof(int32_t) * k);
  uint8_t* dirs = take(sizeof(int32_t) * (D > 0 ? D : 1));
  uint8_t* wh = take(sizeof(uint32_t) * (size_t)(nt / 32) * 256);
  uint8_t* mand = take((size_t)cap);
  uint8_t* cand = take(sizeof(uint32_t) * (size_t)(cc > 0 ? cc : 1));
  if (s) {
    s->gs = (GroupScalars*)gs;
    s->keys = (uint32_t*)keys;
    s->sp = (int32_t*)sp;
    s->lu = (int32_t*)lu;
    s->flist = (int32_t*)fl;
    s->sel = (int32_t*)sl;
    s->sslot = (int32_t*)ss;
    s->hit = (int32_t*)hit;
    s->mrank = (int32_t*)mrank;
    s->dirs = (int32_t*)dirs;
    s->whist = (uint32_t*)wh;
    s->mand = mand;
    s->cand = (uint32_t*)cand;
    s->cand_cap = cc;
  }
  return off;
}

// Memory-order helpers. A GPU-scope fence waits for the executing thread's earlier
// accesses, and on an SM whose other warps have host-link loads queued that takes many
// microseconds: the manager uses as few as its ordering needs.
__device__ __forceinline__ void fence_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void st_relaxed_i32(int32_t* p, int32_t v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t atom_add_acq_rel_i32(int32_t* p, int32_t v) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t atom_or_acquire(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acquire.gpu.global.or.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Claim a free segment of the shared pool (bitmap, lock free). -1 when exhausted. The
// first try sets the hinted bit of the hinted word (one round trip when it is free); the
// bits the atomic returns pick the next tries. Acquire: the previous owner's writes to
// the segment come before ours (bits past S are set for good, so they are never taken).
__device__ inline int alloc_segment(const LayerArgs& a, uint32_t hint) {
  const int nwords = (a.S + 31) >> 5;
  const int w0 = (int)(hint % (uint32_t)nwords);
  const uint32_t m0 = 1u << ((hint / (uint32_t)nwords) & 31u);
  uint32_t bits = atom_or_acquire(&a.seg_bitmap[w0], m0);
  if (!(bits & m0)) return w0 * 32 + (__ffs(m0) - 1);
  for (int i = 0; i < nwords; ++i) {
    const int w = (w0 + i) % nwords;
    if (i > 0) bits = *((volatile uint32_t*)&a.seg_bitmap[w]);
    for (int tries = 0; tries < 33 && bits != 0xffffffffu; ++tries) {
      const int bit = __ffs(~bits) - 1;
      const uint32_t old = atom_or_acquire(&a.seg_bitmap[w], 1u << bit);
      if (!(old & (1u << bit))) return w * 32 + bit;
      bits = old | (1u << bit);
    }
  }
  return -1;
}

__device__ __forceinline__ void release_segment(const LayerArgs& a, int sg) {
  fence_rel();  // the unit's writes to the segment come before the next owner's
  atomicAnd(&a.seg_bitmap[sg >> 5], ~(1u << (sg & 31)));
}

__device__ __forceinline__ void st_release_i32(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Publishes unit ul, by one thread after a barrier of the group that wrote it: the
// release fence covers every write the barrier ordered before it (the group's), and is
// followed by the tags of the unit's miss-list entries [mbase, mbase + misses) (entries
// at or past kmax were never written), the unit's ready flag and the managed count.
__device__ inline void publish_unit(const LayerArgs& a, int ul, int tag, int mbase = 0, int misses = 0,
                                    int kmax = 0) {
  fence_rel();
  for (int r = 0; r < misses && mbase + r < kmax; ++r) st_relaxed_i32(a.miss_tag + mbase + r, tag);
  st_relaxed_i32(a.unit_ready + ul, tag);
  atomicAdd(&a.counters[kCtrManaged], 1);
}

// Select + manage unit ul of the layer at step t, once its scores are all in sc ([P], this
// step's buffer). sc_reset (the pipelined kernel): the unit's slots in the other buffer,
// set back to kScoreEmpty for the next step.
// Writes the selection, slots, attention order, page state, two-level table, stats and
// this step's miss-list entries, then (one thread, one release fence) the entries' tags
// in miss_tag, the unit's flag (unit_ready = tag) and its count in kCtrManaged. A unit whose
// page state can no longer be trusted (device error word) or whose top-k failed is
// published with nothing selected.
template <int NT>
__device__ void manage_unit(const LayerArgs& a, int ul, int t, int tag, const MgrSmem& sm, int bar, int gt,
                            const float* sc, float* sc_reset) {
  constexpr int kW = NT / 32;
  GroupScalars* gs = sm.gs;
  const int lane = gt & 31;
  const int b = ul / a.Hkv, h = ul % a.Hkv;
  const int P = a.P_b[b];
  const int k = a.k, cap = a.cap;
  int keff = P < k ? P : k;
  const int64_t unit = a.unit_base + ul;
  if (sc_reset)  // the next step's buffer: every slot it will write starts empty
    for (int p = gt; p < P; p += NT) sc_reset[p] = __uint_as_float(kScoreEmpty);
  // the device error word: read now, used once the unit's loads below are on their way
  const uint32_t err0 = *((volatile uint32_t*)a.err);

  // The unit's page state does not depend on the selection: its loads go out now, into
  // registers, and land in shared memory after the top-k (when it fits kPf entries a thread).
  constexpr int kPf = 4;
  int32_t* g_sp = a.slot_part + unit * cap;
  int32_t* g_lu = a.last_use + unit * cap;
  const int32_t* g_dir = a.dir + unit * a.D;
  const bool pf = cap <= kPf * NT && a.D <= 2 * NT;
  // 16-byte loads when the rows are 16-byte aligned: thread gt holds slots 4gt .. 4gt+3
  const bool pf4 = pf && (cap & 3) == 0;
  int32_t pf_sp[kPf], pf_lu[kPf], pf_dir[2];
  if (pf4) {
    const int4 z4 = make_int4(-1, -1, -1, -1), l4 = make_int4(0, 0, 0, 0);
    const int4 v = 4 * gt < cap ? reinterpret_cast<const int4*>(g_sp)[gt] : z4;
    const int4 w = 4 * gt < cap ? reinterpret_cast<const int4*>(g_lu)[gt] : l4;
    pf_sp[0] = v.x, pf_sp[1] = v.y, pf_sp[2] = v.z, pf_sp[3] = v.w;
    pf_lu[0] = w.x, pf_lu[1] = w.y, pf_lu[2] = w.z, pf_lu[3] = w.w;
  } else if (pf) {
#pragma unroll
    for (int i = 0; i < kPf; ++i) {
      const int sl = gt + i * NT;
      pf_sp[i] = sl < cap ? g_sp[sl] : -1;
      pf_lu[i] = sl < cap ? g_lu[sl] : 0;
    }
  }
  if (pf) {
#pragma unroll
    for (int i = 0; i < 2; ++i) pf_dir[i] = gt + i * NT < a.D ? g_dir[gt + i * NT] : -1;
  }

  // ---------------- top-k ----------------
  int wide_done = 0;
  if constexpr (NT >= 256) {
    if (a.hist12 != nullptr) {
      // the list lives in the keys' shared memory: P_max / 2 (partition, key) pairs. Run
      // whatever the error word says: it also clears the unit's histogram for the next step.
      const int lmax = a.P_max / 2;
      wide_done = wide_topk<NT>(sc, P, keff, a.hist12 + (int64_t)ul * kHistBins,
                                reinterpret_cast<int32_t*>(sm.keys), sm.keys + lmax, lmax, sm.flist, sm.whist, gs,
                                bar, gt, sm.sel);
    }
  }
  const bool dead = (err0 & (kErrCapacity | kErrInternal | kErrSelCount | kErrSegId | kErrIndex)) != 0;
  bool ok = !dead;
  if (ok && wide_done < 0) {
    ok = false;
    if (gt == 0) atomicOr(a.err, kErrSelCount);
  }
  if (ok && wide_done == 0) {
    for (int p0 = gt; p0 < P; p0 += 8 * NT) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (p0 + u * NT < P) ? __ldcg(sc + p0 + u * NT) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p0 + u * NT < P) sm.keys[p0 + u * NT] = float_key(v[u]);
    }
    gsync<NT>(bar);
    ok = group_topk<NT>(sm.keys, P, keff, sm.whist, sm.cand, sm.cand_cap, gs, bar, gt, sm.sel);
    if (!ok && gt == 0) atomicOr(a.err, kErrSelCount);
  }
  const int has_tail = (a.tail_n != nullptr && a.tail_n[b] > 0) ? 1 : 0;
  if (!ok) {
    // publish the unit with nothing selected (its tail, if any, is still attended)
    for (int j = gt; j < k; j += NT) {
      a.sel[(int64_t)ul * k + j] = -1;
      a.sel_slot[(int64_t)ul * k + j] = -1;
      a.sel_hit[(int64_t)ul * k + j] = 0;
    }
    if (gt == 0) {
      if (has_tail) {
        a.att_slot[(int64_t)ul * a.ka] = cap;
        a.att_valid[(int64_t)ul * a.ka] = a.tail_n[b];
      }
      a.n_hit[ul] = has_tail;
      a.keff[ul] = 0;
    }
    gsync<NT>(bar);
    if (gt == 0) publish_unit(a, ul, tag);
    return;
  }

  // ---------------- the unit's page state into shared memory ----------------
  if (pf) {
#pragma unroll
    for (int i = 0; i < kPf; ++i) {
      const int sl = pf4 ? 4 * gt + i : gt + i * NT;
      if (sl < cap) {
        sm.sp[sl] = pf_sp[i];
        sm.lu[sl] = pf_lu[i];
        sm.mand[sl] = 0;
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (gt + i * NT < a.D) sm.dirs[gt + i * NT] = pf_dir[i];
  } else {
    for (int sl = gt; sl < cap; sl += NT) {
      sm.sp[sl] = g_sp[sl];
      sm.lu[sl] = g_lu[sl];
      sm.mand[sl] = 0;
    }
    for (int d = gt; d < a.D; d += NT) sm.dirs[d] = g_dir[d];
  }
  if (gt == 0) {
    gs->cnt_hits = 0;
    gs->cnt_res = 0;
    gs->cutoff = -1;
    gs->evicted = 0;
  }
  gsync<NT>(bar);

  // ---------------- 1. residency check through the two-level table; 2. bump ----------------
  for (int j = gt; j < keff; j += NT) {
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
      atomicAdd(&gs->cnt_hits, 1);
    } else if (slot >= cap) {
      sm.sslot[j] = -1;
      sm.hit[j] = 0;
    }
  }
  {
    int res = 0;
    for (int s = gt; s < cap; s += NT) res += sm.sp[s] >= 0;
    res = __reduce_add_sync(0xffffffffu, res);
    if (lane == 0 && res) atomicAdd(&gs->cnt_res, res);
  }
  gsync<NT>(bar);
  const int hits = gs->cnt_hits;
  const int misses = keff - hits;
  const int resident = gs->cnt_res;
  // free pages are counted against the request's budget (buffer elasticity): after a
  // shrink the demand includes the excess and the LRU reclaims down to the budget
  const int demand = misses - (a.budget_b[b] - resident);
  // the unit's entries in the step's miss list (ranks 0 .. misses-1): one reservation, sent
  // now so that its round trip overlaps the LRU and the slot assignment
  int mres = 0;
  if (gt == 0 && misses > 0) mres = atomicAdd(&a.counters[kCtrMiss], misses);

  // ---------------- 3. bucketed LRU ----------------
  if (demand > 0) {
    uint32_t* hist = sm.whist;  // 64 bins
    for (int i = gt; i < kBuckets; i += NT) hist[i] = 0;
    gsync<NT>(bar);
    for (int s = gt; s < cap; s += NT) {
      if (sm.sp[s] < 0 || sm.mand[s]) continue;
      const int age = t - sm.lu[s];
      const int bucket = kBuckets - 1 - min(kBuckets - 1, age);
      atomicAdd(&hist[bucket], 1u);
    }
    gsync<NT>(bar);
    if (gt < 32) {
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
      if (lane == __ffs(m) - 1) gs->cutoff = (excl + c0 >= demand) ? 2 * lane : 2 * lane + 1;
    }
    gsync<NT>(bar);
    const int cutoff = gs->cutoff;
    for (int s = gt; s < cap; s += NT) {
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
        // acq_rel: the last page out of the segment sees every clear before it frees it
        if (atom_add_acq_rel_i32(&a.seg_live[sg], -1) == 1) {
          sm.dirs[p >> 6] = -1;
          release_segment(a, sg);
        }
      } else {
        atomicOr(a.err, kErrInternal);  // a resident page without a table entry
      }
      sm.sp[s] = -1;
      atomicAdd(&gs->evicted, 1);
    }
    gsync<NT>(bar);
  }

  // ---------------- 4. assign free slots to misses, allocate segments ----------------
  {
    int base = 0;
    for (int r = 0; r < cap; r += NT) {
      const int s = r + gt;
      const int f = (s < cap && sm.sp[s] < 0) ? 1 : 0;
      int tot;
      const int ex = group_exclusive_scan<NT>(f, &tot, gs, gt, bar);
      if (f) sm.flist[base + ex] = s;
      base += tot;
    }
    if (gt == 0) gs->nfree = base;
  }
  // rank of each miss among the misses (ascending partition = ascending j)
  {
    int base = 0;
    for (int r = 0; r < keff; r += NT) {
      const int j = r + gt;
      const int m = (j < keff && !sm.hit[j]) ? 1 : 0;
      int tot;
      const int ex = group_exclusive_scan<NT>(m, &tot, gs, gt, bar);
      if (m) sm.hit[j] = -1 - (base + ex);  // encode: hit = 1, miss = -1 - rank
      if (j < keff) sm.mrank[j] = base + ex;
      base += tot;
    }
  }
  // one segment per 64-range that receives its first page
  for (int j = gt; j < keff; j += NT) {
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
  if (gt == 0) gs->ncand = mres;
  gsync<NT>(bar);
  const int kmax = a.B * a.Hkv * k;  // miss-list capacity
  const int mbase = gs->ncand;
  for (int j = gt; j < keff; j += NT) {
    const int code = sm.hit[j];
    if (code > 0) continue;
    const int rank = -1 - code;
    if (rank >= gs->nfree) {  // cannot happen: the LRU step freed at least `demand` pages
      atomicOr(a.err, kErrInternal);
      if (mbase + rank < kmax) {  // the reserved entry is published as one the retrievers skip
        a.miss_src[mbase + rank] = -1;
        a.miss_dst[mbase + rank] = -1;
        a.miss_att[mbase + rank] = -1;
      }
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
    const int idx = mbase + rank;
    if (idx >= kmax) {
      atomicOr(a.err, kErrIndex);
      continue;
    }
    const int64_t src = host_page_index(a, b, h, p), dst = unit * cap + s;
    const bool in_range = src >= 0 && src < a.host_pages && dst >= 0 && dst < a.pool_slots;
    if (!in_range) atomicOr(a.err, kErrIndex);  // never expected: the retriever skips the copy
    a.miss_src[idx] = in_range ? src : -1;
    a.miss_dst[idx] = in_range ? dst : -1;
    a.miss_att[idx] = ul * a.ka + hits + has_tail + rank;  // misses follow the hits and the tail
    a.miss_valid[idx] = (a.part_valid && in_range) ? (int)a.part_valid[src]
                                                    : ((p == P - 1) ? a.ntok_b[b] - p * kPart : kPart);
  }
  gsync<NT>(bar);

  // ---------------- write back ----------------
  for (int s = gt; s < cap; s += NT) {
    g_sp[s] = sm.sp[s];
    g_lu[s] = sm.lu[s];
  }
  for (int d = gt; d < a.D; d += NT) a.dir[unit * a.D + d] = sm.dirs[d] < 0 ? -1 : sm.dirs[d];
  for (int j = gt; j < k; j += NT) {
    const bool v = j < keff;
    a.sel[(int64_t)ul * k + j] = v ? sm.sel[j] : -1;
    a.sel_slot[(int64_t)ul * k + j] = v ? sm.sslot[j] : -1;
    a.sel_hit[(int64_t)ul * k + j] = v ? (uint8_t)(sm.hit[j] > 0) : 0;
  }
  // attention order: hits (ascending partition) first, then the tail page (slot == cap),
  // then this step's misses
  {
    const int ntok = a.ntok_b[b];
    for (int j = gt; j < keff; j += NT) {
      const int p = sm.sel[j];
      const bool hit = sm.hit[j] > 0;
      const int pos = hit ? j - sm.mrank[j] : hits + has_tail + sm.mrank[j];
      a.att_slot[(int64_t)ul * a.ka + pos] = sm.sslot[j];
      const int64_t hp = host_page_index(a, b, h, p);
      a.att_valid[(int64_t)ul * a.ka + pos] = (a.part_valid && hp >= 0 && hp < a.host_pages)
                                                  ? (int)a.part_valid[hp]
                                                  : ((p == P - 1) ? ntok - p * kPart : kPart);
    }
    if (has_tail && gt == 0) {
      a.att_slot[(int64_t)ul * a.ka + hits] = cap;
      a.att_valid[(int64_t)ul * a.ka + hits] = a.tail_n[b];
    }
  }
  if (gt == 0) {
    a.n_hit[ul] = hits + has_tail;
    a.keff[ul] = keff;
    int32_t* info = a.unit_info + (int64_t)ul * 8;
    info[0] = hits;
    info[1] = misses;
    info[2] = resident;
    info[3] = demand;
    info[4] = demand > 0 ? gs->cutoff : -1;
    info[5] = gs->evicted;
    info[6] = t;
    info[7] = 0;
    if (hits) atomicAdd(&a.stats[kStatHits], (unsigned long long)hits);
    if (misses) atomicAdd(&a.stats[kStatMisses], (unsigned long long)misses);
    if (gs->evicted) atomicAdd(&a.stats[kStatEvictions], (unsigned long long)gs->evicted);
    if (demand > 0) atomicAdd(&a.stats[kStatLruRounds], 1ull);
    if (keff) atomicAdd(&a.stats[kStatSelected], (unsigned long long)keff);
  }
  gsync<NT>(bar);
  // one release for the whole unit: the miss-list entries, the attention order and the
  // page state written above, then the entries' tags and the unit's flag
  if (gt == 0) publish_unit(a, ul, tag, mbase, misses, kmax);
  (void)kW;
}

}  // namespace sel
}  // namespace spin
