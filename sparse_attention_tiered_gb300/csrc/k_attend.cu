// Retrieve (host -> HBM page copies), paged split-KV decode attention and combine.
//
// Retrieve brings the critical partitions that are not resident from CPU memory
// into their HBM pages; Attention is exact softmax attention over the tokens of
// the selected partitions only (m.x-techcon.com SPIN article, section
// "Spin的核心设计" 1 and Figure 3, 2 and Figure 5 step 4; gist.science/pt section
// 2A). The pages give no kernel design; everything below is this library's.
//
// Attention data layout. A page (32 KiB) holds K[64][128] then V[64][128] bf16.
// A TMA tensor map views the whole HBM pool as a 2-D bf16 tensor of 128 columns
// and (slots * 128) rows; a page is loaded as four 64x64 boxes (K left/right, V
// left/right) with the 128-byte swizzle, so ldmatrix reads are bank-conflict free.
//
// Work split. One persistent CTA per SM: one producer warp (one elected lane
// issues TMA loads into a 4-stage ring of pages, guarded by mbarriers) and four
// consumer warps. A task is up to `ppt` consecutive selected pages of one unit;
// tasks are taken from a device counter. Every consumer warp handles 16 of the
// 64 tokens of each page for all G query heads of the unit:
//   S[16 heads][16 tokens] = Q K^T      mma.m16n8k16 bf16 -> fp32 (heads padded to 16)
//   online softmax in fp32 (base-2 exponent, scale log2(e)/sqrt(128))
//   O[16][128] += P V                    P split into bf16 hi + lo parts, two mma each
// At the end of a task the four warps merge (m, l, O) in shared memory and write
// one partial (m, l, acc[128]) per query head; the combine kernel merges the
// partials of a unit into the output.
//
// Every wait on an mbarrier is bounded in time; a wait that runs out sets the
// device error word, stops issuing work and drains the loads already issued.
#include "spin_internal.cuh"

namespace spin {

namespace {

constexpr int kStages = 4;
constexpr int kCWarps = 4;
constexpr int kAttnThreads = (kCWarps + 1) * 32;
constexpr int kMergeFloats = 16 * kD + 32;  // O[16][128], m[16], l[16]
constexpr float kScaleLog2 = 0.12751743074173449f;  // log2(e) / sqrt(128)
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s

struct StageMeta {
  int task, ul, j, valid;
};

struct AttnSmem {
  uint8_t* ring;      // kStages x 32 KiB, 1024-aligned
  float* merge;       // kCWarps x kMergeFloats
  uint64_t* full;     // [kStages]
  uint64_t* empty;    // [kStages]
  uint64_t* mrg;      // [2]: written, read
  StageMeta* meta;    // [kStages]
  int* abort_flag;
};

__host__ __device__ inline size_t attn_smem_layout(AttnSmem* s, uint8_t* base) {
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = (off + align - 1) & ~(align - 1);
    uint8_t* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  };
  uint8_t* ring = take((size_t)kStages * kPageBytes, 1024);
  uint8_t* merge = take(sizeof(float) * kCWarps * kMergeFloats, 16);
  uint8_t* full = take(sizeof(uint64_t) * kStages, 8);
  uint8_t* empty = take(sizeof(uint64_t) * kStages, 8);
  uint8_t* mrg = take(sizeof(uint64_t) * 2, 8);
  uint8_t* meta = take(sizeof(StageMeta) * kStages, 16);
  uint8_t* ab = take(sizeof(int), 4);
  if (s) {
    s->ring = ring;
    s->merge = (float*)merge;
    s->full = (uint64_t*)full;
    s->empty = (uint64_t*)empty;
    s->mrg = (uint64_t*)mrg;
    s->meta = (StageMeta*)meta;
    s->abort_flag = (int*)ab;
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
// Attention kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAttnThreads, 1)
attention_kernel(const __grid_constant__ CUtensorMap tmap, LayerArgs a, int n_tasks) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  AttnSmem sm;
  attn_smem_layout(&sm, base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kCWarps);
    }
    mbar_init(smem_u32(&sm.mrg[0]), kCWarps);
    mbar_init(smem_u32(&sm.mrg[1]), kCWarps);
    *sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort_flag = sm.abort_flag;

  if (warp == kCWarps) {
    // ------------------------------ producer ------------------------------
    if (lane != 0) return;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    int i = 0;
    bool ok = true;
    for (;;) {
      if (*abort_flag) { ok = false; break; }
      const int task = atomicAdd(&a.counters[1], 1);
      if (task >= n_tasks) break;
      const int ul = task / a.n_chunks, c = task - ul * a.n_chunks;
      const int keff = a.keff[ul];
      const int j0 = c * a.ppt, j1 = min(keff, j0 + a.ppt);
      const int b = ul / a.Hkv;
      const int P = a.P_b[b], ntok = a.ntok_b[b];
      const int64_t unit = a.unit_base + ul;
      for (int j = j0; j < j1; ++j) {
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait(smem_u32(&sm.empty[st]), ph ^ 1u)) { ok = false; break; }
        const int p = a.sel[(int64_t)ul * a.k + j];
        const int slot = a.sel_slot[(int64_t)ul * a.k + j];
        StageMeta m;
        m.task = task;
        m.ul = ul;
        m.j = j;
        m.valid = (p == P - 1) ? ntok - p * kPart : kPart;
        sm.meta[st] = m;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, kPageBytes);
        const int y = (int)((unit * a.cap + slot) * 128);
        const uint32_t dst = smem_u32(sm.ring + (size_t)st * kPageBytes);
        tma_load_2d(dst, &tmap, fb, 0, y);
        tma_load_2d(dst + 8192, &tmap, fb, 64, y);
        tma_load_2d(dst + 16384, &tmap, fb, 0, y + 64);
        tma_load_2d(dst + 24576, &tmap, fb, 64, y + 64);
        ++i;
      }
      if (!ok) break;
    }
    if (ok) {
      // sentinel: tells the consumers that no task follows
      const int st = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      if (mbar_wait(smem_u32(&sm.empty[st]), ph ^ 1u)) {
        sm.meta[st].task = -1;
        mbar_arrive(smem_u32(&sm.full[st]));
      } else {
        ok = false;
      }
    }
    if (!ok) {
      atomicOr(a.err, kErrTimeout);
      *abort_flag = 1;
      // drain the loads already issued before leaving (bounded)
      for (int m = max(0, i - kStages); m < i; ++m)
        (void)mbar_wait(smem_u32(&sm.full[m % kStages]), (uint32_t)(m / kStages) & 1u);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int w = warp;               // tokens 16w .. 16w+15 of every page
  const int t0 = 16 * w;
  const int mi = lane >> 3, ri = lane & 7;
  const int qr = lane >> 2, q4 = lane & 3;
  const int tokK = t0 + ri + ((mi >> 1) << 3);
  const int tokV = t0 + ri + ((mi & 1) << 3);
  float* mw = sm.merge + w * kMergeFloats;

  uint32_t qa[8][4];
  float o[16][4];
  float mrow[2], lrow[2];
  int cur = -1, cur_ul = -1;
  uint32_t mph = 0;
  int i = 0;

  for (;;) {
    const int st = i % kStages;
    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
    if (!mbar_wait(smem_u32(&sm.full[st]), ph)) {
      atomicOr(a.err, kErrTimeout);
      *abort_flag = 1;
      break;
    }
    const StageMeta m = sm.meta[st];
    if (m.task != cur || m.task < 0) {
      if (cur >= 0) {
        // ---- finalize the previous task: merge the four warps, write partials ----
        const float l0 = lrow[0] + __shfl_xor_sync(0xffffffffu, lrow[0], 1);
        const float l0b = l0 + __shfl_xor_sync(0xffffffffu, l0, 2);
        const float l1 = lrow[1] + __shfl_xor_sync(0xffffffffu, lrow[1], 1);
        const float l1b = l1 + __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          *reinterpret_cast<float2*>(&mw[qr * kD + 8 * n + 2 * q4]) = make_float2(o[n][0], o[n][1]);
          *reinterpret_cast<float2*>(&mw[(qr + 8) * kD + 8 * n + 2 * q4]) = make_float2(o[n][2], o[n][3]);
        }
        if (q4 == 0) {
          mw[16 * kD + qr] = mrow[0];
          mw[16 * kD + qr + 8] = mrow[1];
          mw[16 * kD + 16 + qr] = l0b;
          mw[16 * kD + 16 + qr + 8] = l1b;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.mrg[0]));
        if (!mbar_wait(smem_u32(&sm.mrg[0]), mph)) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        const int d = w * 32 + lane;  // 0..127
        for (int g = 0; g < a.G; ++g) {
          float M = -INFINITY;
#pragma unroll
          for (int ww = 0; ww < kCWarps; ++ww) M = fmaxf(M, sm.merge[ww * kMergeFloats + 16 * kD + g]);
          float L = 0.f, acc = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int ww = 0; ww < kCWarps; ++ww) {
              const float* src = sm.merge + ww * kMergeFloats;
              const float sc = exp2f(src[16 * kD + g] - M);
              L = fmaf(sc, src[16 * kD + 16 + g], L);
              acc = fmaf(sc, src[g * kD + d], acc);
            }
          }
          float* part = a.partials + ((int64_t)cur * a.G + g) * kPartialStride;
          part[4 + d] = acc;
          if (d == 0) {
            part[0] = M;
            part[1] = L;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.mrg[1]));
        if (!mbar_wait(smem_u32(&sm.mrg[1]), mph)) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        mph ^= 1u;
      }
      if (m.task < 0) break;
      cur = m.task;
      if (m.ul != cur_ul) {
        cur_ul = m.ul;
        const int b = m.ul / a.Hkv, h = m.ul - b * a.Hkv;
        const uint16_t* qb = a.q + ((int64_t)b * a.Hq + (int64_t)h * a.G) * kD;
        const bool r0 = qr < a.G, r1 = qr + 8 < a.G;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int c0 = 16 * kk + 2 * q4;
          qa[kk][0] = r0 ? *reinterpret_cast<const uint32_t*>(qb + qr * kD + c0) : 0u;
          qa[kk][1] = r1 ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * kD + c0) : 0u;
          qa[kk][2] = r0 ? *reinterpret_cast<const uint32_t*>(qb + qr * kD + c0 + 8) : 0u;
          qa[kk][3] = r1 ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * kD + c0 + 8) : 0u;
        }
      }
#pragma unroll
      for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      mrow[0] = mrow[1] = -INFINITY;
      lrow[0] = lrow[1] = 0.f;
    }

    // ---------------- one page: tokens t0..t0+15 ----------------
    const uint32_t kb = smem_u32(sm.ring + (size_t)st * kPageBytes);
    const uint32_t vb = kb + 16384;
    float s[2][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s[0][e] = s[1][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + swz(tokK, 2 * kk + (mi & 1)), b0, b1, b2, b3);
      mma_bf16(s[0], qa[kk], b0, b1);
      mma_bf16(s[1], qa[kk], b2, b3);
    }
    // online softmax (base 2)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool valid = (t0 + 8 * nt + 2 * q4 + e) < m.valid;
        s[nt][e] = valid ? s[nt][e] * kScaleLog2 : -INFINITY;
        s[nt][2 + e] = valid ? s[nt][2 + e] * kScaleLog2 : -INFINITY;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(mrow[0], mx0), mn1 = fmaxf(mrow[1], mx1);
    const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(mrow[0] - mn0);
    const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(mrow[1] - mn1);
    float pr[2][4];
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pr[nt][e] = (mn0 == -INFINITY) ? 0.f : exp2f(s[nt][e] - mn0);
        pr[nt][2 + e] = (mn1 == -INFINITY) ? 0.f : exp2f(s[nt][2 + e] - mn1);
        ps0 += pr[nt][e];
        ps1 += pr[nt][2 + e];
      }
    lrow[0] = fmaf(lrow[0], al0, ps0);
    lrow[1] = fmaf(lrow[1], al1, ps1);
    mrow[0] = mn0;
    mrow[1] = mn1;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= al0;
      o[n][1] *= al0;
      o[n][2] *= al1;
      o[n][3] *= al1;
    }
    uint32_t ph_[4], pl_[4];
    ph_[0] = pack_bf16(pr[0][0], pr[0][1]);
    ph_[1] = pack_bf16(pr[0][2], pr[0][3]);
    ph_[2] = pack_bf16(pr[1][0], pr[1][1]);
    ph_[3] = pack_bf16(pr[1][2], pr[1][3]);
    pl_[0] = pack_bf16(pr[0][0] - bf16_lo_f(ph_[0]), pr[0][1] - bf16_hi_f(ph_[0]));
    pl_[1] = pack_bf16(pr[0][2] - bf16_lo_f(ph_[1]), pr[0][3] - bf16_hi_f(ph_[1]));
    pl_[2] = pack_bf16(pr[1][0] - bf16_lo_f(ph_[2]), pr[1][1] - bf16_hi_f(ph_[2]));
    pl_[3] = pack_bf16(pr[1][2] - bf16_lo_f(ph_[3]), pr[1][3] - bf16_hi_f(ph_[3]));
#pragma unroll
    for (int nd2 = 0; nd2 < 8; ++nd2) {
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vb + swz(tokV, 2 * nd2 + (mi >> 1)), v0, v1, v2, v3);
      mma_bf16(o[2 * nd2], ph_, v0, v1);
      mma_bf16(o[2 * nd2], pl_, v0, v1);
      mma_bf16(o[2 * nd2 + 1], ph_, v2, v3);
      mma_bf16(o[2 * nd2 + 1], pl_, v2, v3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
    ++i;
  }
}

// ---------------------------------------------------------------------------
// Retrieve: copy each missing page from the pinned host store into its HBM slot.
// One warp per page, 16-byte loads over the host link, 8 in flight per lane.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) retrieve_kernel(LayerArgs a) {
  const int n = a.counters[0];
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  constexpr int kVec = kPageBytes / 16;  // 2048
  for (int m = gw; m < n; m += nw) {
    const uint4* src = reinterpret_cast<const uint4*>(a.host_store + a.miss_src[m] * kPageElems);
    uint4* dst = reinterpret_cast<uint4*>(a.pool + a.miss_dst[m] * kPageElems);
#pragma unroll 1
    for (int c = 0; c < kVec; c += 32 * 8) {
      uint4 r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) r[u] = __ldcs(src + c + u * 32 + lane);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[c + u * 32 + lane] = r[u];
    }
  }
}

// ---------------------------------------------------------------------------
// Combine: out_g = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c over the
// unit's task partials. One warp per query head, four columns per lane. Also
// closes the step: resets the miss and task counters, advances t.
// ---------------------------------------------------------------------------
__global__ void combine_kernel(LayerArgs a) {
  const int ul = blockIdx.x;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (g < a.G) {
    const int b = ul / a.Hkv, h = ul - b * a.Hkv;
    const int keff = a.keff[ul];
    const int nch = (keff + a.ppt - 1) / a.ppt;
    float4* out = reinterpret_cast<float4*>(a.out + ((int64_t)b * a.Hq + (int64_t)h * a.G + g) * kD);
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c)
      M = fmaxf(M, a.partials[(((int64_t)ul * a.n_chunks + c) * a.G + g) * kPartialStride]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
      for (int c = 0; c < nch; ++c) {
        const float* part = a.partials + (((int64_t)ul * a.n_chunks + c) * a.G + g) * kPartialStride;
        const float sc = exp2f(part[0] - M);
        L = fmaf(sc, part[1], L);
        const float4 v = reinterpret_cast<const float4*>(part + 4)[lane];
        acc.x = fmaf(sc, v.x, acc.x);
        acc.y = fmaf(sc, v.y, acc.y);
        acc.z = fmaf(sc, v.z, acc.z);
        acc.w = fmaf(sc, v.w, acc.w);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    out[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (ul == 0 && threadIdx.x == 0) {
    a.counters[0] = 0;
    a.counters[1] = 0;
    a.counters[2] += 1;
  }
}

}  // namespace

size_t attention_smem_bytes() { return attn_smem_layout(nullptr, nullptr) + 1024; }

cudaError_t attention_configure() {
  return cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attention_smem_bytes());
}

cudaError_t launch_attention(const LayerArgs& a, const CUtensorMap* tmap, int grid, cudaStream_t st) {
  const int n_tasks = a.B * a.Hkv * a.n_chunks;
  attention_kernel<<<grid, kAttnThreads, attention_smem_bytes(), st>>>(*tmap, a, n_tasks);
  return cudaGetLastError();
}

cudaError_t launch_retrieve(const LayerArgs& a, int grid, cudaStream_t st) {
  retrieve_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const LayerArgs& a, cudaStream_t st) {
  combine_kernel<<<a.B * a.Hkv, a.G * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace spin
