// Internal definitions shared by the kernels and the host runtime of the
// SPIN sparse-decode library (sm_103a). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spin {

constexpr int kD = 128;                       // head dim
constexpr int kPart = 64;                     // tokens per partition / page
constexpr int kSeg = 64;                      // entries per second-level segment
constexpr int kBuckets = 64;                  // LRU timestamp buckets
constexpr int kPageElems = 2 * kPart * kD;    // bf16 elements per page (K then V)
constexpr int kPageBytes = kPageElems * 2;    // 32768
constexpr int kPartialStride = 132;           // floats per (task, head) partial: m, l, pad, pad, acc[128]
constexpr int kMaxTopk = 512;
constexpr int kMaxGroup = 16;

// Device error word bits.
enum : uint32_t {
  kErrCapacity = 1u,   // shared segment pool exhausted
  kErrTimeout = 2u,    // a bounded wait ran out
  kErrInternal = 4u,   // an invariant of the page state was found broken
  kErrSelCount = 8u,   // the top-k produced a selection of the wrong size
  kErrSegId = 16u,     // a directory entry held no valid segment id
  kErrIndex = 32u,     // a miss-list, slot or partial index was out of range (access skipped)
};

// Per-layer arguments of the decode-step kernels (passed by value).
struct LayerArgs {
  int32_t layer, B, Hq, Hkv, G, k, cap, D, P_max, n_chunks, ppt, S;
  int32_t ka;                // attention entries per unit: k, plus one for the tail page in tail mode
  int32_t retr_warps;        // retriever warps active per CTA from the start of phase C
  int32_t retr_late;         // further retriever warps that join once the CTA's resident pages are issued
  int32_t mgr_gs;            // threads of one manager group (32, 128, or the CTA's full group)
  int32_t pipe;              // 1: the pipelined kernel (scoring, one manager group and retrieval run at once)
  int32_t retr_split;        // the first retr_split miss-list entries are copied in kRetrChunks pieces
  const int32_t* P_b;        // [B] selectable partitions of request b in this layer (tail mode: complete ones)
  const int32_t* ntok_b;     // [B] tokens held by those partitions
  const int32_t* tail_n;     // [B] tokens in the request's tail page (tail mode), else nullptr
  const uint8_t* part_valid; // [host pages] tokens of each partition's page (variable partitions), else nullptr
  const int32_t* pstride_b;  // [B] host-store pages per KV head of request b (its partition capacity)
  const int32_t* budget_b;   // [B] resident budget per unit of request b (k <= budget <= cap)
  const int64_t* poff_b;     // [B] sum of pstride over earlier requests
  int64_t layer_page_base;   // first page of this layer in the host store / summaries
  int64_t unit_base;         // first global unit of this layer = layer * B * Hkv
  int64_t host_pages;        // pages in the host store (all layers)
  int64_t pool_slots;        // pages in the HBM pool (all units); the tail page of unit u follows at pool_slots + u
  const float* summ;         // [pages][128] fp32 summaries (all layers)
  const uint16_t* host_store;// mapped pinned pages [pages][16384] (device-usable address)
  uint16_t* pool;            // HBM pages [units * cap][16384]
  int32_t* dir;              // [units][D] segment id or -1
  int32_t* seg;              // [S][64] slot or -1
  int32_t* seg_live;         // [S] live entries
  uint32_t* seg_bitmap;      // [ceil(S/32)] 1 = segment in use
  int32_t* slot_part;        // [units][cap]
  int32_t* last_use;         // [units][cap]
  float* scores;             // [2][U_l][P_max]: step t writes buffer t & 1 (kScoreEmpty where not written yet)
  int32_t* sel;              // [U_l][k]
  int32_t* sel_slot;         // [U_l][k] local slot
  uint8_t* sel_hit;          // [U_l][k]
  int32_t* keff;             // [U_l]
  int32_t* unit_info;        // [U_l][8]
  int64_t* miss_src;         // [U_l * k] host page index of each miss (miss list, append order)
  int64_t* miss_dst;         // [U_l * k] pool slot index of each miss
  int32_t* miss_att;         // [U_l * k] ul * ka + attention position of each miss
  int32_t* miss_valid;       // [U_l * k] valid tokens of each miss's page
  int32_t* ready;            // [U_l * k] per miss-list entry: step tag once its page is in HBM
  uint32_t* ready_cnt;       // [retr_split] pieces of a split entry copied so far (never reset: grows by kRetrChunks a step)
  int32_t* miss_tag;         // [U_l * k] per miss-list entry: step tag once the entry is written
  int32_t* unit_rows;        // [U_l] partitions scored so far in this step (reset by the unit's manager)
  int32_t* unit_ready;       // [U_l] step tag once the unit is managed
  int32_t* hist12;           // [U_l][4096] wide units only (else nullptr): count of keys per top-12-bit value,
                             // filled while scoring, cleared by the unit's manager
  int32_t* att_slot;         // [U_l][ka] slots in attention order: hits, the tail (slot == cap), then misses
  int32_t* att_valid;        // [U_l][ka] valid tokens of those pages
  int32_t* n_hit;            // [U_l] resident pages of the step, tail included (pages [0, n_hit) of att_slot)
  int32_t* counters;         // [kNumCtr]: see kCtr*
  float* partials;           // hits [U_l][n_chunks][G][132], then misses [U_l][ka][G][132]
  unsigned long long* stats; // [8] device counters
  unsigned long long* timeline; // [5] globaltimer stamps of this call (stage timing), else nullptr
  uint32_t* err;             // device error word
  const uint16_t* q;         // [B][Hq][128] bf16 (HBM): the query rows the attention stages through TMA
  const uint16_t* q_src;     // the step's queries: q itself, or pinned host memory (zero copy), in which
                             // case the kernel first copies every unit's rows into q (counted in kCtrQStaged)
  float* out;                // [B][Hq][128] fp32 (device)
};

// Host page index of partition p of (b, h) in the layer described by a (also the
// row of its summary).
__device__ inline int64_t host_page_index(const LayerArgs& a, int b, int h, int64_t p) {
  return a.layer_page_base + (int64_t)a.Hkv * a.poff_b[b] + (int64_t)h * a.pstride_b[b] + p;
}

// Per-layer device counters.
enum : int {
  kCtrMiss = 0,      // miss-list entries allocated in this step
  kCtrTaskHits = 1,  // resident-page tasks claimed
  kCtrTaskMisses = 2,// retrieved pages claimed by producers
  kCtrStep = 3,      // the layer's step t
  kCtrRetrieve = 4,  // miss-list entries claimed by retrievers
  kCtrArrive = 5,    // CTAs done with their pages (grows by the grid size every step)
  kCtrManage = 6,    // units claimed by manager groups
  kCtrManaged = 7,   // units managed and published
  kCtrQStaged = 8,   // units whose query rows were copied from host memory into q (zero-copy queries)
  kNumCtr = 9
};

// Stage stamps of one timed decode-step call (globaltimer ns): first CTA start (stored
// inverted, so that atomicMax keeps the minimum), last CTA done scoring, last unit
// managed, last CTA done with its pages, last combine done.
enum : int { kTlStart = 0, kTlScored = 1, kTlManaged = 2, kTlPages = 3, kTlEnd = 4, kTlSlots = 8 };

// Bit pattern of a score slot not yet written in this step (a signalling NaN the score
// arithmetic never produces): the pipelined kernel's managers wait until none is left.
constexpr uint32_t kScoreEmpty = 0x7FBFFFFFu;

// Pieces of a split miss-list entry (its 32 KB page copied by kRetrChunks warps at once).
// The first entries of a step are split so that a step with few misses still has every
// retriever warp loading; the rest are copied a page per warp.
constexpr int kRetrChunks = 4;

// Device stats slots.
enum : int {
  kStatHits = 0, kStatMisses = 1, kStatEvictions = 2, kStatLruRounds = 3, kStatSelected = 4, kStatFlushes = 5
};

// ---------------------------------------------------------------------------
// Launchers (defined in the kernel translation units).
// ---------------------------------------------------------------------------
cudaError_t launch_summarize_offload(const uint16_t* k, const uint16_t* v, int64_t head_stride, int32_t kv_heads,
                                     int64_t tok0, int64_t ntok_chunk, int64_t ntok_total, float* summ_unit0,
                                     uint16_t* host_unit0, int64_t unit_pages, cudaStream_t st);
cudaError_t launch_gather_offload(const uint16_t* k, const uint16_t* v, int64_t n_tokens, int32_t kv_heads,
                                  const int32_t* order, const int32_t* starts, int32_t n_parts, float* summ_unit0,
                                  uint16_t* host_unit0, int64_t unit_pages, uint8_t* valid_unit0, cudaStream_t st);
cudaError_t launch_warm_store(const void* store, int64_t bytes, int64_t stride, uint32_t* sink, int sm_count,
                              cudaStream_t st);
// KV append of one token per request of the layer (tail mode).
cudaError_t launch_append(const LayerArgs& a, const uint16_t* k_new, const uint16_t* v_new, int32_t* P_b,
                          int32_t* ntok_b, int32_t* tail_n, cudaStream_t st);
// Writes one int on the device, ordered on the stream (request tables).
cudaError_t launch_set_int(int32_t* p, int32_t v, cudaStream_t st);
// Sets the request's layer state (partitions, their tokens, tail tokens) on the device.
cudaError_t launch_set_request(int32_t* P_b, int32_t* ntok_b, int32_t* tail_n, int32_t P, int32_t ntok,
                               int32_t tail, cudaStream_t st);
// The whole decode step of one layer in one cooperative persistent launch (one CTA per SM).
cudaError_t launch_decode_step(const LayerArgs& a, const CUtensorMap* tmap, int grid, cudaStream_t st);
cudaError_t step_configure(const LayerArgs& a);
size_t step_smem_bytes(const LayerArgs& a);   // dynamic shared memory of that launch
size_t step_ring_bytes();                     // the ring of phase C (the manager groups share its bytes)
size_t mgr_group_bytes(int gs, const LayerArgs& a);  // shared memory of one manager group of gs threads
int step_threads(int G);                      // threads per CTA
int step_full_group(int G);                   // the largest manager group (all warps of a CTA's roles)
cudaError_t launch_resolve_all(const LayerArgs& a, int32_t* resolve, int32_t* live_segs, cudaStream_t st);
// Fills n 32-bit words with v, ordered on the stream.
cudaError_t launch_fill_u32(uint32_t* p, uint32_t v, int64_t n, cudaStream_t st);

}  // namespace spin
