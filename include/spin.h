/*
 * spin.h — C ABI of the GB300 (sm_103a) SPIN sparse-decode data path.
 *
 * The library implements, per decode step and per layer, the data path of SPIN
 * ("Unifying Sparse Attention with Hierarchical Memory for Scalable Long-Context
 * LLM Serving", arXiv 2604.26837) over a page-based, per-KV-head KV store split
 * between HBM and pinned host memory:
 *   Select   score every partition summary against the query, per-KV-head top-k;
 *   Resolve  look the selected partitions up in a two-level page table;
 *   Evict    bucketed LRU when the free pages do not cover the misses;
 *   Retrieve copy the missing pages host -> HBM;
 *   Attend   exact softmax attention over the selected tokens only.
 * Page citations: m.x-techcon.com "吞吐量提升5.66倍！微软、港中大等Spin框架如何统一稀疏注意力
 * 与分级内存…" (below [XT]), section "Spin的核心设计" 1-3, Figures 3, 5, 6; and
 * gist.science/pt "Unifying Sparse Attention with Hierarchical Memory…" (below [GS]),
 * section 2 A-C.
 *
 * Fixed geometry: head_dim 128; a page holds one partition of one KV head: 64
 * consecutive tokens, or, in a context with max_partitions > 0, a group of 1 to 64
 * tokens that the caller's Index chose; second-level segment = 64
 * directory-adjacent partitions; 64 LRU buckets. A page is stored as K[64][128]
 * then V[64][128], bf16 (uint16 bits), token-major, zero padded past the last
 * valid token: 32768 bytes.
 *
 * Units. A unit is one (request b, layer l, KV head h). Query head hq belongs to
 * KV head hq / G with G = q_heads / kv_heads (grouped-query attention).
 *
 * Ownership. The caller owns every pointer it passes (queries, outputs, KV
 * sources, streams, host buffers of the debug calls). The library owns, from
 * spin_create to spin_destroy: the HBM page pool, the two-level tables, the
 * partition summaries, the pinned host page store, per-layer scratch, its
 * internal streams and events. KV sources passed to spin_index_offload are
 * copied and may be freed when that call's stream work has completed; those
 * passed to spin_index_offload_parts may be freed when the call returns.
 *
 * Errors. Every int-returning call returns a spin_status. No call throws, traps
 * or aborts. Kernels report device-side conditions (pool exhausted, a bounded
 * wait that ran out) through a device error word that the next synchronising
 * call (spin_stats, spin_debug_*) turns into a status; after a device error the
 * context keeps returning that status. spin_last_error(ctx) gives a message
 * (spin_last_error(NULL) the message of the last failed spin_create).
 *
 * Threading. A context may be used from one host thread at a time. Decode
 * steps of different layers may be enqueued on different streams; the steps of
 * one layer must be ordered on one stream.
 */
#ifndef SPIN_H_
#define SPIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPIN_HEAD_DIM 128
#define SPIN_PART_TOKENS 64
#define SPIN_SEG_ENTRIES 64
#define SPIN_LRU_BUCKETS 64
#define SPIN_PAGE_BYTES 32768
#define SPIN_MAX_GROUP 16

typedef struct spin_ctx spin_ctx;
typedef void* spin_stream_t; /* a cudaStream_t; NULL = the legacy default stream */

typedef enum spin_status {
  SPIN_OK = 0,
  SPIN_ERR_INVALID = 1,  /* bad argument or configuration; nothing was enqueued */
  SPIN_ERR_CUDA = 2,     /* a CUDA runtime call failed (no device, launch failure …) */
  SPIN_ERR_OOM = 3,      /* a device or pinned host allocation failed */
  SPIN_ERR_CAPACITY = 4, /* the shared segment pool ran out during a step */
  SPIN_ERR_TIMEOUT = 5,  /* a bounded device-side wait ran out */
  SPIN_ERR_STATE = 6     /* call out of order (e.g. decode before every request was offloaded) */
} spin_status;

typedef enum spin_flags {
  SPIN_FLAG_STAGE_TIMING = 1u << 0, /* record CUDA events around every stage; read via spin_stats */
  SPIN_FLAG_TIER_SPLIT = 1u << 2,   /* tier-split metadata ([XT] §3, [GS] §2C): the second-level segment
                                       entries live in pinned host memory; the directory, the segments'
                                       live counts and the allocation bitmap stay in HBM */
  SPIN_FLAG_HOST_HUGEPAGES = 1u << 3, /* allocate the pinned host page store as an anonymous mapping aligned to
                                        and advised for transparent huge pages, registered with
                                        cudaHostRegister, instead of with cudaHostAlloc (falls back to
                                        cudaHostAlloc when mapping or registering fails) */
  SPIN_FLAG_PHASED = 1u << 4,       /* run every decode step as phases over the whole grid (score, then
                                       select + manage, then retrieve + attend) instead of the pipelined
                                       kernel that units of at most 4096 partitions and groups of at most
                                       8 query heads otherwise get (scoring, managing and retrieval at once);
                                       the results are the same */
  SPIN_FLAG_TEST_FAIL_PINNED = 1u << 16, /* test hook: the pinned host allocation reports failure */
  SPIN_FLAG_TEST_NO_RETRIEVE = 1u << 17  /* test hook: no page is retrieved, so the bounded wait for the
                                            first missing page runs out and the step reports SPIN_ERR_TIMEOUT */
} spin_flags;

/* Configuration of one context. All counts are per context. */
typedef struct spin_config {
  int32_t batch;             /* 1 <= B <= 16384 requests */
  int32_t layers;            /* L >= 1 */
  int32_t q_heads;           /* Hq; Hq % Hkv == 0 and Hq / Hkv <= SPIN_MAX_GROUP */
  int32_t kv_heads;          /* Hkv >= 1 */
  int32_t head_dim;          /* must be 128 */
  int32_t part_tokens;       /* must be 64 */
  int32_t topk;              /* k >= 1 partitions selected per unit per step, <= 512 */
  int32_t buf_mult;          /* resident capacity per unit = buf_mult * topk pages (mandatory + buffer), >= 1 */
  const int64_t* ctx_len;    /* [batch] tokens per request, >= 0 (host pointer, copied) */
  int32_t seg_entries;       /* 0 or 64 */
  int64_t seg_pool_segments; /* segments in the shared second-level pool; 0 = enough for any page state */
  int32_t device;            /* CUDA device ordinal */
  uint32_t flags;            /* spin_flags */
  int32_t append_tokens;     /* 0: fixed context. > 0: KV-append (tail) mode, each request may grow by up to
                                this many tokens through spin_append_kv. In tail mode only complete 64-token
                                partitions are selectable; the newest ctx % 64 tokens form the request's tail,
                                which every decode step attends in full, and a tail that reaches 64 tokens is
                                summarised, offloaded and becomes the next partition. */
  int32_t max_partitions;    /* 0: fixed partitions of 64 consecutive tokens (the last may be short).
                                > 0: variable partitions ([XT] §1; [GS] §2A): each request may hold up to this
                                many partitions per KV head, each of 1 to 64 tokens in a page of its own, as
                                spin_index_offload_parts groups them; spin_index_offload is then refused.
                                Needs append_tokens == 0, max_partitions <= 2^20 and
                                ceil(ctx_len[b] / 64) <= max_partitions for every request. */
  int64_t max_context;       /* the logical context capacity of a request in tokens ([XT] §3: a flat table is
                                sized for the worst-case logical space, max batch x max context x layers x
                                heads, where the two-level table grows with the resident pages). 0 = the
                                longest ctx_len[b] + append_tokens. Sizes the static first level (the
                                directory) and the flat table spin_stats reports for comparison; must be >=
                                every ctx_len[b] + append_tokens and <= 2^21. */
} spin_config;

/* Counters since spin_create. */
typedef struct spin_stats_t {
  int64_t steps;             /* completed decode-step calls (one per layer) */
  int64_t hits;              /* selected pages found resident */
  int64_t misses;            /* selected pages retrieved from host */
  int64_t evictions;         /* pages reclaimed by the bucketed LRU */
  int64_t lru_rounds;        /* unit-steps that ran the LRU */
  int64_t retrieved_bytes;   /* misses * SPIN_PAGE_BYTES */
  int64_t selected_bytes;    /* selected pages * SPIN_PAGE_BYTES (bytes attention read) */
  int64_t live_segments;     /* second-level segments currently allocated */
  int64_t pool_segments;     /* segments in the shared pool */
  int64_t metadata_bytes;    /* HBM bytes of the page metadata: directory + segment pool (unless tier
                                split) + live counts + bitmap + per-page state */
  int64_t flat_table_bytes;  /* HBM bytes of the flat table of the worst-case logical space ([XT] §3): one
                                int32 entry per (request, layer, KV head, partition of max_context), plus the
                                same per-page state */
  int64_t hbm_pool_bytes;    /* HBM page pool */
  int64_t host_store_bytes;  /* pinned host page store */
  int64_t summary_bytes;     /* HBM partition summaries (fp32) */
  int64_t timed_calls;       /* decode calls with stage timing */
  /* Summed stage times of the timed calls (SPIN_FLAG_STAGE_TIMING), milliseconds. A decode
     step is one kernel whose phases overlap across SMs; the stages are consecutive spans of
     its critical path, from in-kernel timer stamps: */
  double ms_score;           /* first CTA starts -> every partition scored */
  double ms_manage;          /* -> the last unit's top-k and page manager done (misses published) */
  double ms_pages;           /* -> the last page retrieved and attended (retrieval overlaps attention) */
  double ms_combine;         /* -> the last output row combined */
  double ms_kernel;          /* the whole kernel, from CUDA events around it */
  uint32_t device_error;     /* raw device error word (0 = none) */
  int64_t appended_tokens;   /* tokens appended through spin_append_kv (all layers, all requests) */
  int64_t tail_flushes;      /* tails that filled and became partitions (per layer and request) */
} spin_stats_t;

/* Host-side view filled by spin_debug_export; any pointer may be NULL. Shapes use
 * U = batch * kv_heads units of the layer (unit ul = b * kv_heads + h), k = topk,
 * cap = buf_mult * topk, Pmax = the largest partition count of any request (in tail
 * mode: the largest count a request can reach, ceil((ctx_len + append_tokens) / 64);
 * with variable partitions: max_partitions). */
typedef struct spin_state_view {
  int32_t* keff;       /* [U] partitions selected in the last step = min(k, P_b) */
  int32_t* sel;        /* [U][k] selected partitions of the last step, ascending, -1 padded */
  int32_t* sel_slot;   /* [U][k] slot (0..cap-1) holding each selected partition */
  uint8_t* sel_hit;    /* [U][k] 1 when the partition was resident before the step */
  int32_t* slot_part;  /* [U][cap] partition held by each slot, -1 = free */
  int32_t* last_use;   /* [U][cap] step of each slot's last use */
  int32_t* resolve;    /* [U][Pmax] slot found by the two-level walk, -1 = not resident */
  int32_t* live_segs;  /* [U] second-level segments the unit holds */
  int32_t* unit_info;  /* [U][8] last step: hits, misses, resident before, demand, cutoff (-1 none), evicted, step, 0 */
  float* scores;       /* [U][Pmax] fp32 scores of the last step (entries >= P_b undefined) */
} spin_state_view;

/* Create a context ([XT] §1 and Figure 3: the state the five operations share; [XT] §2
 * and [GS] §2B: per-head mandatory + buffer pages, cap = buf_mult * topk; [XT] §3 and
 * Figure 6: the two-level table): validates cfg, allocates the pinned host page store
 * (sum_b S_b * L * Hkv pages, S_b = ceil(ctx_len[b]/64); ceil((ctx_len[b] +
 * append_tokens)/64) in tail mode; max_partitions with variable partitions), the
 * HBM page pool (B*L*Hkv*cap pages, plus one tail page per unit in tail mode), the
 * summaries, the two-level tables (directory [units][ceil(Pmax/64)], shared
 * segment pool) and per-layer scratch, on cfg->device. Every page starts on the
 * host and the GPU holds nothing. *out is set only on SPIN_OK. */
int spin_create(const spin_config* cfg, spin_ctx** out);

/* Index + Offload ([XT] §1, Fig 3; [GS] §2A) of request b in `layer`:
 * k, v: bf16 [kv_heads][n_tokens][128], row-major; n_tokens must equal
 * cfg->ctx_len[b]. src_is_host != 0: k and v are host pointers (pinned or
 * pageable); 0: device pointers on the context's device. Computes the fp32 mean
 * key of every partition (the partition summary) and writes every page into the
 * pinned host store. Asynchronous on `stream`. */
int spin_index_offload(spin_ctx* ctx, int32_t b, int32_t layer, const uint16_t* k, const uint16_t* v,
                       int64_t n_tokens, int32_t src_is_host, spin_stream_t stream);

/* Index + Offload of variable partitions ([XT] §1: a partition is the unit of selection and
 * retrieval, either a fixed-size block or a cluster found dynamically; [GS] §2A: blocks,
 * clusters and tokens all map onto one page substrate). The grouping is the algorithm's Index
 * and comes from the caller, as host arrays:
 *   order  int32 [kv_heads][n_tokens]: for each head, a permutation of 0 .. n_tokens-1;
 *   starts int32 [kv_heads][n_parts + 1]: starts[h][0] = 0, starts[h][n_parts] = n_tokens and
 *          1 <= starts[h][p+1] - starts[h][p] <= 64.
 * Partition p of head h holds the tokens order[h][starts[h][p]] .. order[h][starts[h][p+1] - 1];
 * they are written in that order from row 0 of the partition's page (zero padded), the page
 * records its token count, and the summary is their fp32 mean key. Selection, the page
 * manager, retrieval and attention then work on these partitions as on fixed ones; attention
 * reads each page's own token count. k, v: bf16 [kv_heads][n_tokens][128], host or device
 * as in spin_index_offload; n_tokens == ctx_len[b]; 1 <= n_parts <= max_partitions, or 0
 * when n_tokens == 0; every head of the request has n_parts partitions. Needs a context
 * created with max_partitions > 0 (else SPIN_ERR_STATE). A grouping that breaks these rules
 * returns SPIN_ERR_INVALID with nothing enqueued. Synchronous: returns once the work
 * enqueued on `stream` has finished, so the host arrays may be reused at once. */
int spin_index_offload_parts(spin_ctx* ctx, int32_t b, int32_t layer, const uint16_t* k, const uint16_t* v,
                             int64_t n_tokens, const int32_t* order, const int32_t* starts, int32_t n_parts,
                             int32_t src_is_host, spin_stream_t stream);

/* KV append ([XT] §1, Figure 3: Index and Offload also run for the tokens decode
 * produces; the pages leave the mechanics open). Appends ONE token to every request
 * of `layer`: k_new, v_new are device bf16 [batch][kv_heads][128], 16-byte aligned.
 * The token goes into the request's tail page in HBM (one per unit); when that tail
 * holds 64 tokens it is summarised (fp32 mean key), written into the pinned host
 * store as the request's next partition and emptied, all on the device. Needs a
 * context created with append_tokens > 0 (else SPIN_ERR_STATE) whose requests of
 * `layer` have all been offloaded; a request that would grow past
 * ctx_len[b] + append_tokens tokens returns SPIN_ERR_CAPACITY and nothing is
 * enqueued. Asynchronous on `stream`; the appends and decode steps of one layer must
 * be ordered on one stream. In a decode loop the token of step t is appended before
 * that step's spin_decode_step, which then attends it. */
int spin_append_kv(spin_ctx* ctx, int32_t layer, const uint16_t* k_new, const uint16_t* v_new, spin_stream_t stream);

/* Buffer elasticity ([XT] §2: the buffer part of a request's pages is resized by
 * the scheduler with load; [GS] §2B). Sets the resident budget of request b to
 * `pages` per unit (every layer and KV head of the request), topk <= pages <=
 * buf_mult * topk; spin_create starts every request at buf_mult * topk. The
 * manager counts free pages against the budget, so after a shrink the next step's
 * demand includes the excess and the bucketed LRU reclaims down to the budget;
 * after a growth the extra pages fill on later misses. Takes effect for the decode
 * steps enqueued on `stream` after it (asynchronous; order it on the stream of the
 * steps). Returns SPIN_ERR_INVALID for b or pages out of range. */
int spin_set_buffer(spin_ctx* ctx, int32_t b, int32_t pages, spin_stream_t stream);

/* One decode step of one layer for the whole batch ([XT] §2 and Fig 5 steps 1-4,
 * §3; [GS] §2B-C). q: device bf16 [batch][q_heads][128]; out: device fp32
 * [batch][q_heads][128] = softmax(q K_sel^T / sqrt(128)) V_sel over the tokens of
 * the k selected partitions of the query head's KV head, plus, in tail mode, the
 * request's tail tokens (zeros for an empty request). Asynchronous on `stream`; the
 * layer's step counter t advances by one per call. Requires every request of `layer`
 * to have been offloaded.
 * The first step after any spin_index_offload or spin_index_offload_parts call (of
 * any layer) first enqueues one read pass over the whole host store: a 4-byte load
 * every host page (at most every 32 KiB). The GPU translates each host page's
 * address on its first read, and those translations resolve slowly; the pass pays
 * for them once, so the steps' retrieval does not. */
int spin_decode_step(spin_ctx* ctx, int32_t layer, const uint16_t* q, float* out, spin_stream_t stream);

/* The same step with host buffers: q_host [batch][q_heads][128] bf16 and
 * out_host [batch][q_heads][128] fp32. Pinned, device-mapped buffers (cudaHostAlloc'd or
 * registered) are used in place: the kernel copies q_host (8-byte aligned) into device
 * memory at its start and writes out_host (16-byte aligned), both over the host link.
 * Other buffers go through HBM with host<->device copies enqueued on `stream` around
 * the step. out_host is valid once the
 * stream has reached the end of the step, and neither buffer may be reused before then. */
int spin_decode_step_host(spin_ctx* ctx, int32_t layer, const uint16_t* q_host, float* out_host,
                          spin_stream_t stream);

/* Synchronises the context's device work and fills *out: hits, misses, evictions and
 * LRU rounds of the bucketed LRU ([XT] §2 and Figure 5; [GS] §2B), bytes selected and
 * retrieved, and the metadata bytes of the two-level table next to a flat table of the
 * worst-case logical space ([XT] §3 and Figure 6, and its "性能评估" metadata figure).
 * Returns the device error status if a kernel reported one. */
int spin_stats(spin_ctx* ctx, spin_stats_t* out);

/* Synchronises, then copies the page state and last-step selection of `layer`
 * into the caller's host buffers (parity testing and inspection). */
int spin_debug_export(spin_ctx* ctx, int32_t layer, spin_state_view* view);

/* Synchronises, then copies the 32768-byte HBM page in slot `slot` of unit
 * (layer, b, h) to dst (host). In tail mode slot == buf_mult * topk names the
 * unit's tail page. */
int spin_debug_read_page(spin_ctx* ctx, int32_t layer, int32_t b, int32_t h, int32_t slot, uint16_t* dst);

/* Synchronises, then copies the fp32 summaries [P_b][128] of unit (layer, b, h) to dst (host);
 * P_b = the request's current partition count (in tail mode: its complete partitions). */
int spin_debug_summaries(spin_ctx* ctx, int32_t layer, int32_t b, int32_t h, float* dst);

/* Allocation-free Select, for callers that cannot allocate device memory (code
 * that runs while a CUDA graph is being captured, engines whose allocator owns all
 * device memory, hosts that forbid run-time allocation); every other entry point
 * needs the buffers spin_create allocates. No counterpart on the SPIN pages: this
 * is the decode step's Select (fp32 score = (sum of the group's queries) . summary,
 * per-unit top-k, equal scores to the lower index, ascending output) without the
 * context, computed by the same device code as the decode step. It calls no
 * allocator of any kind.
 *   summ  device fp32 [units][parts][128] partition summaries (16-byte aligned)
 *   q     device bf16 [units][group][128] queries of each unit's query heads (8-byte aligned)
 *   sel   device int32 [units][topk] output: selected partitions, ascending, -1 padded
 *         when parts < topk
 * Limits: units * parts <= SPIN_NOALLOC_MAX_SCORES, parts <= 32768, group <= 16,
 * topk <= 512; larger sizes return SPIN_ERR_INVALID. The scores live in one static
 * device array of SPIN_NOALLOC_MAX_SCORES floats (4 MiB). CUDA reserves it when the
 * library's kernels are loaded into a context: with lazy module loading (the CUDA
 * default) that happens on the first call in each context, so a caller whose pool
 * will claim the device, or that will capture a graph, makes one call first (or sets
 * CUDA_MODULE_LOADING=EAGER). The context holds the array until it is destroyed. All
 * calls share it and it keeps the last call's contents; calls whose work overlaps on
 * the GPU (different streams, different host threads on one device) race on it and
 * must be serialised by the caller. Each call looks the array's device address up in
 * the current context. A CUDA error left pending by earlier work is reported as
 * SPIN_ERR_CUDA without launching anything. Asynchronous on `stream`; on failure
 * spin_last_error(NULL) gives the reason. */
#define SPIN_NOALLOC_MAX_SCORES (1 << 20)
int spin_select_noalloc(const float* summ, const uint16_t* q, int32_t units, int32_t parts, int32_t group,
                        int32_t topk, int32_t* sel, spin_stream_t stream);

/* Host-link probe ([XT] "理想与现实的差距", Figure 1: the pages measure against an
 * envelope with retrieval at the link's peak). Streams `bytes` of the pinned,
 * device-mapped host buffer `host` (16-byte aligned) through the SMs with 16-byte
 * zero-copy loads, ctas_per_sm (1..4) CTAs of 512 threads per SM, twice on `stream`
 * (the first pass resolves the pages' address translations), and writes the second
 * pass's rate in GB/s (1e9 bytes/s) to *gbs. Synchronises `stream`. Uses the current
 * device; allocates nothing. SPIN_ERR_INVALID for a buffer that is not pinned host
 * memory mapped for the device. */
int spin_measure_host_read(const void* host, int64_t bytes, int32_t ctas_per_sm, double* gbs, spin_stream_t stream);

/* Releases everything the context owns (synchronises first). NULL is a no-op. */
void spin_destroy(spin_ctx* ctx);

/* Message of the last failure on ctx (or of the last failed spin_create when
 * ctx is NULL). The string lives until the next call on the same context. */
const char* spin_last_error(const spin_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* SPIN_H_ */
