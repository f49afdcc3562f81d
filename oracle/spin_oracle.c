/*
 * SPIN decode-step ORACLE: plain, slow, double-precision CPU restatement of the
 * per-decode-step sparse-attention data path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library. The product path (the CUDA
 * library) shares no code with it and never calls it.
 *
 * Sources. The method is described on four web pages about
 * "Unifying Sparse Attention with Hierarchical Memory for Scalable Long-Context
 * LLM Serving" (SPIN, arXiv 2604.26837). Citations below use:
 *   [XT] m.x-techcon.com, "吞吐量提升5.66倍！微软、港中大等Spin框架如何统一稀疏注意力与
 *        分级内存，让稀疏注意力算法真正高效落地", section "Spin的核心设计" with its
 *        sub-sections 1 (统一的分区抽象), 2 (动态的、局部性感知的KV管理),
 *        3 (分级元数据组织) and Figures 3, 5, 6;
 *   [GS] gist.science/pt, "Unifying Sparse Attention with Hierarchical Memory for
 *        Scalable Long-Context LLM Serving", section 2 (Metodologia) A, B, C.
 * The pages give no formulas. Where they leave a rule open this file takes the
 * plainest reading and says so ("reading:").
 *
 * Layout conventions (shared with the tests, not with the CUDA code):
 *   a partition = a page of one KV head (reading of [XT] §1 "分区" + [GS] §2B
 *   "Páginas Físicas por Cabeça"): 64 consecutive tokens, or, for variable
 *   partitions, a group of 1 to 64 tokens given as a token order and
 *   boundaries; head_dim = 128; a page in page format is K[64][128] then
 *   V[64][128], bf16, token-major, zero padded past the last valid token.
 *
 * Parity pins: every function here is pinned by tests/oracle_pins.py, run by
 * tests/test_oracle_pins.py and tests/test_oracle_properties.py (dense-attention
 * identity, brute-force top-k, LRU invariants, page-table round trip,
 * closed-form summaries, byte-equal retrieve, variable-partition means).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OD 128            /* head dim */
#define OPART 64          /* tokens per partition / page */
#define OSEG 64           /* entries per second-level segment */
#define OBUCKETS 64       /* LRU timestamp buckets */
#define OPAGE_ELEMS (2 * OPART * OD)

static double bf(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Index + Offload ([XT] §1 / Fig 3: Index organises KV into partitions and    */
/* produces summaries; Offload puts the partitions into CPU memory).           */
/* reading: the summary of a partition is its mean key.                        */
/* ------------------------------------------------------------------------- */

/* summ[p][i] = (1/n_p) * sum over the n_p valid tokens t of partition p of K[t][i] */
void oracle_index(const uint16_t* k, int64_t ntok, double* summ) {
  int64_t P = (ntok + OPART - 1) / OPART;
  for (int64_t p = 0; p < P; ++p) {
    int64_t t0 = p * OPART;
    int64_t t1 = t0 + OPART < ntok ? t0 + OPART : ntok;
    for (int i = 0; i < OD; ++i) {
      double s = 0.0;
      for (int64_t t = t0; t < t1; ++t) s += bf(k[t * OD + i]);
      summ[p * OD + i] = s / (double)(t1 - t0);
    }
  }
}

/* Offload: page-format copy of K, V [ntok][128] into host pages [P][2][64][128]. */
void oracle_offload(const uint16_t* k, const uint16_t* v, int64_t ntok, uint16_t* pages) {
  int64_t P = (ntok + OPART - 1) / OPART;
  memset(pages, 0, sizeof(uint16_t) * (size_t)(P * OPAGE_ELEMS));
  for (int64_t t = 0; t < ntok; ++t) {
    int64_t p = t / OPART, r = t % OPART;
    memcpy(pages + p * OPAGE_ELEMS + r * OD, k + t * OD, OD * sizeof(uint16_t));
    memcpy(pages + p * OPAGE_ELEMS + OPART * OD + r * OD, v + t * OD, OD * sizeof(uint16_t));
  }
}

/* ------------------------------------------------------------------------- */
/* Variable partitions ([XT] §1: a partition is a group of tokens that is the  */
/* unit of selection and retrieval, either a fixed-size block or a cluster     */
/* found dynamically; [GS] §2A: blocks, clusters and tokens are all mapped      */
/* onto one page-based KV substrate). The grouping is the algorithm's Index;   */
/* here it arrives as a token order and partition boundaries: partition p holds */
/* tokens order[starts[p]] .. order[starts[p+1] - 1], 1 to 64 of them.          */
/* reading: each partition occupies one page, its tokens in that order from row */
/* 0, zero padded; its summary is the mean key of its tokens.                   */
/* ------------------------------------------------------------------------- */
void oracle_index_parts(const uint16_t* k, const int32_t* order, const int32_t* starts, int32_t P, double* summ) {
  for (int32_t p = 0; p < P; ++p) {
    const int32_t j0 = starts[p], j1 = starts[p + 1];
    for (int i = 0; i < OD; ++i) {
      double s = 0.0;
      for (int32_t j = j0; j < j1; ++j) s += bf(k[(int64_t)order[j] * OD + i]);
      summ[(int64_t)p * OD + i] = s / (double)(j1 - j0);
    }
  }
}

void oracle_offload_parts(const uint16_t* k, const uint16_t* v, const int32_t* order, const int32_t* starts,
                          int32_t P, uint16_t* pages) {
  memset(pages, 0, sizeof(uint16_t) * (size_t)((int64_t)P * OPAGE_ELEMS));
  for (int32_t p = 0; p < P; ++p)
    for (int32_t j = starts[p]; j < starts[p + 1]; ++j) {
      const int64_t t = order[j], r = j - starts[p];
      memcpy(pages + (int64_t)p * OPAGE_ELEMS + r * OD, k + t * OD, OD * sizeof(uint16_t));
      memcpy(pages + (int64_t)p * OPAGE_ELEMS + OPART * OD + r * OD, v + t * OD, OD * sizeof(uint16_t));
    }
}

/* ------------------------------------------------------------------------- */
/* Select ([XT] §1 / Fig 3: Select picks the critical partitions for the       */
/* query; [GS] §2A). reading: score_p = sum over the G query heads of the GQA  */
/* group of q_g . summary_p; take the k highest scores, equal scores going to  */
/* the lower partition index; return the chosen indices in ascending order.   */
/* ------------------------------------------------------------------------- */

void oracle_scores(const double* summ, int64_t P, const uint16_t* q, int32_t G, double* sc) {
  for (int64_t p = 0; p < P; ++p) {
    double s = 0.0;
    for (int g = 0; g < G; ++g)
      for (int i = 0; i < OD; ++i) s += bf(q[g * OD + i]) * summ[p * OD + i];
    sc[p] = s;
  }
}

typedef struct {
  double s;
  int32_t p;
} scored;

/* rank order: higher score first; equal scores: lower index first */
static int rank_cmp(const void* a, const void* b) {
  const scored* x = (const scored*)a;
  const scored* y = (const scored*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->p > y->p) - (x->p < y->p);
}

static int int_cmp(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Returns k_eff = min(k, P); sel[0..k_eff) ascending. */
int32_t oracle_topk(const double* sc, int64_t P, int32_t k, int32_t* sel) {
  int32_t keff = (int64_t)k < P ? k : (int32_t)P;
  scored* r = (scored*)malloc(sizeof(scored) * (size_t)(P > 0 ? P : 1));
  for (int64_t p = 0; p < P; ++p) {
    r[p].s = sc[p];
    r[p].p = (int32_t)p;
  }
  qsort(r, (size_t)P, sizeof(scored), rank_cmp);
  for (int32_t j = 0; j < keff; ++j) sel[j] = r[j].p;
  qsort(sel, (size_t)keff, sizeof(int32_t), int_cmp);
  free(r);
  return keff;
}

/* ------------------------------------------------------------------------- */
/* Per-unit page state. A unit is one (request, layer, KV head): physical      */
/* pages are per head ([GS] §2B "Páginas Físicas por Cabeça").                  */
/*                                                                           */
/* Two-level table ([XT] §3 / Fig 6; [GS] §2C): a small static top-level        */
/* directory whose entries point to second-level segments; a segment is taken  */
/* from a pool only when a page of its range gets a physical page, and returned */
/* when its last page leaves. reading: a segment covers 64 consecutive          */
/* partitions; entry = resident slot or -1.                                    */
/* ------------------------------------------------------------------------- */
typedef struct oracle_unit {
  int32_t P;           /* partitions of the unit (in tail mode: the complete ones) */
  int32_t P_cap;       /* partitions the unit may grow to (tail mode), else P */
  int32_t ntok;        /* valid tokens (last partition may be short) */
  int32_t* part_n;     /* [P] tokens of each partition (variable partitions), else NULL */
  int32_t cap;         /* resident capacity in pages (mandatory + buffer) */
  int32_t budget;      /* pages the unit may keep resident now, k <= budget <= cap (buffer elasticity) */
  int32_t D;           /* directory entries = ceil(P / 64) */
  int32_t S;           /* segments in this unit's pool */
  int32_t* dir;        /* [D] segment id or -1 */
  int32_t* seg;        /* [S][64] slot or -1 */
  int32_t* seg_live;   /* [S] live entries, -1 = segment free */
  int32_t* slot_part;  /* [cap] partition held by the slot, -1 = free */
  int32_t* last_use;   /* [cap] step of the last use */
  uint16_t* slots;     /* [cap][2][64][128] resident page copies ("HBM") */
} oracle_unit;

oracle_unit* oracle_unit_create(int32_t ntok, int32_t cap) {
  oracle_unit* u = (oracle_unit*)calloc(1, sizeof(oracle_unit));
  u->ntok = ntok;
  u->P = (ntok + OPART - 1) / OPART;
  u->cap = cap;
  u->budget = cap;
  u->P_cap = u->P;
  u->D = (u->P + OSEG - 1) / OSEG;
  u->S = u->D < cap ? u->D : cap;
  if (u->S < 1) u->S = 1;
  u->dir = (int32_t*)malloc(sizeof(int32_t) * (size_t)(u->D > 0 ? u->D : 1));
  u->seg = (int32_t*)malloc(sizeof(int32_t) * (size_t)u->S * OSEG);
  u->seg_live = (int32_t*)malloc(sizeof(int32_t) * (size_t)u->S);
  u->slot_part = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  u->last_use = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  u->slots = (uint16_t*)calloc((size_t)cap * OPAGE_ELEMS, sizeof(uint16_t));
  for (int32_t i = 0; i < u->D; ++i) u->dir[i] = -1;
  for (int32_t i = 0; i < u->S; ++i) u->seg_live[i] = -1;
  for (int32_t i = 0; i < cap; ++i) {
    u->slot_part[i] = -1;
    u->last_use[i] = 0;
  }
  return u;
}

/* Unit of variable partitions: partition p holds part_n[p] tokens (1..64). */
oracle_unit* oracle_unit_create_parts(const int32_t* part_n, int32_t P, int32_t cap) {
  oracle_unit* u = oracle_unit_create(P * OPART, cap);
  u->part_n = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
  int32_t n = 0;
  for (int32_t p = 0; p < P; ++p) {
    u->part_n[p] = part_n[p];
    n += part_n[p];
  }
  u->ntok = n;
  return u;
}

/* Tokens held by partition p's page. */
static int32_t unit_valid(const oracle_unit* u, int32_t p) {
  if (u->part_n) return u->part_n[p];
  return (p == u->P - 1) ? u->ntok - p * OPART : OPART;
}

/* ------------------------------------------------------------------------- */
/* KV append (tail mode). reading: new tokens go into a tail partition that is */
/* attended at every step; it is not selectable until it holds 64 tokens, when */
/* it is summarised, offloaded and becomes partition P (the caller appends its */
/* summary and host page, then calls oracle_unit_grow). The two-level table is */
/* sized for the partitions the unit may grow to.                              */
/* ------------------------------------------------------------------------- */
oracle_unit* oracle_unit_create_tail(int32_t P_complete, int32_t P_capacity, int32_t cap) {
  oracle_unit* u = oracle_unit_create(P_capacity * OPART, cap);
  u->P = P_complete;
  u->ntok = P_complete * OPART;
  return u;
}

/* ------------------------------------------------------------------------- */
/* Buffer elasticity ([XT] §2: the buffer part of a request's pages is resized */
/* by the scheduler with load; [GS] §2B). reading: the budget bounds the       */
/* resident pages; the manager counts free pages against it, so after a shrink */
/* the next step's demand includes the excess and the bucketed LRU reclaims    */
/* down to the budget. The budget never drops below the mandatory pages (k).   */
/* ------------------------------------------------------------------------- */
int32_t oracle_unit_set_budget(oracle_unit* u, int32_t pages) {
  if (pages < 1 || pages > u->cap) return -1;
  u->budget = pages;
  return 0;
}

int32_t oracle_unit_grow(oracle_unit* u) {
  if (u->P >= u->P_cap) return -1;
  u->P += 1;
  u->ntok = u->P * OPART;
  return 0;
}

void oracle_unit_destroy(oracle_unit* u) {
  if (!u) return;
  free(u->dir);
  free(u->seg);
  free(u->seg_live);
  free(u->slot_part);
  free(u->last_use);
  free(u->slots);
  free(u->part_n);
  free(u);
}

/* Walk: directory entry for p/64 -> segment -> entry p%64. */
int32_t oracle_resolve(const oracle_unit* u, int32_t p) {
  if (p < 0 || p >= u->P) return -1;
  int32_t s = u->dir[p / OSEG];
  if (s < 0) return -1;
  return u->seg[s * OSEG + p % OSEG];
}

static int table_set(oracle_unit* u, int32_t p, int32_t slot) {
  int32_t d = p / OSEG;
  if (u->dir[d] < 0) {
    int32_t s = -1;
    for (int32_t i = 0; i < u->S; ++i)
      if (u->seg_live[i] < 0) { s = i; break; }
    if (s < 0) return -1; /* pool exhausted */
    for (int e = 0; e < OSEG; ++e) u->seg[s * OSEG + e] = -1;
    u->seg_live[s] = 0;
    u->dir[d] = s;
  }
  int32_t s = u->dir[d];
  u->seg[s * OSEG + p % OSEG] = slot;
  u->seg_live[s] += 1;
  return 0;
}

static void table_clear(oracle_unit* u, int32_t p) {
  int32_t d = p / OSEG;
  int32_t s = u->dir[d];
  u->seg[s * OSEG + p % OSEG] = -1;
  u->seg_live[s] -= 1;
  if (u->seg_live[s] == 0) {
    u->seg_live[s] = -1;
    u->dir[d] = -1;
  }
}

int32_t oracle_live_segments(const oracle_unit* u) {
  int32_t n = 0;
  for (int32_t i = 0; i < u->S; ++i) n += u->seg_live[i] > 0;
  return n;
}

/* Per-step record of what the manager did. */
typedef struct oracle_manage_out {
  int32_t hits, misses, resident_before, free_before, demand, cutoff, evicted;
  int32_t error;        /* 0 ok, 1 = segment pool exhausted, 2 = no free page for a miss */
} oracle_manage_out;

/* ------------------------------------------------------------------------- */
/* Manage + Retrieve for one unit at step t ([XT] §2 and Fig 5 steps 1-4;       */
/* [GS] §2B):                                                                   */
/*  1. residency check of every selected partition through the table;         */
/*  2. selected pages are this step's mandatory pages: hits get timestamp t;  */
/*  3. if the misses do not fit in the free pages, bucketed LRU: every         */
/*     resident non-mandatory page falls in one of 64 timestamp buckets,        */
/*     one histogram pass, then whole buckets are reclaimed from the oldest     */
/*     upward until the reclaimed count covers the demand;                      */
/*  4. each miss gets a free page and its bytes are copied from the host page. */
/* readings: capacity = mandatory + buffer pages, free pages counted against  */
/* the unit's current budget (buffer elasticity); bucket of a page =            */
/* 63 - min(63, t - last_use) (0 = oldest); misses in ascending partition      */
/* order take free slots in ascending slot order.                              */
/* sel_slot[j], sel_hit[j] describe sel[j]; victims[] gets the evicted         */
/* partitions in ascending slot order. host_pages: [P][2][64][128].            */
/* ------------------------------------------------------------------------- */
void oracle_manage(oracle_unit* u, const int32_t* sel, int32_t keff, int32_t t, const uint16_t* host_pages,
                   int32_t* sel_slot, uint8_t* sel_hit, int32_t* victims, oracle_manage_out* out) {
  memset(out, 0, sizeof(*out));
  out->cutoff = -1;
  uint8_t* mand = (uint8_t*)calloc((size_t)u->cap, 1);

  /* 1 + 2: residency and timestamp bump */
  for (int32_t j = 0; j < keff; ++j) {
    int32_t s = oracle_resolve(u, sel[j]);
    sel_slot[j] = s;
    sel_hit[j] = s >= 0;
    if (s >= 0) {
      out->hits += 1;
      u->last_use[s] = t;
      mand[s] = 1;
    }
  }
  out->misses = keff - out->hits;
  for (int32_t s = 0; s < u->cap; ++s) out->resident_before += u->slot_part[s] >= 0;
  out->free_before = u->budget - out->resident_before; /* negative after a shrink */
  out->demand = out->misses - out->free_before;

  /* 3: bucketed LRU */
  if (out->demand > 0) {
    int32_t hist[OBUCKETS];
    memset(hist, 0, sizeof(hist));
    for (int32_t s = 0; s < u->cap; ++s) {
      if (u->slot_part[s] < 0 || mand[s]) continue;
      int32_t age = t - u->last_use[s];
      int32_t bucket = OBUCKETS - 1 - (age < OBUCKETS - 1 ? age : OBUCKETS - 1);
      hist[bucket] += 1;
    }
    int32_t cum = 0;
    for (int32_t c = 0; c < OBUCKETS; ++c) {
      cum += hist[c];
      if (cum >= out->demand) { out->cutoff = c; break; }
    }
    for (int32_t s = 0; s < u->cap; ++s) {
      if (u->slot_part[s] < 0 || mand[s]) continue;
      int32_t age = t - u->last_use[s];
      int32_t bucket = OBUCKETS - 1 - (age < OBUCKETS - 1 ? age : OBUCKETS - 1);
      if (bucket <= out->cutoff) {
        if (victims) victims[out->evicted] = u->slot_part[s];
        out->evicted += 1;
        table_clear(u, u->slot_part[s]);
        u->slot_part[s] = -1;
      }
    }
  }

  /* 4: assign free slots to the misses and retrieve their bytes */
  int32_t next = 0;
  for (int32_t j = 0; j < keff; ++j) {
    if (sel_hit[j]) continue;
    while (next < u->cap && u->slot_part[next] >= 0) ++next;
    if (next >= u->cap) { /* cannot happen: the LRU step freed at least `demand` pages */
      out->error = 2;
      sel_slot[j] = -1;
      continue;
    }
    int32_t s = next++;
    int32_t p = sel[j];
    u->slot_part[s] = p;
    u->last_use[s] = t;
    if (table_set(u, p, s) != 0) out->error = 1;
    memcpy(u->slots + (int64_t)s * OPAGE_ELEMS, host_pages + (int64_t)p * OPAGE_ELEMS,
           sizeof(uint16_t) * OPAGE_ELEMS);
    sel_slot[j] = s;
  }
  free(mand);
}

/* ------------------------------------------------------------------------- */
/* Attention over the selected tokens ([XT] §1 / Fig 3, Attention).            */
/* reading: exact softmax attention with scale 1/sqrt(128) over every valid     */
/* token of the selected partitions, read from their resident pages.           */
/* out[g][i], double.                                                          */
/* ------------------------------------------------------------------------- */
/* Attention over the selected pages plus, when tail_n > 0, the first tail_n tokens of
 * the tail page tail_kv ([2][64][128]: K rows then V rows). */
void oracle_attend_tail(const oracle_unit* u, const int32_t* sel, const int32_t* sel_slot, int32_t keff,
                        const uint16_t* q, int32_t G, const uint16_t* tail_kv, int32_t tail_n, double* out) {
  int64_t n = tail_n;
  for (int32_t j = 0; j < keff; ++j) {
    int32_t p = sel[j];
    n += unit_valid(u, p);
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  const double scale = 1.0 / sqrt((double)OD);
  for (int32_t g = 0; g < G; ++g) {
    double* o = out + g * OD;
    for (int i = 0; i < OD; ++i) o[i] = 0.0;
    if (n == 0) continue;
    /* scores of every attended token, pages in selection order, then the tail */
    int64_t c = 0;
    double m = -INFINITY;
    for (int32_t j = 0; j <= keff; ++j) {
      const uint16_t* K;
      int32_t valid;
      if (j < keff) {
        int32_t p = sel[j];
        valid = unit_valid(u, p);
        K = u->slots + (int64_t)sel_slot[j] * OPAGE_ELEMS;
      } else {
        valid = tail_n;
        K = tail_kv;
      }
      for (int32_t r = 0; r < valid; ++r) {
        double sdot = 0.0;
        for (int i = 0; i < OD; ++i) sdot += bf(q[g * OD + i]) * bf(K[r * OD + i]);
        x[c] = sdot * scale;
        if (x[c] > m) m = x[c];
        ++c;
      }
    }
    double l = 0.0;
    c = 0;
    for (int32_t j = 0; j <= keff; ++j) {
      const uint16_t* V;
      int32_t valid;
      if (j < keff) {
        int32_t p = sel[j];
        valid = unit_valid(u, p);
        V = u->slots + (int64_t)sel_slot[j] * OPAGE_ELEMS + OPART * OD;
      } else {
        valid = tail_n;
        V = tail_kv + OPART * OD;
      }
      for (int32_t r = 0; r < valid; ++r) {
        double w = exp(x[c] - m);
        l += w;
        for (int i = 0; i < OD; ++i) o[i] += w * bf(V[r * OD + i]);
        ++c;
      }
    }
    for (int i = 0; i < OD; ++i) o[i] /= l;
  }
  free(x);
}

void oracle_attend(const oracle_unit* u, const int32_t* sel, const int32_t* sel_slot, int32_t keff,
                   const uint16_t* q, int32_t G, double* out) {
  int64_t n = 0;
  for (int32_t j = 0; j < keff; ++j) {
    int32_t p = sel[j];
    int32_t valid = unit_valid(u, p);
    n += valid;
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  const double scale = 1.0 / sqrt((double)OD);
  for (int32_t g = 0; g < G; ++g) {
    double* o = out + g * OD;
    for (int i = 0; i < OD; ++i) o[i] = 0.0;
    if (n == 0) continue;
    int64_t c = 0;
    double m = -INFINITY;
    for (int32_t j = 0; j < keff; ++j) {
      int32_t p = sel[j];
      int32_t valid = unit_valid(u, p);
      const uint16_t* K = u->slots + (int64_t)sel_slot[j] * OPAGE_ELEMS;
      for (int32_t r = 0; r < valid; ++r) {
        double s = 0.0;
        for (int i = 0; i < OD; ++i) s += bf(q[g * OD + i]) * bf(K[r * OD + i]);
        x[c] = s * scale;
        if (x[c] > m) m = x[c];
        ++c;
      }
    }
    double l = 0.0;
    c = 0;
    for (int32_t j = 0; j < keff; ++j) {
      int32_t p = sel[j];
      int32_t valid = unit_valid(u, p);
      const uint16_t* V = u->slots + (int64_t)sel_slot[j] * OPAGE_ELEMS + OPART * OD;
      for (int32_t r = 0; r < valid; ++r) {
        double w = exp(x[c] - m);
        l += w;
        for (int i = 0; i < OD; ++i) o[i] += w * bf(V[r * OD + i]);
        ++c;
      }
    }
    for (int i = 0; i < OD; ++i) o[i] /= l;
  }
  free(x);
}

/* ------------------------------------------------------------------------- */
/* One whole decode step for one unit: Select -> Manage/Retrieve -> Attention. */
/* ------------------------------------------------------------------------- */
typedef struct oracle_step_io {
  const double* summ;         /* [P][128] */
  const uint16_t* host_pages; /* [P][2][64][128] */
  const uint16_t* q;          /* [G][128] bf16 */
  int32_t G, k, t;
  double* scores;             /* [P] out (may be NULL) */
  int32_t* sel;               /* [k] out */
  int32_t* sel_slot;          /* [k] out */
  uint8_t* sel_hit;           /* [k] out */
  int32_t* victims;           /* [cap] out (may be NULL) */
  double* out;                /* [G][128] out */
  oracle_manage_out mo;       /* out */
  int32_t keff;               /* out */
} oracle_step_io;

void oracle_step_unit(oracle_unit* u, oracle_step_io* io) {
  double* sc = io->scores ? io->scores : (double*)malloc(sizeof(double) * (size_t)(u->P > 0 ? u->P : 1));
  oracle_scores(io->summ, u->P, io->q, io->G, sc);
  io->keff = oracle_topk(sc, u->P, io->k, io->sel);
  oracle_manage(u, io->sel, io->keff, io->t, io->host_pages, io->sel_slot, io->sel_hit, io->victims, &io->mo);
  oracle_attend(u, io->sel, io->sel_slot, io->keff, io->q, io->G, io->out);
  if (!io->scores) free(sc);
}

/* Many units in parallel (independent units; used for CPU timing). */
int32_t oracle_step_units(oracle_unit** units, oracle_step_io* ios, int32_t n, int32_t nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int32_t i = 0; i < n; ++i) oracle_step_unit(units[i], &ios[i]);
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* State export for comparisons. */
void oracle_unit_export(const oracle_unit* u, int32_t* slot_part, int32_t* last_use, int32_t* resolve) {
  if (slot_part) memcpy(slot_part, u->slot_part, sizeof(int32_t) * (size_t)u->cap);
  if (last_use) memcpy(last_use, u->last_use, sizeof(int32_t) * (size_t)u->cap);
  if (resolve)
    for (int32_t p = 0; p < u->P; ++p) resolve[p] = oracle_resolve(u, p);
}

const uint16_t* oracle_unit_slot(const oracle_unit* u, int32_t s) { return u->slots + (int64_t)s * OPAGE_ELEMS; }
int32_t oracle_unit_P(const oracle_unit* u) { return u->P; }
int32_t oracle_unit_cap(const oracle_unit* u) { return u->cap; }
