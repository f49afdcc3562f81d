/*
 * Seeded synthetic inputs for the SPIN sparse-decode data path.
 *
 * This module only DRAWS inputs: keys, values, per-partition offsets, query
 * trajectories and per-request context lengths. It contains none of the
 * method's arithmetic (no summaries, scores, selection, paging or attention),
 * so the oracle and the CUDA path can both take their inputs from it.
 *
 * Workload recipe (the synthetic stand-in for the long-context benchmarks the
 * SPIN pages evaluate on, "Unifying Sparse Attention with Hierarchical Memory
 * for Scalable Long-Context LLM Serving", evaluation section):
 *   K[t][i] = bf16( n_K[t][i] + mu_p[i] ),  V[t][i] = bf16( n_V[t][i] + mu_p[i] )
 *     with n ~ N(0,1) independent per element and p = t / 64 the partition;
 *   mu_p[i] ~ N(0, mu_std^2), one 128-vector per (layer, request, kv head,
 *     partition), the same vector added to every token of the partition;
 *   optionally a fraction of partitions gets mu_p = hot_norm * qhat, where
 *     qhat is the normalised sum of the group's step-0 queries;
 *   q_0 ~ N(0,1);  q_t = a * q_{t-1} + c * N(0,1) in fp32, rounded to bf16
 *     each step (no renormalisation).
 *
 * Randomness is counter based: every value is a pure function of (seed, a
 * stream tag, the indices of the element), so results do not depend on the
 * number of threads or the order of calls. The counter hash is the SplitMix64
 * output function (Steele, Lea and Flood, "Fast Splittable Pseudorandom
 * Number Generators", OOPSLA 2014). Normal deviates come from inverse-CDF
 * table lookup on 16-bit uniforms (65536 equiprobable quantiles of N(0,1)).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define WL_D 128
#define WL_PART 64

typedef struct wl_cfg {
  uint64_t seed;
  int32_t B, L, Hq, Hkv, d;
  float drift_a, drift_c; /* q_t = a q_{t-1} + c N(0,1) */
  float mu_std;           /* std of the per-partition offset */
  float hot_norm;         /* norm of the query-aligned offsets; 0 = none */
  double hot_frac;        /* fraction of partitions given an aligned offset */
  const int64_t* ctx_len; /* [B] tokens per request */
} wl_cfg;

enum {
  TAG_KNOISE = 1,
  TAG_VNOISE = 2,
  TAG_MU = 3,
  TAG_Q0 = 4,
  TAG_QN = 5,
  TAG_CTX = 6,
  TAG_HOT = 7,
};

static inline uint64_t splitmix64(uint64_t z) {
  z += 0x9e3779b97f4a7c15ULL;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b, uint64_t c,
                                  uint64_t d) {
  uint64_t k = splitmix64(seed ^ (tag * 0xd1b54a32d192ed03ULL));
  k = splitmix64(k + a);
  k = splitmix64(k + b);
  k = splitmix64(k + c);
  return splitmix64(k + d);
}

/* 65536 equiprobable quantiles of N(0,1): table[i] = Phi^-1((i + 0.5) / 65536). */
static float g_ntab[65536];
static int g_ntab_ready = 0;

static double phi_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

void wl_init(void) {
  if (__atomic_load_n(&g_ntab_ready, __ATOMIC_ACQUIRE)) return;
  for (int i = 0; i < 32768; ++i) {
    double p = ((double)i + 0.5) / 65536.0;
    double lo = -12.0, hi = 0.0;
    for (int it = 0; it < 64; ++it) {
      double mid = 0.5 * (lo + hi);
      if (phi_cdf(mid) < p) lo = mid; else hi = mid;
    }
    float x = (float)(0.5 * (lo + hi));
    g_ntab[i] = x;
    g_ntab[65535 - i] = -x;
  }
  __atomic_store_n(&g_ntab_ready, 1, __ATOMIC_RELEASE);
}

/* Normal deviate number `idx` of the stream `key`: four deviates per hash. */
static inline float normal_at(uint64_t key, uint64_t idx) {
  uint64_t h = splitmix64(key + (idx >> 2));
  unsigned sh = (unsigned)(idx & 3) * 16u;
  return g_ntab[(h >> sh) & 0xffffu];
}

static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0; /* NaN */
  u += 0x7fffu + ((u >> 16) & 1u);                    /* round to nearest even */
  return (uint16_t)(u >> 16);
}

static inline float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ---- per-request context length (stress workload: whole partitions) ---- */
int64_t wl_ctx_partitions(uint64_t seed, int32_t b, int32_t pmin, int32_t pmax) {
  uint64_t h = splitmix64(stream_key(seed, TAG_CTX, (uint64_t)b, 0, 0, 0));
  uint64_t span = (uint64_t)(pmax - pmin + 1);
  return (int64_t)pmin + (int64_t)(h % span);
}

/* ---- queries ---- */
/* state: fp32 [L][B][Hq][128]; q_0 ~ N(0,1). */
void wl_query_init(const wl_cfg* c, float* state) {
  wl_init();
  for (int l = 0; l < c->L; ++l)
    for (int b = 0; b < c->B; ++b)
      for (int hq = 0; hq < c->Hq; ++hq) {
        uint64_t key = stream_key(c->seed, TAG_Q0, (uint64_t)l, (uint64_t)b, (uint64_t)hq, 0);
        float* s = state + (((int64_t)l * c->B + b) * c->Hq + hq) * WL_D;
        for (int i = 0; i < WL_D; ++i) s[i] = normal_at(key, (uint64_t)i);
      }
}

/* Advance the fp32 state from step t-1 to step t (t >= 1). */
void wl_query_step(const wl_cfg* c, int32_t t, float* state) {
  wl_init();
  const float a = c->drift_a, cc = c->drift_c;
  for (int l = 0; l < c->L; ++l)
    for (int b = 0; b < c->B; ++b)
      for (int hq = 0; hq < c->Hq; ++hq) {
        uint64_t key = stream_key(c->seed, TAG_QN, (uint64_t)l, (uint64_t)b, (uint64_t)hq, (uint64_t)t);
        float* s = state + (((int64_t)l * c->B + b) * c->Hq + hq) * WL_D;
        for (int i = 0; i < WL_D; ++i) {
          float keep = a * s[i];
          float fresh = cc * normal_at(key, (uint64_t)i);
          s[i] = keep + fresh;
        }
      }
}

void wl_to_bf16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(x[i]);
}

/* ---- per-partition offsets ---- */
static int64_t n_hot(const wl_cfg* c, int64_t P) {
  if (c->hot_norm <= 0.0f || c->hot_frac <= 0.0) return 0;
  int64_t n = (int64_t)llround(c->hot_frac * (double)P);
  return n > P ? P : n;
}

/* hot[p] = 1 for the partitions of unit (l,b,h) that get a query-aligned offset:
 * a partial Fisher-Yates shuffle draws n_hot of the P indices without replacement. */
static void hot_mask(const wl_cfg* c, int l, int b, int h, int64_t P, uint8_t* hot) {
  memset(hot, 0, (size_t)P);
  int64_t n = n_hot(c, P);
  if (n == 0) return;
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
  for (int64_t i = 0; i < P; ++i) perm[i] = (int32_t)i;
  uint64_t key = stream_key(c->seed, TAG_HOT, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
  for (int64_t i = 0; i < n; ++i) {
    uint64_t r = splitmix64(key + (uint64_t)i);
    int64_t j = i + (int64_t)(r % (uint64_t)(P - i));
    int32_t tmp = perm[i];
    perm[i] = perm[j];
    perm[j] = tmp;
    hot[perm[i]] = 1;
  }
  free(perm);
}

/* Unit direction of the sum of the group's bf16 step-0 queries. */
static void group_qhat(const wl_cfg* c, int l, int b, int h, float* qhat) {
  int G = c->Hq / c->Hkv;
  double acc[WL_D];
  for (int i = 0; i < WL_D; ++i) acc[i] = 0.0;
  for (int g = 0; g < G; ++g) {
    int hq = h * G + g;
    uint64_t key = stream_key(c->seed, TAG_Q0, (uint64_t)l, (uint64_t)b, (uint64_t)hq, 0);
    for (int i = 0; i < WL_D; ++i) acc[i] += (double)bf16_to_f32(f32_to_bf16(normal_at(key, (uint64_t)i)));
  }
  double nrm = 0.0;
  for (int i = 0; i < WL_D; ++i) nrm += acc[i] * acc[i];
  nrm = sqrt(nrm);
  for (int i = 0; i < WL_D; ++i) qhat[i] = nrm > 0.0 ? (float)(acc[i] / nrm) : 0.0f;
}

/* mu: fp32 [np][128] for partitions p0 .. p0+np-1 of unit (l,b,h). */
void wl_unit_mu(const wl_cfg* c, int32_t l, int32_t b, int32_t h, int64_t p0, int64_t np, float* mu) {
  wl_init();
  int64_t P = (c->ctx_len[b] + WL_PART - 1) / WL_PART;
  uint8_t* hot = NULL;
  float qhat[WL_D];
  if (n_hot(c, P) > 0) {
    hot = (uint8_t*)malloc((size_t)P);
    hot_mask(c, l, b, h, P, hot);
    group_qhat(c, l, b, h, qhat);
  }
  uint64_t key = stream_key(c->seed, TAG_MU, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
  for (int64_t j = 0; j < np; ++j) {
    int64_t p = p0 + j;
    float* m = mu + j * WL_D;
    if (hot && p < P && hot[p]) {
      for (int i = 0; i < WL_D; ++i) m[i] = c->hot_norm * qhat[i];
    } else {
      for (int i = 0; i < WL_D; ++i) m[i] = c->mu_std * normal_at(key, (uint64_t)(p * WL_D + i));
    }
  }
  free(hot);
}

/* Number of hot partitions of a unit (for workload statistics). */
int64_t wl_unit_hot_count(const wl_cfg* c, int32_t b) {
  int64_t P = (c->ctx_len[b] + WL_PART - 1) / WL_PART;
  return n_hot(c, P);
}

void wl_unit_hot_mask(const wl_cfg* c, int32_t l, int32_t b, int32_t h, uint8_t* hot) {
  wl_init();
  int64_t P = (c->ctx_len[b] + WL_PART - 1) / WL_PART;
  hot_mask(c, l, b, h, P, hot);
}

/* ---- keys and values ---- */
static void fill_tokens(const wl_cfg* c, int l, int b, int h, int64_t tok0, int64_t ntok, const float* mu,
                        int64_t mu_p0, uint16_t* k, uint16_t* v) {
  uint64_t kk = stream_key(c->seed, TAG_KNOISE, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
  uint64_t kv = stream_key(c->seed, TAG_VNOISE, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
  for (int64_t t = 0; t < ntok; ++t) {
    int64_t tok = tok0 + t;
    const float* m = mu + (tok / WL_PART - mu_p0) * WL_D;
    uint64_t base = (uint64_t)tok * WL_D;
    for (int i = 0; i < WL_D; i += 4) {
      /* one hash yields the four deviates idx .. idx+3 (idx is a multiple of 4) */
      uint64_t hk = splitmix64(kk + ((base + (uint64_t)i) >> 2));
      uint64_t hv = splitmix64(kv + ((base + (uint64_t)i) >> 2));
      for (int j = 0; j < 4; ++j) {
        float nk = g_ntab[(hk >> (16 * j)) & 0xffffu];
        float nv = g_ntab[(hv >> (16 * j)) & 0xffffu];
        k[t * WL_D + i + j] = f32_to_bf16(nk + m[i + j]);
        v[t * WL_D + i + j] = f32_to_bf16(nv + m[i + j]);
      }
    }
  }
}

/* K, V bf16 [ntok][128] for tokens tok0 .. tok0+ntok-1 of unit (l,b,h). */
void wl_unit_kv(const wl_cfg* c, int32_t l, int32_t b, int32_t h, int64_t tok0, int64_t ntok, uint16_t* k,
                uint16_t* v) {
  wl_init();
  if (ntok <= 0) return;
  int64_t p0 = tok0 / WL_PART, p1 = (tok0 + ntok - 1) / WL_PART;
  float* mu = (float*)malloc(sizeof(float) * (size_t)((p1 - p0 + 1) * WL_D));
  wl_unit_mu(c, l, b, h, p0, p1 - p0 + 1, mu);
  fill_tokens(c, l, b, h, tok0, ntok, mu, p0, k, v);
  free(mu);
}

/* K, V bf16 [Hkv][ctx_len[b]][128] for all kv heads of request b in layer l,
 * the layout the index/offload entry point takes. */
void wl_request_kv(const wl_cfg* c, int32_t l, int32_t b, uint16_t* k, uint16_t* v, int32_t nthreads) {
  wl_init();
  const int64_t n = c->ctx_len[b];
  if (n <= 0) return;
  const int64_t P = (n + WL_PART - 1) / WL_PART;
  const int64_t blk = 16; /* partitions per work item */
  const int64_t nblk = (P + blk - 1) / blk;
  const int64_t items = (int64_t)c->Hkv * nblk;
  (void)nthreads;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t it = 0; it < items; ++it) {
    int h = (int)(it / nblk);
    int64_t pb = (it % nblk) * blk;
    int64_t pe = pb + blk < P ? pb + blk : P;
    int64_t tok0 = pb * WL_PART;
    int64_t tok1 = pe * WL_PART < n ? pe * WL_PART : n;
    wl_unit_kv(c, l, b, h, tok0, tok1 - tok0, k + ((int64_t)h * n + tok0) * WL_D,
               v + ((int64_t)h * n + tok0) * WL_D);
  }
}

/* Raw deviates for statistical checks of the generator itself. */
void wl_normals(uint64_t seed, uint64_t tag, int64_t n, float* out) {
  wl_init();
  uint64_t key = stream_key(seed, 100 + tag, 0, 0, 0, 0);
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, (uint64_t)i);
}
