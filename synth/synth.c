/*
 * Seeded synthetic Q/K/V generator with planted attention structure.
 *
 * Shared input source for the CUDA path and the CPU oracle: it produces the
 * bytes both sides consume and holds none of the sparse-attention method's
 * arithmetic (no softmax, no routing, no selection).
 *
 * Random numbers: splitmix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based hash
 * of (seed, tensor, flat index); normals by the Box-Muller transform.
 *
 * Layouts (bf16 bit patterns, row-major, contiguous):
 *   q [hq][n][128], k [hkv][n][128], v [hkv][n][128].
 *
 * Feature dimensions of q and k:
 *   [0, 96)    N(0,1) background noise (q, k); slash copies add to q here
 *   96         sink direction   (keys j < sink_tokens)
 *   97         needle direction (needle key columns)
 *   98..105    cluster directions (one per key/query block, 8 clusters)
 *   106..111   zero
 *   112..127   8 low-frequency rotary pairs (local band)
 * v is N(0,1) in all 128 dimensions.
 *
 * A structure with logit strength D adds D to q_i . k_j / sqrt(128) at the
 * positions it targets: symmetric amplitudes sqrt(D * sqrt(128)) on the
 * dedicated q and k dimensions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYNTH_D 128
#define SYNTH_NOISE_DIMS 96
#define SYNTH_BAND_PAIRS 8
#define SYNTH_CLUSTERS 8
#define SYNTH_BLOCK 128

typedef struct {
  int32_t hq, hkv, n;
  uint64_t seed;
  int32_t sink_tokens;
  float d_sink;
  int32_t n_needles;
  float d_needle;
  int32_t n_slash;
  float d_slash;
  int32_t slash_min, slash_max;
  int32_t band_w;
  float d_band;
  float d_cluster;
  const uint8_t* head_is_vs; /* [hq]: 1 = sink/slash/needle head, 0 = diffuse cluster head */
  int32_t nthreads;
} synth_config;

static inline uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

static inline uint64_t hash3(uint64_t seed, uint64_t tensor, uint64_t idx) {
  return splitmix64(splitmix64(seed ^ (tensor << 56)) ^ idx);
}

/* Uniform in [0, 1) with 53 random bits. */
static inline double uniform01(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

/* Standard normal pair for (seed, tensor, pair index). */
static inline void normal_pair(uint64_t seed, uint64_t tensor, uint64_t pair, double* z0, double* z1) {
  uint64_t h1 = hash3(seed, tensor, pair);
  uint64_t h2 = splitmix64(h1 ^ 0xD1B54A32D192ED03ull);
  double u1 = ((double)(h1 >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0, 1] */
  double u2 = uniform01(h2);
  double r = sqrt(-2.0 * log(u1));
  *z0 = r * cos(6.283185307179586 * u2);
  *z1 = r * sin(6.283185307179586 * u2);
}

static inline uint16_t to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline double from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

enum { T_Q = 0, T_K = 1, T_V = 2, T_NEEDLE = 3, T_SLASH = 4, T_BAND = 5, T_CLUSTER = 6 };

/* Cluster id of a 128-token block (same mapping for queries and keys). */
static inline int cluster_of(uint64_t seed, int block) {
  return (int)(hash3(seed, T_CLUSTER, (uint64_t)block) % SYNTH_CLUSTERS);
}

typedef struct {
  const synth_config* c;
  uint16_t *q, *k, *v;
  const uint8_t* needle_mask; /* [hkv][n] */
  const double* band_theta;   /* [hkv][SYNTH_BAND_PAIRS] */
  const int32_t* slash_off;   /* [hq][n_slash] */
  int phase;                  /* 0: k and v, 1: q */
  int tid, nthreads;
} job_t;

static void gen_kv_rows(const job_t* jb, int64_t row0, int64_t row1) {
  const synth_config* c = jb->c;
  const double s = sqrt(sqrt((double)SYNTH_D));
  const double a_sink = s * sqrt(c->d_sink > 0 ? c->d_sink : 0);
  const double a_needle = s * sqrt(c->d_needle > 0 ? c->d_needle : 0);
  const double a_cluster = s * sqrt(c->d_cluster > 0 ? c->d_cluster : 0);
  const double a_band = s * sqrt((c->d_band > 0 ? c->d_band : 0) / SYNTH_BAND_PAIRS);
  for (int64_t row = row0; row < row1; ++row) {
    const int g = (int)(row / c->n);
    const int j = (int)(row % c->n);
    double kr[SYNTH_D];
    for (int t = 0; t < SYNTH_NOISE_DIMS; t += 2) {
      uint64_t pair = ((uint64_t)row * SYNTH_D + (uint64_t)t) >> 1;
      normal_pair(c->seed, T_K, pair, &kr[t], &kr[t + 1]);
    }
    for (int t = SYNTH_NOISE_DIMS; t < SYNTH_D; ++t) kr[t] = 0.0;
    if (j < c->sink_tokens) kr[96] = a_sink;
    if (jb->needle_mask[(int64_t)g * c->n + j]) kr[97] = a_needle;
    kr[98 + cluster_of(c->seed, j / SYNTH_BLOCK)] = a_cluster;
    for (int p = 0; p < SYNTH_BAND_PAIRS; ++p) {
      double th = jb->band_theta[g * SYNTH_BAND_PAIRS + p] * (double)j;
      kr[112 + 2 * p] = a_band * cos(th);
      kr[113 + 2 * p] = a_band * sin(th);
    }
    uint16_t* ko = jb->k + row * SYNTH_D;
    for (int t = 0; t < SYNTH_D; ++t) ko[t] = to_bf16(kr[t]);
    uint16_t* vo = jb->v + row * SYNTH_D;
    for (int t = 0; t < SYNTH_D; t += 2) {
      double z0, z1;
      uint64_t pair = ((uint64_t)row * SYNTH_D + (uint64_t)t) >> 1;
      normal_pair(c->seed, T_V, pair, &z0, &z1);
      vo[t] = to_bf16(z0);
      vo[t + 1] = to_bf16(z1);
    }
  }
}

static void gen_q_rows(const job_t* jb, int64_t row0, int64_t row1) {
  const synth_config* c = jb->c;
  const int G = c->hq / c->hkv;
  const double s = sqrt(sqrt((double)SYNTH_D));
  const double a_sink = s * sqrt(c->d_sink > 0 ? c->d_sink : 0);
  const double a_needle = s * sqrt(c->d_needle > 0 ? c->d_needle : 0);
  const double a_cluster = s * sqrt(c->d_cluster > 0 ? c->d_cluster : 0);
  const double a_band = s * sqrt((c->d_band > 0 ? c->d_band : 0) / SYNTH_BAND_PAIRS);
  /* A copy of the key's noise part: peak logit lambda * |k_noise|^2 / sqrt(d)
   * with E|k_noise|^2 = 96, so lambda = d_slash * sqrt(d) / 96. */
  const double lam = (c->d_slash > 0 ? c->d_slash : 0) * sqrt((double)SYNTH_D) / SYNTH_NOISE_DIMS;
  for (int64_t row = row0; row < row1; ++row) {
    const int h = (int)(row / c->n);
    const int i = (int)(row % c->n);
    const int g = h / G;
    double qr[SYNTH_D];
    for (int t = 0; t < SYNTH_NOISE_DIMS; t += 2) {
      uint64_t pair = ((uint64_t)row * SYNTH_D + (uint64_t)t) >> 1;
      normal_pair(c->seed, T_Q, pair, &qr[t], &qr[t + 1]);
    }
    for (int t = SYNTH_NOISE_DIMS; t < SYNTH_D; ++t) qr[t] = 0.0;
    if (c->head_is_vs[h]) {
      for (int t = 0; t < c->n_slash; ++t) {
        int src = i - jb->slash_off[h * c->n_slash + t];
        if (src < 0) continue;
        const uint16_t* kk = jb->k + ((int64_t)g * c->n + src) * SYNTH_D;
        for (int u = 0; u < SYNTH_NOISE_DIMS; ++u) qr[u] += lam * from_bf16(kk[u]);
      }
      qr[96] = a_sink;
      qr[97] = a_needle;
      for (int p = 0; p < SYNTH_BAND_PAIRS; ++p) {
        double th = jb->band_theta[g * SYNTH_BAND_PAIRS + p] * (double)i;
        qr[112 + 2 * p] = a_band * cos(th);
        qr[113 + 2 * p] = a_band * sin(th);
      }
    } else {
      qr[98 + cluster_of(c->seed, i / SYNTH_BLOCK)] = a_cluster;
    }
    uint16_t* qo = jb->q + row * SYNTH_D;
    for (int t = 0; t < SYNTH_D; ++t) qo[t] = to_bf16(qr[t]);
  }
}

static void* worker(void* arg) {
  const job_t* jb = (const job_t*)arg;
  const synth_config* c = jb->c;
  const int64_t rows = (jb->phase == 0 ? (int64_t)c->hkv : (int64_t)c->hq) * c->n;
  const int64_t per = (rows + jb->nthreads - 1) / jb->nthreads;
  int64_t r0 = per * jb->tid, r1 = r0 + per;
  if (r1 > rows) r1 = rows;
  if (r0 < r1) {
    if (jb->phase == 0)
      gen_kv_rows(jb, r0, r1);
    else
      gen_q_rows(jb, r0, r1);
  }
  return NULL;
}

/* Needle key positions of kv group g: n_needles distinct uniform positions. */
int synth_needle_positions(const synth_config* c, int g, int32_t* out) {
  int cnt = 0;
  for (uint64_t t = 0; cnt < c->n_needles && t < (uint64_t)c->n_needles * 64 + 64; ++t) {
    int p = (int)(hash3(c->seed, T_NEEDLE, ((uint64_t)g << 32) | t) % (uint64_t)c->n);
    int dup = 0;
    for (int u = 0; u < cnt; ++u) dup |= (out[u] == p);
    if (!dup) out[cnt++] = p;
  }
  return cnt;
}

/* Slash offsets of q-head h, uniform in [slash_min, slash_max). */
void synth_slash_offsets(const synth_config* c, int h, int32_t* out) {
  const int span = c->slash_max > c->slash_min ? c->slash_max - c->slash_min : 1;
  for (int t = 0; t < c->n_slash; ++t)
    out[t] = c->slash_min + (int)(hash3(c->seed, T_SLASH, ((uint64_t)h << 32) | (uint64_t)t) % (uint64_t)span);
}

int synth_generate(const synth_config* c, uint16_t* q, uint16_t* k, uint16_t* v) {
  if (!c || !q || !k || !v || c->hq <= 0 || c->hkv <= 0 || c->hq % c->hkv || c->n <= 0) return 1;
  const int nt = c->nthreads > 0 ? c->nthreads : 1;
  uint8_t* needle_mask = (uint8_t*)calloc((size_t)c->hkv * c->n, 1);
  double* theta = (double*)malloc(sizeof(double) * c->hkv * SYNTH_BAND_PAIRS);
  int32_t* slash = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->hq * (c->n_slash > 0 ? c->n_slash : 1));
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (c->n_needles > 0 ? c->n_needles : 1));
  if (!needle_mask || !theta || !slash || !pos) {
    free(needle_mask); free(theta); free(slash); free(pos);
    return 2;
  }
  for (int g = 0; g < c->hkv; ++g) {
    int cnt = synth_needle_positions(c, g, pos);
    for (int u = 0; u < cnt; ++u) needle_mask[(int64_t)g * c->n + pos[u]] = 1;
    for (int p = 0; p < SYNTH_BAND_PAIRS; ++p)
      theta[g * SYNTH_BAND_PAIRS + p] =
          (c->band_w > 0 ? 3.141592653589793 / c->band_w : 0.0) * uniform01(hash3(c->seed, T_BAND, (uint64_t)(g * 64 + p)));
  }
  for (int h = 0; h < c->hq; ++h) synth_slash_offsets(c, h, slash + (size_t)h * (c->n_slash > 0 ? c->n_slash : 1));
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * nt);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
  for (int phase = 0; phase < 2; ++phase) { /* q copies rows of k: k first */
    for (int t = 0; t < nt; ++t) {
      jobs[t] = (job_t){c, q, k, v, needle_mask, theta, slash, phase, t, nt};
      pthread_create(&th[t], NULL, worker, &jobs[t]);
    }
    for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
  }
  free(jobs); free(th); free(needle_mask); free(theta); free(slash); free(pos);
  return 0;
}
