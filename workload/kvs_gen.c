/*
 * Seeded synthetic inputs for the sparse KV-cache decode step.
 *
 * This module only draws random numbers and lays them out; it holds none of the
 * decode method's arithmetic (no index keys, scores, selection, cache policy or
 * attention).  Both the CPU oracle and the CUDA path read the bytes it writes.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014) used counter-style: the n-th output for a seed is
 * mix(seed + (n + 1) * gamma).  The counter packs (stream, request, layer, head,
 * position, dim pair) so any slice can be regenerated without storing the rest.
 * Normals come from the Box-Muller transform (fp32 libm), then are rounded to bf16
 * with round-to-nearest-even.
 *
 * Streams: 1 = K (or the MLA latent row), 2 = V, 3 = query innovations,
 *          4 = draft-query noise, 5 = heavy-position shuffle, 6 = heavy-position carry-over.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC -pthread (no fused multiply-add,
 * so results do not depend on the host ISA's contraction choices).
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define GEN_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t gen_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t gen_at(uint64_t seed, uint64_t ctr) { return gen_mix(seed + (ctr + 1) * GEN_GAMMA); }

/* 4 + 6 + 6 + 8 + 24 + 10 = 58 bits: stream<16, req<64, layer<64, head<256, pos<2^24, pair<1024 */
static inline uint64_t gen_ctr(int stream, int req, int layer, int head, int64_t pos, int pair) {
  uint64_t c = (uint64_t)stream;
  c = (c << 6) | (uint64_t)req;
  c = (c << 6) | (uint64_t)layer;
  c = (c << 8) | (uint64_t)head;
  c = (c << 24) | (uint64_t)pos;
  c = (c << 10) | (uint64_t)pair;
  return c;
}

static inline void gen_normal_pair(uint64_t x, double* z0, double* z1) {
  /* Box-Muller in single precision from two 24-bit uniforms in (0, 1); the outputs are
   * stored as bf16, so fp32 carries more precision than is kept. */
  float u1 = ((float)(x >> 40) + 0.5f) * (1.0f / 16777216.0f);
  float u2 = ((float)(x & 0xffffffull) + 0.5f) * (1.0f / 16777216.0f);
  float r = sqrtf(-2.0f * logf(u1));
  float s, c;
  sincosf(6.28318530717958647692f * u2, &s, &c);
  *z0 = (double)(r * c);
  *z1 = (double)(r * s);
}

static inline uint16_t gen_bf16(double v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
  uint32_t lo = u & 0xffffu, hi = u >> 16;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

/* Stored value of a drawn real number: bf16 of v, or, in integer mode (int_scale > 0), bf16 of
 * round(v * int_scale) clipped to [-int_clip, int_clip] (small integers are exact in bf16). */
static inline uint16_t gen_store(double v, float int_scale, float int_clip) {
  if (int_scale > 0.f) {
    double x = nearbyint(v * (double)int_scale);
    if (x > int_clip) x = int_clip;
    if (x < -int_clip) x = -int_clip;
    return gen_bf16(x);
  }
  return gen_bf16(v);
}

int kvs_gen_counter_limits_ok(int n_req, int n_layer, int n_head, int64_t n_pos, int d) {
  return n_req <= 64 && n_layer <= 64 && n_head <= 256 && n_pos <= (1 << 24) && d <= 2048 && (d % 2) == 0;
}

/* ------------------------------------------------------------------ K / V */

typedef struct {
  uint64_t seed;
  int32_t n_req, n_layer, n_kv_head, d_k, d_v; /* d_v == 0: no separate V (V shares the K row) */
  int32_t ctx0;                                /* prefilled tokens; positions >= ctx0 are zero */
  int32_t n_heavy;                             /* heavy key positions per heavy set */
  int64_t max_ctx;                             /* allocated tokens per (layer, req, head) row */
  float heavy_scale;
  int32_t heavy_shared_layers;                 /* 1: one heavy set per (req, head) for all layers */
  double rho_layer;                            /* 0: layers independent; else AR(1) mix across layers */
  int32_t n_threads;
  float int_scale;                             /* > 0: integer-valued mode (see gen_store) */
  float int_clip;
  double heavy_keep;                           /* per-layer sets: share of layer l-1's heavy positions
                                                  layer l keeps (0: independent sets) */
} kvs_gen_kv_params;

/* Heavy positions of one set.  Each position of `prev` (the layer below's set, or NULL) is kept
 * when its stream-6 draw falls below heavy_keep; the set is then filled up to n_heavy with the
 * entries of a partial Fisher-Yates shuffle of [0, ctx0) driven by stream 5, in shuffle order,
 * skipping positions already in the set.  With prev == NULL (or heavy_keep == 0) the set is the
 * first n_heavy shuffle entries. */
static void gen_heavy_set(const kvs_gen_kv_params* p, int req, int layer, int head, int32_t* perm, uint8_t* mask,
                          const uint8_t* prev) {
  int64_t n = p->ctx0;
  if (n <= 0) return;
  int64_t k = p->n_heavy < n ? p->n_heavy : n;
  memset(mask, 0, (size_t)n);
  int64_t cnt = 0;
  if (prev && p->heavy_keep > 0.0) {
    const double keep = p->heavy_keep >= 1.0 ? 1.0 : p->heavy_keep;
    for (int64_t pos = 0; pos < n && cnt < k; ++pos) {
      if (!prev[pos]) continue;
      uint64_t x = gen_at(p->seed, gen_ctr(6, req, layer, head, pos, 0));
      if ((double)(x >> 11) * (1.0 / 9007199254740992.0) < keep) {
        mask[pos] = 1;
        ++cnt;
      }
    }
  }
  for (int64_t i = 0; i < n; ++i) perm[i] = (int32_t)i;
  for (int64_t i = 0; i < n && cnt < k; ++i) {
    uint64_t x = gen_at(p->seed, gen_ctr(5, req, layer, head, i, 0));
    uint64_t range = (uint64_t)(n - i);
    int64_t j = i + (int64_t)(((unsigned __int128)x * range) >> 64);
    int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    if (!mask[perm[i]]) {
      mask[perm[i]] = 1;
      ++cnt;
    }
  }
}

int kvs_gen_heavy_positions(const kvs_gen_kv_params* p, int req, int layer, int head, int32_t* out) {
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)(p->ctx0 > 0 ? p->ctx0 : 1));
  uint8_t* mask = (uint8_t*)malloc((size_t)(p->ctx0 > 0 ? p->ctx0 : 1));
  if (!perm || !mask) { free(perm); free(mask); return -1; }
  if (p->heavy_shared_layers) {
    gen_heavy_set(p, req, 0, head, perm, mask, NULL);
  } else {
    /* chained sets: build layers 0..layer in order */
    uint8_t* prev = (uint8_t*)malloc((size_t)(p->ctx0 > 0 ? p->ctx0 : 1));
    if (!prev) { free(perm); free(mask); return -1; }
    for (int l = 0; l <= layer; ++l) {
      gen_heavy_set(p, req, l, head, perm, mask, l > 0 ? prev : NULL);
      if (l < layer) memcpy(prev, mask, (size_t)p->ctx0);
    }
    free(prev);
  }
  int c = 0;
  for (int64_t i = 0; i < p->ctx0; ++i) if (mask[i]) out[c++] = (int32_t)i;
  free(perm); free(mask);
  return c;
}

typedef struct {
  const kvs_gen_kv_params* p;
  uint16_t* k;
  uint16_t* v;
  const uint8_t* heavy; /* [n_sets][ctx0] */
  int64_t job_begin, job_end; /* jobs = (req, head, pos chunk) */
  int64_t chunk;
} gen_kv_job;

static void* gen_kv_worker(void* arg) {
  gen_kv_job* J = (gen_kv_job*)arg;
  const kvs_gen_kv_params* p = J->p;
  int64_t n_chunks = (p->max_ctx + J->chunk - 1) / J->chunk;
  int dk = p->d_k, dv = p->d_v;
  double* prev_k = (double*)malloc(sizeof(double) * (size_t)dk);
  double* prev_v = (double*)malloc(sizeof(double) * (size_t)(dv > 0 ? dv : 1));
  double sk = sqrt(1.0 - p->rho_layer * p->rho_layer);
  for (int64_t job = J->job_begin; job < J->job_end; ++job) {
    int64_t c = job % n_chunks;
    int head = (int)((job / n_chunks) % p->n_kv_head);
    int req = (int)(job / n_chunks / p->n_kv_head);
    int64_t p0 = c * J->chunk, p1 = p0 + J->chunk < p->max_ctx ? p0 + J->chunk : p->max_ctx;
    for (int64_t pos = p0; pos < p1; ++pos) {
      for (int layer = 0; layer < p->n_layer; ++layer) {
        size_t row = ((size_t)((int64_t)layer * p->n_req + req) * p->n_kv_head + head) * (size_t)p->max_ctx + (size_t)pos;
        uint16_t* krow = J->k + row * (size_t)dk;
        uint16_t* vrow = dv > 0 ? J->v + row * (size_t)dv : NULL;
        if (pos >= p->ctx0) {
          memset(krow, 0, sizeof(uint16_t) * (size_t)dk);
          if (vrow) memset(vrow, 0, sizeof(uint16_t) * (size_t)dv);
          continue;
        }
        int set_layer = p->heavy_shared_layers ? 0 : layer;
        size_t set = ((size_t)req * (size_t)(p->heavy_shared_layers ? 1 : p->n_layer) + (size_t)set_layer) * (size_t)p->n_kv_head + (size_t)head;
        double hs = (p->n_heavy > 0 && J->heavy[set * (size_t)p->ctx0 + (size_t)pos]) ? (double)p->heavy_scale : 1.0;
        for (int pr = 0; pr < dk / 2; ++pr) {
          double z0, z1;
          gen_normal_pair(gen_at(p->seed, gen_ctr(1, req, layer, head, pos, pr)), &z0, &z1);
          if (p->rho_layer != 0.0 && layer > 0) {
            z0 = p->rho_layer * prev_k[2 * pr] + sk * z0;
            z1 = p->rho_layer * prev_k[2 * pr + 1] + sk * z1;
          }
          prev_k[2 * pr] = z0; prev_k[2 * pr + 1] = z1;
          krow[2 * pr] = gen_store(z0, p->int_scale, p->int_clip);
          krow[2 * pr + 1] = gen_store(z1, p->int_scale, p->int_clip);
          if (hs != 1.0) {
            krow[2 * pr] = gen_store(z0 * hs, p->int_scale, p->int_clip * (float)hs);
            krow[2 * pr + 1] = gen_store(z1 * hs, p->int_scale, p->int_clip * (float)hs);
          }
        }
        for (int pr = 0; vrow && pr < dv / 2; ++pr) {
          double z0, z1;
          gen_normal_pair(gen_at(p->seed, gen_ctr(2, req, layer, head, pos, pr)), &z0, &z1);
          if (p->rho_layer != 0.0 && layer > 0) {
            z0 = p->rho_layer * prev_v[2 * pr] + sk * z0;
            z1 = p->rho_layer * prev_v[2 * pr + 1] + sk * z1;
          }
          prev_v[2 * pr] = z0; prev_v[2 * pr + 1] = z1;
          vrow[2 * pr] = gen_store(z0, p->int_scale, p->int_clip);
          vrow[2 * pr + 1] = gen_store(z1, p->int_scale, p->int_clip);
        }
      }
    }
  }
  free(prev_k); free(prev_v);
  return NULL;
}

static int gen_threads(int requested) {
  if (requested > 0) return requested;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* Fills K [n_layer][n_req][n_kv_head][max_ctx][d_k] and, when d_v > 0, V likewise. */
int kvs_gen_fill_kv(const kvs_gen_kv_params* p, uint16_t* k, uint16_t* v) {
  if (!kvs_gen_counter_limits_ok(p->n_req, p->n_layer, p->n_kv_head, p->max_ctx, p->d_k)) return -1;
  if (p->d_v > 0 && (p->d_v % 2)) return -1;
  if (p->ctx0 > p->max_ctx) return -1;
  int n_sets = p->n_req * (p->heavy_shared_layers ? 1 : p->n_layer) * p->n_kv_head;
  uint8_t* heavy = NULL;
  if (p->n_heavy > 0 && p->ctx0 > 0) {
    heavy = (uint8_t*)malloc((size_t)n_sets * (size_t)p->ctx0);
    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)p->ctx0);
    if (!heavy || !perm) { free(heavy); free(perm); return -2; }
    for (int req = 0; req < p->n_req; ++req)
      for (int l = 0; l < (p->heavy_shared_layers ? 1 : p->n_layer); ++l)
        for (int h = 0; h < p->n_kv_head; ++h) {
          size_t set = ((size_t)req * (size_t)(p->heavy_shared_layers ? 1 : p->n_layer) + (size_t)l) * (size_t)p->n_kv_head + (size_t)h;
          const uint8_t* prev = NULL;
          if (!p->heavy_shared_layers && l > 0)
            prev = heavy + (((size_t)req * (size_t)p->n_layer + (size_t)(l - 1)) * (size_t)p->n_kv_head + (size_t)h) *
                               (size_t)p->ctx0;
          gen_heavy_set(p, req, l, h, perm, heavy + set * (size_t)p->ctx0, prev);
        }
    free(perm);
  }
  int nt = gen_threads(p->n_threads);
  int64_t chunk = 256;
  int64_t n_jobs = (int64_t)p->n_req * p->n_kv_head * ((p->max_ctx + chunk - 1) / chunk);
  if (nt > n_jobs) nt = (int)(n_jobs > 0 ? n_jobs : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  gen_kv_job* jobs = (gen_kv_job*)malloc(sizeof(gen_kv_job) * (size_t)nt);
  for (int i = 0; i < nt; ++i) {
    jobs[i].p = p; jobs[i].k = k; jobs[i].v = v; jobs[i].heavy = heavy; jobs[i].chunk = chunk;
    jobs[i].job_begin = n_jobs * i / nt;
    jobs[i].job_end = n_jobs * (i + 1) / nt;
    pthread_create(&th[i], NULL, gen_kv_worker, &jobs[i]);
  }
  for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
  free(th); free(jobs); free(heavy);
  return 0;
}

/* One new token row for every (layer, req, head) at position pos:
 * out_k [n_layer][n_req][n_kv_head][d_k], out_v likewise (when d_v > 0).  Same streams as
 * the prefilled rows, so a token appended at pos equals what a prefill to pos+1 would hold. */
int kvs_gen_token(const kvs_gen_kv_params* p, int64_t pos, uint16_t* out_k, uint16_t* out_v) {
  if (!kvs_gen_counter_limits_ok(p->n_req, p->n_layer, p->n_kv_head, pos + 1, p->d_k)) return -1;
  double sk = sqrt(1.0 - p->rho_layer * p->rho_layer);
  int dk = p->d_k, dv = p->d_v;
  double* prev = (double*)malloc(sizeof(double) * (size_t)(dk > dv ? dk : dv));
  for (int req = 0; req < p->n_req; ++req)
    for (int head = 0; head < p->n_kv_head; ++head)
      for (int which = 0; which < (dv > 0 ? 2 : 1); ++which) {
        int d = which ? dv : dk;
        for (int layer = 0; layer < p->n_layer; ++layer) {
          size_t row = (size_t)((int64_t)layer * p->n_req + req) * (size_t)p->n_kv_head + (size_t)head;
          uint16_t* o = (which ? out_v : out_k) + row * (size_t)d;
          for (int pr = 0; pr < d / 2; ++pr) {
            double z0, z1;
            gen_normal_pair(gen_at(p->seed, gen_ctr(which ? 2 : 1, req, layer, head, pos, pr)), &z0, &z1);
            if (p->rho_layer != 0.0 && layer > 0) {
              z0 = p->rho_layer * prev[2 * pr] + sk * z0;
              z1 = p->rho_layer * prev[2 * pr + 1] + sk * z1;
            }
            prev[2 * pr] = z0; prev[2 * pr + 1] = z1;
            o[2 * pr] = gen_store(z0, p->int_scale, p->int_clip);
            o[2 * pr + 1] = gen_store(z1, p->int_scale, p->int_clip);
          }
        }
      }
  free(prev);
  return 0;
}

/* ------------------------------------------------------------------ queries */

typedef struct {
  uint64_t seed;
  int32_t n_req, n_layer, n_q_head, d;
  double rho;       /* AR(1) coefficient over decode steps */
  double rho_layer; /* 0: layers independent; else AR(1) mix across layers */
  float int_scale;  /* > 0: integer-valued mode (see gen_store) */
  float int_clip;
} kvs_gen_q_params;

/* Base state e[layer][req][head][d] (fp64) of the per-layer AR(1) over steps:
 * e_0 = eps_0, e_t = rho * e_{t-1} + sqrt(1 - rho^2) * eps_t, eps from stream 3 at pos = t. */
int kvs_gen_q_advance(const kvs_gen_q_params* p, double* state, int64_t t) {
  if (!kvs_gen_counter_limits_ok(p->n_req, p->n_layer, p->n_q_head, t + 1, p->d)) return -1;
  double s = sqrt(1.0 - p->rho * p->rho);
  size_t i = 0;
  for (int l = 0; l < p->n_layer; ++l)
    for (int r = 0; r < p->n_req; ++r)
      for (int h = 0; h < p->n_q_head; ++h)
        for (int pr = 0; pr < p->d / 2; ++pr, i += 2) {
          double z0, z1;
          gen_normal_pair(gen_at(p->seed, gen_ctr(3, r, l, h, t, pr)), &z0, &z1);
          if (t == 0) { state[i] = z0; state[i + 1] = z1; }
          else { state[i] = p->rho * state[i] + s * z0; state[i + 1] = p->rho * state[i + 1] + s * z1; }
        }
  return 0;
}

/* Query values q[layer][req][head][d] (fp64) from the base state: layer 0 is e^0; layer l mixes
 * q^{l-1} and e^l with rho_layer (identity when rho_layer == 0). */
void kvs_gen_q_values(const kvs_gen_q_params* p, const double* state, double* q) {
  size_t per_layer = (size_t)p->n_req * (size_t)p->n_q_head * (size_t)p->d;
  double s = sqrt(1.0 - p->rho_layer * p->rho_layer);
  for (int l = 0; l < p->n_layer; ++l)
    for (size_t i = 0; i < per_layer; ++i) {
      size_t j = (size_t)l * per_layer + i;
      q[j] = (p->rho_layer != 0.0 && l > 0) ? p->rho_layer * q[j - per_layer] + s * state[j] : state[j];
    }
}

void kvs_gen_to_bf16(const kvs_gen_q_params* p, const double* x, size_t n, uint16_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = gen_store(x[i], p->int_scale, p->int_clip);
}

/* Draft query j of step t: q_future (the fp64 query of step t + j) plus sigma * N(0,1) noise
 * from stream 4 at pos = 8 t + j.  Output bf16 [layer][req][head][d] at out (strided by the
 * caller through out_layer_stride / out_req_stride / out_head_stride elements). */
int kvs_gen_draft(const kvs_gen_q_params* p, const double* q_future, int64_t t, int j, double sigma,
                  uint16_t* out, int64_t out_layer_stride, int64_t out_req_stride, int64_t out_head_stride) {
  if (!kvs_gen_counter_limits_ok(p->n_req, p->n_layer, p->n_q_head, 8 * t + j + 1, p->d)) return -1;
  size_t i = 0;
  for (int l = 0; l < p->n_layer; ++l)
    for (int r = 0; r < p->n_req; ++r)
      for (int h = 0; h < p->n_q_head; ++h) {
        uint16_t* o = out + l * out_layer_stride + r * out_req_stride + h * out_head_stride;
        for (int pr = 0; pr < p->d / 2; ++pr, i += 2) {
          double z0, z1;
          gen_normal_pair(gen_at(p->seed, gen_ctr(4, r, l, h, 8 * t + j, pr)), &z0, &z1);
          o[2 * pr] = gen_store(q_future[i] + sigma * z0, p->int_scale, p->int_clip);
          o[2 * pr + 1] = gen_store(q_future[i + 1] + sigma * z1, p->int_scale, p->int_clip);
        }
      }
  return 0;
}

/* Draft noise of draft slot j at step t, as an AR(1) over steps with coefficient rho_d:
 * n_0 = eps_0, n_t = rho_d * n_{t-1} + sqrt(1 - rho_d^2) * eps_t, eps from stream 4 at pos = 8 t + j
 * (the draws kvs_gen_draft uses), so every n_t is N(0, 1) and rho_d = 0 gives kvs_gen_draft's noise.
 * state [layer][req][head][d] fp64 holds n_{t-1} on entry (ignored at t = 0) and n_t on return. */
int kvs_gen_draft_noise_advance(const kvs_gen_q_params* p, double* state, int64_t t, int j, double rho_d) {
  if (!kvs_gen_counter_limits_ok(p->n_req, p->n_layer, p->n_q_head, 8 * t + j + 1, p->d)) return -1;
  double s = sqrt(1.0 - rho_d * rho_d);
  size_t i = 0;
  for (int l = 0; l < p->n_layer; ++l)
    for (int r = 0; r < p->n_req; ++r)
      for (int h = 0; h < p->n_q_head; ++h)
        for (int pr = 0; pr < p->d / 2; ++pr, i += 2) {
          double z0, z1;
          gen_normal_pair(gen_at(p->seed, gen_ctr(4, r, l, h, 8 * t + j, pr)), &z0, &z1);
          if (t == 0) { state[i] = z0; state[i + 1] = z1; }
          else { state[i] = rho_d * state[i] + s * z0; state[i + 1] = rho_d * state[i + 1] + s * z1; }
        }
  return 0;
}

/* Draft query from the fp64 future query and a noise state: bf16(q_future + sigma * noise), laid
 * out like kvs_gen_draft's output. */
void kvs_gen_draft_with_noise(const kvs_gen_q_params* p, const double* q_future, const double* noise, double sigma,
                              uint16_t* out, int64_t out_layer_stride, int64_t out_req_stride,
                              int64_t out_head_stride) {
  size_t i = 0;
  for (int l = 0; l < p->n_layer; ++l)
    for (int r = 0; r < p->n_req; ++r)
      for (int h = 0; h < p->n_q_head; ++h) {
        uint16_t* o = out + l * out_layer_stride + r * out_req_stride + h * out_head_stride;
        for (int k = 0; k < p->d; ++k, ++i) o[k] = gen_store(q_future[i] + sigma * noise[i], p->int_scale, p->int_clip);
      }
}

/* Seeded uniform fp32 array in [lo, hi) from stream `stream` (used for stand-alone score arrays). */
void kvs_gen_uniform_f32(uint64_t seed, int stream, int64_t n, float lo, float hi, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint64_t x = gen_at(seed, ((uint64_t)stream << 54) | (uint64_t)i);
    double u = (double)(x >> 11) * (1.0 / 9007199254740992.0);
    out[i] = (float)(lo + (hi - lo) * u);
  }
}

/* Seeded integers in [0, range) (for stand-alone selection sequences). */
void kvs_gen_randint(uint64_t seed, int stream, int64_t n, int64_t range, int64_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint64_t x = gen_at(seed, ((uint64_t)stream << 54) | (uint64_t)i);
    out[i] = (int64_t)(((unsigned __int128)x * (uint64_t)range) >> 64);
  }
}
