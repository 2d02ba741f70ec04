/*
 * Seeded synthetic inputs for the MoE-layer forward (shared by the oracle side and
 * the CUDA side; holds none of the layer's arithmetic).
 *
 * Every value is a pure function of (seed, stream, index): a SplitMix64 sequence
 * (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014) keyed by (seed, stream) and indexed by the element position, so any
 * slice can be produced in any order by any number of threads.
 *
 * Streams: 1 = x, 2 = router weight, 3 = router bias, 6 = token ids, 7 = hash table,
 * 8 = hot-expert set; expert weights: 4/9 = routed gate-up codes/scales, 11/12 = routed
 * down codes/scales, 5/10 = shared gate-up codes/scales, 13/14 = shared down codes/scales.
 *
 * Expert weights are produced directly in MXFP4 form (E2M1 codes + E8M0 scale bytes):
 * no quantiser lives here.  The code distribution is a fixed categorical law chosen
 * to look like N(0, 1/d) values after per-32 MX quantisation: the maximum of 32 such
 * normals is about 2.2 / sqrt(d), which fixes the usual block exponent e0, and a block
 * gets the next lower exponent with probability 0.22 (the share of blocks whose maximum
 * falls below the power of two); the scale byte per block is 127 + e0 or 127 + e0 - 1
 * with e0 = floor(log2(2.2 / sqrt(d))) - 2.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread synth.c -o libsynth.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + GOLDEN) ^ (stream * GOLDEN + 0x632BE59BD9B4E019ULL));
}

/* index-th output of the SplitMix64 sequence whose state starts at key */
static inline uint64_t draw(uint64_t key, uint64_t index) { return mix64(key + (index + 1) * GOLDEN); }

/* uniform in (0, 1] with 53 random bits */
static inline double unit_open0(uint64_t u) { return ((double)(u >> 11) + 1.0) * 0x1.0p-53; }
static inline double unit_closed0(uint64_t u) { return (double)(u >> 11) * 0x1.0p-53; }

/* standard normal by Box-Muller from two consecutive draws */
static inline double normal_at(uint64_t key, uint64_t index) {
  double u1 = unit_open0(draw(key, 2 * index));
  double u2 = unit_closed0(draw(key, 2 * index + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t index) { return draw(stream_key(seed, stream), index); }
double synth_normal(uint64_t seed, uint64_t stream, uint64_t index) { return normal_at(stream_key(seed, stream), index); }

/* ---------------- threading helper ---------------- */
typedef struct {
  void (*fn)(void* ctx, int64_t lo, int64_t hi);
  void* ctx;
  int64_t lo, hi;
} job_t;

static void* job_run(void* p) {
  job_t* j = (job_t*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t n, int threads, void (*fn)(void*, int64_t, int64_t), void* ctx) {
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if (n < 4096 || threads == 1) { fn(ctx, 0, n); return; }
  pthread_t th[64];
  job_t jobs[64];
  int64_t chunk = (n + threads - 1) / threads;
  int used = 0;
  for (int t = 0; t < threads; ++t) {
    int64_t lo = t * chunk, hi = lo + chunk;
    if (lo >= n) break;
    if (hi > n) hi = n;
    jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].lo = lo; jobs[t].hi = hi;
    if (pthread_create(&th[t], NULL, job_run, &jobs[t]) != 0) { fn(ctx, lo, hi); jobs[t].fn = NULL; }
    used = t + 1;
  }
  for (int t = 0; t < used; ++t)
    if (jobs[t].fn) pthread_join(th[t], NULL);
}

/* ---------------- x: bf16 ~ N(0, scale^2), one attempt counter per row ---------------- */
typedef struct { uint64_t key; int64_t d; double scale; const int32_t* attempt; uint16_t* out; } x_ctx;

static void x_body(void* p, int64_t lo, int64_t hi) {
  x_ctx* c = (x_ctx*)p;
  for (int64_t t = lo; t < hi; ++t) {
    uint64_t a = c->attempt ? (uint64_t)c->attempt[t] : 0;
    uint64_t base = (((uint64_t)t << 8) + a) * (uint64_t)c->d;
    for (int64_t i = 0; i < c->d; ++i)
      c->out[t * c->d + i] = float_to_bf16_rne((float)(c->scale * normal_at(c->key, base + (uint64_t)i)));
  }
}

/* Rows of x (bf16 bits).  attempt[t] (0..255, may be NULL) selects an independent redraw of row t. */
void synth_x_bf16(uint64_t seed, int64_t T, int64_t d, double scale, const int32_t* attempt, uint16_t* out, int threads) {
  x_ctx c = {stream_key(seed, 1), d, scale, attempt, out};
  parallel_for(T, threads, x_body, &c);
}

/* ---------------- router weight fp32 ~ N(0, 1/d), bias fp32 ~ U(-0.1, 0.1) ---------------- */
void synth_router(uint64_t seed, int64_t E, int64_t d, float* w, float* bias) {
  uint64_t kw = stream_key(seed, 2), kb = stream_key(seed, 3);
  double s = 1.0 / sqrt((double)d);
  for (int64_t i = 0; i < E * d; ++i) w[i] = (float)(s * normal_at(kw, (uint64_t)i));
  for (int64_t e = 0; e < E; ++e) bias[e] = (float)(-0.1 + 0.2 * unit_closed0(draw(kb, (uint64_t)e)));
}

/* Skewed-load bias: n_hot experts chosen by a seeded partial Fisher-Yates shuffle get +hot_bias. */
void synth_hot_bias(uint64_t seed, int64_t E, int64_t n_hot, float hot_bias, float* bias, int32_t* hot_ids) {
  uint64_t k = stream_key(seed, 8);
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int64_t e = 0; e < E; ++e) perm[e] = (int32_t)e;
  for (int64_t i = 0; i < n_hot && i < E; ++i) {
    int64_t j = i + (int64_t)(draw(k, (uint64_t)i) % (uint64_t)(E - i));
    int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    bias[perm[i]] += hot_bias;
    if (hot_ids) hot_ids[i] = perm[i];
  }
  free(perm);
}

/* ---------------- MXFP4 expert weights ---------------- */
/* Cumulative probabilities (x 65536) of E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}: the law of
 * round-to-nearest(2.2 |z|), z ~ N(0,1), saturated at 6 -- close to what a block of 32 normals
 * looks like after division by its E8M0 scale; with the scale bytes below the decoded weights have
 * standard deviation close to 1/sqrt(d_in). */
static const uint32_t kMagCdf[8] = {5929, 17487, 28186, 37595, 48772, 58220, 64026, 65536};

static inline uint8_t code_from_bits(uint32_t bits17) {
  uint32_t u = bits17 & 0xFFFFu;
  uint8_t mag = 0;
  while (mag < 7 && u >= kMagCdf[mag]) ++mag;
  return (uint8_t)(mag | (((bits17 >> 16) & 1u) << 3));
}

typedef struct { uint64_t kc, ks; int64_t cols; int e0; uint8_t* codes; uint8_t* scales; int64_t row0; } w_ctx;

static void w_body(void* p, int64_t lo, int64_t hi) {
  w_ctx* c = (w_ctx*)p;
  int64_t bpr = c->cols / 2, spr = c->cols / 32;
  for (int64_t r = lo; r < hi; ++r) {
    uint64_t gr = (uint64_t)(c->row0 + r);
    for (int64_t b = 0; b < bpr; ++b) {
      uint64_t u = draw(c->kc, gr * (uint64_t)bpr + (uint64_t)b);
      uint8_t lo4 = code_from_bits((uint32_t)(u & 0x1FFFFu));
      uint8_t hi4 = code_from_bits((uint32_t)((u >> 32) & 0x1FFFFu));
      c->codes[r * bpr + b] = (uint8_t)(lo4 | (hi4 << 4));
    }
    for (int64_t s = 0; s < spr; ++s) {
      uint64_t u = draw(c->ks, gr * (uint64_t)spr + (uint64_t)s);
      int down = unit_closed0(u) < 0.22 ? 1 : 0;
      c->scales[r * spr + s] = (uint8_t)(127 + c->e0 - down);
    }
  }
}

/* Nominal block exponent for N(0, 1/d_in) weights: floor(log2(2.2/sqrt(d_in))) - 2. */
int synth_weight_e0(int64_t d_in) { return (int)floor(log2(2.2 / sqrt((double)d_in))) - 2; }

/* A [rows x cols] MXFP4 matrix (cols multiple of 32): codes (element 2i in the low nibble of
 * byte i) and E8M0 scale bytes.  row0 offsets the counter so sub-blocks of one logical matrix can
 * be produced separately.  stream_codes / stream_scales pick the matrix (see the stream list above). */
void synth_mxfp4(uint64_t seed, int stream_codes, int stream_scales, int64_t row0, int64_t rows, int64_t cols,
                 int64_t d_in, uint8_t* codes, uint8_t* scales, int threads) {
  w_ctx c = {stream_key(seed, (uint64_t)stream_codes), stream_key(seed, (uint64_t)stream_scales), cols,
             synth_weight_e0(d_in), codes, scales, row0};
  parallel_for(rows, threads, w_body, &c);
}

/* ---------------- hash routing inputs ---------------- */
void synth_token_ids(uint64_t seed, int64_t T, int64_t V, int32_t* tok) {
  uint64_t k = stream_key(seed, 6);
  for (int64_t t = 0; t < T; ++t) tok[t] = (int32_t)(draw(k, (uint64_t)t) % (uint64_t)V);
}

/* table[V][k]: k distinct expert ids per row by a partial Fisher-Yates shuffle of 0..E-1. */
void synth_hash_table(uint64_t seed, int64_t V, int64_t E, int64_t k, int32_t* table) {
  uint64_t key = stream_key(seed, 7);
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int64_t v = 0; v < V; ++v) {
    for (int64_t e = 0; e < E; ++e) perm[e] = (int32_t)e;
    for (int64_t i = 0; i < k; ++i) {
      int64_t j = i + (int64_t)(draw(key, (uint64_t)(v * k + i)) % (uint64_t)(E - i));
      int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
      table[v * k + i] = perm[i];
    }
  }
  free(perm);
}
