/*
 * Seeded synthetic input generators shared by the oracle side and the GPU
 * side of every test and benchmark.  This file holds no quantization or
 * linear-layer arithmetic: it only turns (seed, key, index) into numbers.
 *
 * Randomness is counter based, so any element can be produced independently
 * and the work splits across threads without changing a single bit:
 *
 *   stream base  b(seed, key) = fmix(seed * 0x9E3779B97F4A7C15 ^ fmix(key + 0x632BE59BD9B4E019))
 *   raw word     h(i)         = fmix(b + (i + 1) * 0x9E3779B97F4A7C15)
 *   uniform      U(i)         = ((h(i) >> 11) + 0.5) * 2^-53      in (0, 1)
 *
 * fmix is the SplitMix64 output function (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).
 *
 * Normal draws use the Box-Muller transform on the pair (U(2j), U(2j+1)):
 *   Z(2j)   = sqrt(-2 ln U(2j)) * cos(2 pi U(2j+1))
 *   Z(2j+1) = sqrt(-2 ln U(2j)) * sin(2 pi U(2j+1))
 * computed in double.
 *
 * Student-t with nu = 3 degrees of freedom: T(i) = Z_a(i) / sqrt((Z_b(3i)^2 +
 * Z_b(3i+1)^2 + Z_b(3i+2)^2) / 3), Z_a and Z_b being the normal streams of
 * two different keys.
 *
 * bf16 conversion is round-to-nearest-even on the fp32 bit pattern.
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t fmix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t key) {
  return fmix(seed * GOLDEN ^ fmix(key + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t raw_word(uint64_t base, uint64_t i) {
  return fmix(base + (i + 1) * GOLDEN);
}

static inline double uniform01(uint64_t base, uint64_t i) {
  return ((double)(raw_word(base, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t base, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t j = i >> 1;
  double u1 = uniform01(base, 2 * j);
  double u2 = uniform01(base, 2 * j + 1);
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

uint16_t qs_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* threaded driver                                                      */

typedef struct {
  int kind; /* 0 normal f32, 1 student-t f32, 2 X bf16 rows */
  uint64_t seed, key, key2;
  int64_t begin, end;
  double scale;
  float* out_f32;
  uint16_t* out_bf16;
  int64_t row_len;            /* X: columns per row */
  const uint8_t* chan_boost;  /* X: per-column flag, 1 = boosted channel */
  double boost;
} job_t;

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  uint64_t b1 = stream_base(j->seed, j->key);
  uint64_t b2 = stream_base(j->seed, j->key2);
  for (int64_t i = j->begin; i < j->end; ++i) {
    if (j->kind == 0) {
      j->out_f32[i] = (float)(j->scale * normal_at(b1, (uint64_t)i));
    } else if (j->kind == 1) {
      double z0 = normal_at(b1, (uint64_t)i);
      double c0 = normal_at(b2, 3 * (uint64_t)i);
      double c1 = normal_at(b2, 3 * (uint64_t)i + 1);
      double c2 = normal_at(b2, 3 * (uint64_t)i + 2);
      double t = z0 / sqrt((c0 * c0 + c1 * c1 + c2 * c2) / 3.0);
      j->out_f32[i] = (float)(j->scale * t);
    } else {
      double z = j->scale * normal_at(b1, (uint64_t)i);
      int64_t col = i % j->row_len;
      if (j->chan_boost && j->chan_boost[col]) z *= j->boost;
      j->out_bf16[i] = qs_bf16_from_f32((float)z);
    }
  }
  return NULL;
}

static int thread_count(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  if (n < 1) n = 1;
  if (n > 32) n = 32;
  return (int)n;
}

static void run_parallel(job_t proto, int64_t n) {
  int nt = thread_count();
  if (n < 65536) nt = 1;
  pthread_t th[32];
  job_t jobs[32];
  int64_t chunk = (n + nt - 1) / nt;
  int started = 0;
  for (int t = 0; t < nt; ++t) {
    jobs[t] = proto;
    jobs[t].begin = t * chunk;
    jobs[t].end = (t + 1) * chunk < n ? (t + 1) * chunk : n;
    if (jobs[t].begin >= jobs[t].end) break;
    if (t == 0) continue;
    if (pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0) {
      run_job(&jobs[t]);
      jobs[t].begin = jobs[t].end;
      th[t] = 0;
    }
    started = t;
  }
  if (n > 0) run_job(&jobs[0]);
  for (int t = 1; t <= started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* exported entry points                                                */

/* out[i] = (float)(sigma * Z(i)), i in [0, n), normal stream of (seed, key). */
void qs_normal_f32(uint64_t seed, uint64_t key, float sigma, int64_t n, float* out) {
  job_t j = {0};
  j.kind = 0; j.seed = seed; j.key = key; j.scale = sigma; j.out_f32 = out;
  run_parallel(j, n);
}

/* out[i] = (float)(scale * T(i)), Student-t(3) from normal keys key_z, key_chi. */
void qs_student_t3_f32(uint64_t seed, uint64_t key_z, uint64_t key_chi, float scale, int64_t n,
                       float* out) {
  job_t j = {0};
  j.kind = 1; j.seed = seed; j.key = key_z; j.key2 = key_chi; j.scale = scale; j.out_f32 = out;
  run_parallel(j, n);
}

/* Picks `count` distinct channels out of K with a partial Fisher-Yates
 * shuffle driven by the raw words of (seed, key): for step i, swap position
 * i with i + (h(i) mod (K - i)).  The chosen channels are written sorted
 * ascending.  Returns 0 on success, -1 on bad arguments. */
static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}
int qs_pick_channels(uint64_t seed, uint64_t key, int32_t K, int32_t count, int32_t* out) {
  if (K <= 0 || count < 0 || count > K) return -1;
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  if (!perm) return -1;
  for (int32_t i = 0; i < K; ++i) perm[i] = i;
  uint64_t b = stream_base(seed, key);
  for (int32_t i = 0; i < count; ++i) {
    uint64_t span = (uint64_t)(K - i);
    int32_t r = i + (int32_t)(raw_word(b, (uint64_t)i) % span);
    int32_t t = perm[i]; perm[i] = perm[r]; perm[r] = t;
  }
  memcpy(out, perm, sizeof(int32_t) * (size_t)count);
  free(perm);
  qsort(out, (size_t)count, sizeof(int32_t), cmp_i32);
  return 0;
}

/* Activation matrix X[M][K] as bf16 bit patterns: element (m, k) is
 * bf16(sigma * Z(m*K + k) * (k boosted ? boost : 1)).  `boosted` is an
 * optional list of `nboost` channel indices (may be NULL). */
int qs_activations_bf16(uint64_t seed, uint64_t key, int64_t M, int64_t K, float sigma,
                        const int32_t* boosted, int32_t nboost, float boost, uint16_t* out) {
  if (M < 0 || K <= 0) return -1;
  uint8_t* flag = NULL;
  if (boosted && nboost > 0) {
    flag = (uint8_t*)calloc((size_t)K, 1);
    if (!flag) return -1;
    for (int32_t i = 0; i < nboost; ++i) {
      if (boosted[i] < 0 || boosted[i] >= K) { free(flag); return -1; }
      flag[boosted[i]] = 1;
    }
  }
  job_t j = {0};
  j.kind = 2; j.seed = seed; j.key = key; j.scale = sigma; j.out_bf16 = out;
  j.row_len = K; j.chan_boost = flag; j.boost = boost;
  run_parallel(j, M * K);
  free(flag);
  return 0;
}

/* Rounds an fp32 array to bf16 bit patterns (round to nearest even). */
void qs_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = qs_bf16_from_f32(in[i]);
}
