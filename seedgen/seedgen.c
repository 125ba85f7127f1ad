/* Seeded synthetic inputs shared by the tests, the oracle runs and the
 * benchmark. It holds none of the training step's arithmetic: only random
 * bits, normal deviates and constant fills.
 *
 * Bits: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used counter-based: draw i
 * of stream (seed, stream) is mix64(key + (i+1) * GOLDEN) with
 * key = mix64(seed ^ mix64(stream)), so any element can be produced
 * independently of the others and fills can run on many threads.
 * Normals: Box-Muller (1958) on the pair of draws (2j, 2j+1), giving
 * elements 2j (cosine branch) and 2j+1 (sine branch), computed in double and
 * then rounded to the output type (round-to-nearest-even for bf16).
 * Token ids: draw mod V (V is far below 2^64, so the bias is negligible).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

static uint64_t stream_key(uint64_t seed, uint64_t stream) { return mix64(seed ^ mix64(stream + GOLDEN)); }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffff) ? 0x40 : 0));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Normal deviate for element e of the stream (pairs share two draws). */
static inline double normal_at(uint64_t key, uint64_t e) {
  const uint64_t j = e >> 1;
  const uint64_t b1 = draw(key, 2 * j), b2 = draw(key, 2 * j + 1);
  const double u1 = ((double)(b1 >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0,1] */
  const double u2 = (double)(b2 >> 11) * (1.0 / 9007199254740992.0);         /* [0,1) */
  const double r = sqrt(-2.0 * log(u1));
  const double a = 6.283185307179586476925 * u2;
  return (e & 1) ? r * sin(a) : r * cos(a);
}

typedef struct {
  void* out;
  uint64_t begin, end, key;
  double mean, std;
  int kind; /* 0 normal f32, 1 normal bf16 */
} job_t;

static void* run_job(void* p) {
  job_t* J = (job_t*)p;
  if (J->kind == 0) {
    float* o = (float*)J->out;
    for (uint64_t e = J->begin; e < J->end; ++e) o[e] = (float)(J->mean + J->std * normal_at(J->key, e));
  } else {
    uint16_t* o = (uint16_t*)J->out;
    for (uint64_t e = J->begin; e < J->end; ++e)
      o[e] = f32_to_bf16_rne((float)(J->mean + J->std * normal_at(J->key, e)));
  }
  return NULL;
}

static void parallel_fill(void* out, uint64_t n, uint64_t key, double mean, double std, int kind, int threads) {
  if (threads < 1) threads = 1;
  if (n < (1u << 20)) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t th[256];
  job_t jobs[256];
  const uint64_t chunk = ((n + threads - 1) / threads + 1) & ~1ull;
  int started = 0;
  for (int t = 0; t < threads; ++t) {
    uint64_t b = (uint64_t)t * chunk, e = b + chunk;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[t] = (job_t){out, b, e, key, mean, std, kind};
    if (threads == 1 || pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0) {
      run_job(&jobs[t]);
      th[t] = 0;
    }
    started++;
  }
  for (int t = 0; t < started; ++t)
    if (threads > 1 && th[t]) pthread_join(th[t], NULL);
}

/* out[e] = mean + std * N(0,1)_e of stream (seed, stream), e in [0, n). */
void seedgen_normal_f32(float* out, uint64_t n, uint64_t seed, uint64_t stream, double mean, double std,
                        int threads) {
  parallel_fill(out, n, stream_key(seed, stream), mean, std, 0, threads);
}

/* The same values rounded to bf16 (stored as uint16 bit patterns). */
void seedgen_normal_bf16(uint16_t* out, uint64_t n, uint64_t seed, uint64_t stream, double mean, double std,
                         int threads) {
  parallel_fill(out, n, stream_key(seed, stream), mean, std, 1, threads);
}

void seedgen_fill_f32(float* out, uint64_t n, float value) {
  for (uint64_t i = 0; i < n; ++i) out[i] = value;
}

void seedgen_fill_bf16(uint16_t* out, uint64_t n, float value) {
  const uint16_t b = f32_to_bf16_rne(value);
  for (uint64_t i = 0; i < n; ++i) out[i] = b;
}

/* Token ids uniform in [0, V): out[i] = draw(i) mod V. */
void seedgen_tokens(int32_t* out, uint64_t n, uint64_t seed, uint64_t stream, int32_t V) {
  const uint64_t key = stream_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)(draw(key, i) % (uint64_t)V);
}

/* Raw 64-bit draws (for checking the generator against its definition). */
void seedgen_bits(uint64_t* out, uint64_t n, uint64_t seed, uint64_t stream) {
  const uint64_t key = stream_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = draw(key, i);
}
