/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file produces INPUT data only (weights, gradients and Adam moments of
 * the right shapes and scales). It holds none of the optimizer's arithmetic and
 * is shared by the tests, the bench and the oracle's callers; neither the CUDA
 * library nor the oracle includes or links it.
 *
 * Value i of stream s under seed S is a pure function of (S, s, i):
 *   key  = splitmix64(S ^ splitmix64(s))
 *   h    = splitmix64(key + i)
 *   k    = (h & 0xffff) + (h>>16 & 0xffff) + (h>>32 & 0xffff) + (h>>48) - 131070
 *   x    = (float)k * scale            (one IEEE fp32 multiply)
 * k is an Irwin-Hall(4) draw on a 16-bit lattice, centred, so x has mean 0 and
 * standard deviation sigma when scale = sigma / sqrt((2^32 - 1) / 3). It is a
 * stand-in for N(0, sigma): variance-matched, bounded at about 3.46 sigma, and
 * computed with integer steps plus one correctly rounded multiply so that any
 * implementation of the same definition gives the same bits.
 *
 * splitmix64 is the published mixing function of Steele, Lea and Flood
 * ("Fast splittable pseudorandom number generators", OOPSLA 2014).
 *
 * bf16 fields take the upper 16 bits of x (round toward zero). That choice is
 * deliberate: it is a data-preparation step, distinct from the round-to-nearest
 * conversion the optimizer performs on its outputs.
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off -pthread gen.c -o libsynth.so
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

static inline float draw(uint64_t key, uint64_t i, float scale) {
  uint64_t h = splitmix64(key + i);
  int64_t k = (int64_t)(h & 0xffffu) + (int64_t)((h >> 16) & 0xffffu) +
              (int64_t)((h >> 32) & 0xffffu) + (int64_t)(h >> 48) - 131070;
  return (float)k * scale;
}

static inline uint16_t upper16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return (uint16_t)(u >> 16);
}

enum { KIND_F32 = 0, KIND_BF16 = 1, KIND_SQ_F32 = 2 };

typedef struct {
  int kind;
  uint64_t key;
  uint64_t start;
  int64_t n;
  float scale;
  void* out;
} job_t;

static void run_job(const job_t* j) {
  if (j->kind == KIND_F32) {
    float* o = (float*)j->out;
    for (int64_t i = 0; i < j->n; ++i) o[i] = draw(j->key, j->start + (uint64_t)i, j->scale);
  } else if (j->kind == KIND_SQ_F32) {
    float* o = (float*)j->out;
    for (int64_t i = 0; i < j->n; ++i) {
      float x = draw(j->key, j->start + (uint64_t)i, j->scale);
      o[i] = x * x;
    }
  } else {
    uint16_t* o = (uint16_t*)j->out;
    for (int64_t i = 0; i < j->n; ++i) o[i] = upper16(draw(j->key, j->start + (uint64_t)i, j->scale));
  }
}

static void* thread_main(void* p) {
  run_job((const job_t*)p);
  return NULL;
}

static int fill(int kind, uint64_t seed, uint64_t stream, uint64_t start, int64_t n, float scale,
                void* out, int threads) {
  if (n < 0 || (n > 0 && out == NULL)) return -1;
  uint64_t key = splitmix64(seed ^ splitmix64(stream));
  size_t esz = (kind == KIND_BF16) ? 2 : 4;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < (int64_t)1 << 20) threads = 1;
  job_t jobs[256];
  pthread_t tids[256];
  int64_t per = (n + threads - 1) / threads;
  int started = 0;
  for (int t = 0; t < threads; ++t) {
    int64_t a = per * t, b = a + per;
    if (b > n) b = n;
    if (a >= b) break;
    jobs[t].kind = kind;
    jobs[t].key = key;
    jobs[t].start = start + (uint64_t)a;
    jobs[t].n = b - a;
    jobs[t].scale = scale;
    jobs[t].out = (char*)out + (size_t)a * esz;
    if (t == 0) continue; /* run on the calling thread below */
    if (pthread_create(&tids[t], NULL, thread_main, &jobs[t]) != 0) {
      run_job(&jobs[t]); /* no thread available: do it here */
      tids[t] = 0;
    }
    started = t + 1;
  }
  if (n > 0) run_job(&jobs[0]);
  for (int t = 1; t < started; ++t)
    if (tids[t]) pthread_join(tids[t], NULL);
  return 0;
}

/* x_i ~ the lattice stand-in for N(0, sigma); fp32 output. */
int synth_fill_f32(uint64_t seed, uint64_t stream, uint64_t start, int64_t n, float scale, float* out,
                   int threads) {
  return fill(KIND_F32, seed, stream, start, n, scale, out, threads);
}

/* Same draw, stored as the upper 16 bits (bf16, toward zero). */
int synth_fill_bf16(uint64_t seed, uint64_t stream, uint64_t start, int64_t n, float scale,
                    uint16_t* out, int threads) {
  return fill(KIND_BF16, seed, stream, start, n, scale, out, threads);
}

/* Square of the same draw (fp32 multiply), e.g. a second moment v = x^2. */
int synth_fill_sq_f32(uint64_t seed, uint64_t stream, uint64_t start, int64_t n, float scale,
                      float* out, int threads) {
  return fill(KIND_SQ_F32, seed, stream, start, n, scale, out, threads);
}

/* Raw 64-bit hash output, for the generator's own determinism tests. */
uint64_t synth_hash(uint64_t seed, uint64_t stream, uint64_t i) {
  return splitmix64(splitmix64(seed ^ splitmix64(stream)) + i);
}

/* Random access: out[j] = value at index idx[j] (for sampled checks of big blocks). */
int synth_gather(int kind, uint64_t seed, uint64_t stream, const uint64_t* idx, int64_t n, float scale,
                 void* out) {
  if (n < 0 || (n > 0 && (idx == NULL || out == NULL))) return -1;
  uint64_t key = splitmix64(seed ^ splitmix64(stream));
  for (int64_t j = 0; j < n; ++j) {
    float x = draw(key, idx[j], scale);
    if (kind == KIND_F32)
      ((float*)out)[j] = x;
    else if (kind == KIND_SQ_F32)
      ((float*)out)[j] = x * x;
    else
      ((uint16_t*)out)[j] = upper16(x);
  }
  return 0;
}
