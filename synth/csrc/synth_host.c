/* synth_host.c - host-side standard-normal draws for the synthetic inputs.
 *
 * The same counter-based definition as synth/rng.py, written in C and spread
 * over threads so that the ~10^8 draws of a multi-hundred-megabyte fp8 cache
 * take a second instead of a minute:
 *
 *   splitmix64(x): z = x + 0x9E3779B97F4A7C15;
 *                  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                  z = (z ^ (z >> 27)) * 0x94D049BB133111EB;  z ^ (z >> 31)
 *   key          = splitmix64(splitmix64(seed) ^ stream)
 *   uniform01(i) = (splitmix64(key ^ i) >> 11) * 2^-53
 *   normal(i)    = sqrt(-2 log1p(-uniform01(2i))) * cos(2 pi uniform01(2i+1))
 *
 * (SplitMix64: Steele, Lea and Flood, OOPSLA 2014; Box-Muller transform.)
 * Holds no attention arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline double uniform01(uint64_t key, uint64_t i) {
  return (double)(splitmix64(key ^ i) >> 11) * 0x1p-53;
}

typedef struct {
  uint64_t key, start, n;
  double* out;
} span_t;

static void* run_span(void* arg) {
  const span_t* s = (const span_t*)arg;
  const double two_pi = 2.0 * 3.14159265358979311600;  /* the double nearest pi, times 2 */
  for (uint64_t k = 0; k < s->n; ++k) {
    const uint64_t i = s->start + k;
    const double r0 = uniform01(s->key, 2 * i);
    const double r1 = uniform01(s->key, 2 * i + 1);
    s->out[k] = sqrt(-2.0 * log1p(-r0)) * cos(two_pi * r1);
  }
  return 0;
}

/* Standard normals for counters start .. start+n-1 into out[0..n), on up to
 * `threads` threads.  Returns 0. */
int synth_normal(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, double* out, int threads) {
  const uint64_t key = splitmix64(splitmix64(seed) ^ stream);
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if (n < 65536) threads = 1;
  pthread_t tid[64];
  span_t sp[64];
  const uint64_t per = (n + (uint64_t)threads - 1) / (uint64_t)threads;
  int made = 0;
  for (int t = 0; t < threads; ++t) {
    const uint64_t a = (uint64_t)t * per;
    if (a >= n) break;
    sp[t].key = key;
    sp[t].start = start + a;
    sp[t].n = (a + per <= n) ? per : n - a;
    sp[t].out = out + a;
    if (t == 0) continue;
    if (pthread_create(&tid[t], 0, run_span, &sp[t]) != 0) {
      run_span(&sp[t]);       /* no thread: do the span here */
      sp[t].n = 0;
    }
    made = t + 1;
  }
  run_span(&sp[0]);
  for (int t = 1; t < made; ++t)
    if (sp[t].n) pthread_join(tid[t], 0);
  return 0;
}

/* Uniform integers in [lo, hi] as two's-complement bytes for counters
 * start .. start+n-1:  lo + (((splitmix64(key ^ i) >> 32) * (hi - lo + 1)) >> 32)
 * (the multiply-shift draw of synth/rng.py and of the device generator,
 * integer arithmetic throughout, so the bytes are identical on every side). */
typedef struct {
  uint64_t key, start, n, range;
  int64_t lo;
  uint8_t* out;
} ispan_t;

static void* run_ispan(void* arg) {
  const ispan_t* s = (const ispan_t*)arg;
  for (uint64_t k = 0; k < s->n; ++k) {
    const uint64_t hi32 = splitmix64(s->key ^ (s->start + k)) >> 32;
    const int64_t v = s->lo + (int64_t)((hi32 * s->range) >> 32);
    s->out[k] = (uint8_t)(v & 0xFF);
  }
  return 0;
}

int synth_uniform_i8(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, int32_t lo,
                     int32_t hi, uint8_t* out, int threads) {
  const uint64_t key = splitmix64(splitmix64(seed) ^ stream);
  if (hi < lo || lo < -128 || hi > 127) return 1;
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if (n < (1u << 20)) threads = 1;
  pthread_t tid[64];
  ispan_t sp[64];
  const uint64_t per = (n + (uint64_t)threads - 1) / (uint64_t)threads;
  int made = 0;
  for (int t = 0; t < threads; ++t) {
    const uint64_t a = (uint64_t)t * per;
    if (a >= n) break;
    sp[t].key = key;
    sp[t].start = start + a;
    sp[t].n = (a + per <= n) ? per : n - a;
    sp[t].range = (uint64_t)(hi - lo + 1);
    sp[t].lo = lo;
    sp[t].out = out + a;
    if (t == 0) continue;
    if (pthread_create(&tid[t], 0, run_ispan, &sp[t]) != 0) {
      run_ispan(&sp[t]);
      sp[t].n = 0;
    }
    made = t + 1;
  }
  run_ispan(&sp[0]);
  for (int t = 1; t < made; ++t)
    if (sp[t].n) pthread_join(tid[t], 0);
  return 0;
}
