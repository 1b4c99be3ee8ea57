/* Host implementation of the counter-based normal generator defined in synth/__init__.py, for
 * large host-side draws: splitmix64 output function over key + (i + 1) * golden, Box-Muller on
 * the two 32-bit halves in fp64, mean + std * z, then fp64 -> fp32 -> 16-bit storage type with
 * round-to-nearest-even at each step.  The range is split over threads; every element depends
 * only on its index, so the split does not change any value.  Built without floating-point
 * contraction so each operation rounds as numpy's does.  Synthetic-input plumbing only: it holds
 * none of the decode step's arithmetic. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* fp32 -> bf16 bits, nearest-even: add 0x7fff plus the lowest kept bit, keep the top half. */
static uint16_t to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* fp32 -> IEEE binary16 bits, nearest-even (normal, subnormal, overflow to infinity). */
static uint16_t to_f16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  const uint32_t sign = (u >> 16) & 0x8000u;
  const uint32_t absu = u & 0x7FFFFFFFu;
  if (absu >= 0x7F800000u) return (uint16_t)(sign | (absu > 0x7F800000u ? 0x7E00u : 0x7C00u));
  const int e = (int)(absu >> 23) - 127 + 15;
  uint32_t mant = (absu & 0x7FFFFFu) | 0x800000u;
  if (e >= 31) return (uint16_t)(sign | 0x7C00u);
  if (e <= 0) { /* subnormal half: shift the 24-bit significand right by 14 - e */
    const int shift = 14 - e;
    if (shift > 24) return (uint16_t)sign;
    const uint32_t kept = mant >> shift, rem = mant & ((1u << shift) - 1u), halfw = 1u << (shift - 1);
    uint32_t r = kept + ((rem > halfw || (rem == halfw && (kept & 1u))) ? 1u : 0u);
    return (uint16_t)(sign | r);
  }
  const uint32_t kept = mant >> 13, rem = mant & 0x1FFFu;
  uint32_t r = ((uint32_t)e << 10) + (kept & 0x3FFu);
  if (rem > 0x1000u || (rem == 0x1000u && (kept & 1u))) r += 1u; /* a carry may reach infinity */
  return (uint16_t)(sign | r);
}

typedef struct {
  uint16_t* dst;
  uint64_t lo, hi, key, offset;
  double mean, std_;
  int is_bf16;
} job_t;

static void* run(void* arg) {
  const job_t* j = (const job_t*)arg;
  for (uint64_t i = j->lo; i < j->hi; ++i) {
    const uint64_t w = mix64(j->key + (j->offset + i + 1) * 0x9E3779B97F4A7C15ull);
    const double u1 = ((double)(w >> 32) + 1.0) * (1.0 / 4294967296.0);
    const double u2 = (double)(w & 0xFFFFFFFFull) * (1.0 / 4294967296.0);
    const double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
    const double s = j->std_ * z;
    const float v = (float)(j->mean + s);
    j->dst[i] = j->is_bf16 ? to_bf16(v) : to_f16(v);
  }
  return NULL;
}

int synth_fill_normal_host(void* dst, unsigned long long count, unsigned long long key,
                           unsigned long long offset, double mean, double std_, int is_bf16,
                           int threads) {
  if (count == 0) return 0;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  job_t jobs[256];
  const uint64_t per = (count + (uint64_t)threads - 1) / (uint64_t)threads;
  int started = 0;
  for (int t = 0; t < threads; ++t) {
    const uint64_t lo = per * (uint64_t)t;
    if (lo >= count) break;
    jobs[t].dst = (uint16_t*)dst;
    jobs[t].lo = lo;
    jobs[t].hi = lo + per < count ? lo + per : count;
    jobs[t].key = key;
    jobs[t].offset = offset;
    jobs[t].mean = mean;
    jobs[t].std_ = std_;
    jobs[t].is_bf16 = is_bf16;
    if (pthread_create(&tid[t], NULL, run, &jobs[t]) != 0) { /* run the rest here */
      run(&jobs[t]);
      for (int u = t + 1; u < threads && per * (uint64_t)u < count; ++u) {
        jobs[u] = jobs[t];
        jobs[u].lo = per * (uint64_t)u;
        jobs[u].hi = jobs[u].lo + per < count ? jobs[u].lo + per : count;
        run(&jobs[u]);
      }
      break;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  return 0;
}
