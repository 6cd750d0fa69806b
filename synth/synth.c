/*
 * Seeded, counter-based synthetic tensor generator.
 *
 * This file holds no convolution arithmetic. It only turns (seed, tensor id,
 * flat element index) into a value, so that any slice of any tensor can be
 * regenerated on its own (a >4 GB input is produced sample by sample, with no
 * full host copy). Both the CPU oracle's tests and the GPU path's tests draw
 * their inputs from here; neither side generates inputs by itself.
 *
 * Definition (the single source of truth for every stored input):
 *   mix(z)      = the SplitMix64 output function (Steele, Lea, Flood,
 *                 "Fast splittable pseudorandom number generators", 2014):
 *                 z += 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
 *                 z = (z ^ z>>27) * 0x94D049BB133111EB; return z ^ z>>31.
 *   key         = mix(mix(seed) ^ (tensor_id * 0xD1B54A32D192ED03))
 *   bits(i)     = mix(key + i * 0x9E3779B97F4A7C15)
 *   u53(i)      = (bits(i) >> 11) * 2^-53                  in [0, 1)
 *   uniform     : v = lo + (hi - lo) * u53(i)
 *   normal      : pair j = i / 2 uses u1 = 1 - u53(2j), u2 = u53(2j + 1);
 *                 rad = sqrt(-2 ln u1); v = sigma * rad * (i even ? cos : sin)(2 pi u2)
 *                 (the Box-Muller transform, Box & Muller 1958)
 *   stored      : float(v) by round-to-nearest-even, then for 16-bit targets
 *                 bf16 / fp16 by round-to-nearest-even from that float.
 *   integers    : v = lo + (bits(i) % (hi - lo + 1)), stored exactly (small
 *                 integer-valued tensors for exact-arithmetic tests).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { SYNTH_F32 = 0, SYNTH_BF16 = 1, SYNTH_F16 = 2 };
enum { SYNTH_UNIFORM = 0, SYNTH_NORMAL = 1, SYNTH_INTEGER = 2 };

static inline uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(mix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03ull));
}

static inline uint64_t bits_at(uint64_t key, uint64_t i) {
  return mix64(key + i * 0x9E3779B97F4A7C15ull);
}

static inline double u53(uint64_t b) { return (double)(b >> 11) * 0x1.0p-53; }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u);
  uint32_t lsb = (x >> 16) & 1u;
  x += 0x7fffu + lsb;
  return (uint16_t)(x >> 16);
}

static inline uint16_t f32_to_f16_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7fffffffu;
  if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);
  if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* >= 65520 rounds to inf */
  uint32_t e = ax >> 23;
  if (e >= 113u) { /* normal half */
    uint32_t m = ax & 0x7fffffu;
    uint32_t h = ((e - 112u) << 10) | (m >> 13);
    uint32_t rem = m & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
  }
  if (e == 0u) return (uint16_t)sign; /* float subnormal: far below half range */
  /* half subnormal: value = M * 2^(e-150), unit 2^-24 -> M >> (126 - e) */
  uint32_t m = (ax & 0x7fffffu) | 0x800000u;
  uint32_t sh = 126u - e;
  if (sh > 24u) return (uint16_t)sign;
  uint32_t q = m >> sh;
  uint32_t rem = m & ((1u << sh) - 1u);
  uint32_t half = 1u << (sh - 1u);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  return (uint16_t)(sign | q);
}

static double value_at(uint64_t key, uint64_t i, int dist, double a, double b) {
  if (dist == SYNTH_UNIFORM) return a + (b - a) * u53(bits_at(key, i));
  if (dist == SYNTH_INTEGER) {
    int64_t lo = (int64_t)a, hi = (int64_t)b;
    uint64_t span = (uint64_t)(hi - lo) + 1u;
    return (double)(lo + (int64_t)(bits_at(key, i) % span));
  }
  uint64_t j = i >> 1;
  double u1 = 1.0 - u53(bits_at(key, 2 * j));
  double u2 = u53(bits_at(key, 2 * j + 1));
  double rad = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586476925286766559 * u2;
  /* a = mean, b = standard deviation */
  return a + b * rad * ((i & 1u) ? sin(ang) : cos(ang));
}

typedef struct {
  void* out;
  uint64_t begin, end;   /* local element range [begin, end) */
  uint64_t offset;       /* global index of local element 0 */
  uint64_t key;
  int dtype, dist;
  double a, b;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  for (uint64_t e = j->begin; e < j->end; ++e) {
    float f = (float)value_at(j->key, j->offset + e, j->dist, j->a, j->b);
    if (j->dtype == SYNTH_F32) {
      ((float*)j->out)[e] = f;
    } else if (j->dtype == SYNTH_BF16) {
      ((uint16_t*)j->out)[e] = f32_to_bf16_rne(f);
    } else {
      ((uint16_t*)j->out)[e] = f32_to_f16_rne(f);
    }
  }
  return NULL;
}

/*
 * Fill out[0..count) with elements offset..offset+count of tensor
 * (seed, tensor_id). dist: 0 uniform [a, b); 1 normal (mean a, std b);
 * 2 integers in [a, b]. Returns 0 on success, -1 on a bad argument.
 */
int synth_fill(void* out, uint64_t count, int dtype, int dist, double a, double b,
               uint64_t seed, uint64_t tensor_id, uint64_t offset, int nthreads) {
  if (!out && count) return -1;
  if (dtype < 0 || dtype > 2 || dist < 0 || dist > 2) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (count < 65536u) nthreads = 1;
  uint64_t key = synth_key(seed, tensor_id);
  fill_job jobs[256];
  pthread_t tids[256];
  int started[256];
  uint64_t per = (count + (uint64_t)nthreads - 1u) / (uint64_t)nthreads;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t lo = per * (uint64_t)t, hi = lo + per;
    if (lo > count) lo = count;
    if (hi > count) hi = count;
    jobs[t] = (fill_job){out, lo, hi, offset, key, dtype, dist, a, b};
    started[t] = (t > 0) && pthread_create(&tids[t], NULL, fill_worker, &jobs[t]) == 0;
  }
  fill_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t]) pthread_join(tids[t], NULL);
    else fill_worker(&jobs[t]);
  }
  return 0;
}

/* Conversions exposed for tests of the storage rounding itself. */
uint16_t synth_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
uint16_t synth_f32_to_f16(float f) { return f32_to_f16_rne(f); }
