/*
 * Seeded, counter-based input generator for the fused MoE layer workloads.
 *
 * This file holds no arithmetic of the MoE method itself: it only turns
 * (seed, stream, index) into pseudo-random numbers.  Both the CUDA path's
 * callers (bench, tests) and the CPU oracle's callers get their inputs from
 * here, so that the two sides see bit-identical tensors.
 *
 * Definition (one value per element index i of a tensor):
 *   mix64(z)      = the splitmix64 output finaliser (Steele, Lea, Flood,
 *                   "Fast splittable pseudorandom number generators",
 *                   OOPSLA 2014; constants as published by S. Vigna):
 *                     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                     z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                     z =  z ^ (z >> 31)
 *   base(seed,s)  = mix64(seed ^ (s * 0xD1B54A32D192ED03))
 *   r(c)          = mix64(base + (c + 1) * 0x9E3779B97F4A7C15)
 *   U(c)          = ((r(c) >> 11) + 1) * 2^-53          in (0, 1]
 *   Box-Muller on the pair p = i / 2 (Box & Muller 1958):
 *     rad = sqrt(-2 ln U(2p)),  th = 2 pi U(2p+1)
 *     z(2p) = rad cos th,  z(2p+1) = rad sin th
 *   value(i) = mean + std * z(i)  (double), then
 *     fp32 tensors: rounded to float (round to nearest even),
 *     bf16 tensors: rounded to float, then to bf16 (round to nearest even).
 *
 * Work is split over POSIX threads by contiguous index ranges; the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GEN_PI 3.14159265358979323846

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return mix64(seed ^ (stream * 0xD1B54A32D192ED03ULL));
}

static double uniform01(uint64_t base, uint64_t c) {
  uint64_t r = mix64(base + (c + 1) * 0x9E3779B97F4A7C15ULL);
  return (double)((r >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static double normal_at(uint64_t base, uint64_t i) {
  uint64_t p = i >> 1;
  double u1 = uniform01(base, 2 * p);
  double u2 = uniform01(base, 2 * p + 1);
  double rad = sqrt(-2.0 * log(u1));
  double th = 2.0 * GEN_PI * u2;
  return (i & 1) ? rad * sin(th) : rad * cos(th);
}

static uint16_t float_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf/nan: never produced */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint64_t base;
  uint64_t lo, hi;
  double mean, std;
  void* out;
  int kind; /* 0 = bf16, 1 = f32, 2 = raw uint64 */
} gen_job;

static void store_value(gen_job* j, uint64_t i, double z) {
  float f = (float)(j->mean + j->std * z);
  if (j->kind == 0)
    ((uint16_t*)j->out)[i] = float_to_bf16_bits(f);
  else
    ((float*)j->out)[i] = f;
}

static void* gen_worker(void* arg) {
  gen_job* j = (gen_job*)arg;
  uint64_t i = j->lo;
  if (j->kind == 2) {
    for (; i < j->hi; ++i) ((uint64_t*)j->out)[i] = mix64(j->base + (i + 1) * 0x9E3779B97F4A7C15ULL);
    return NULL;
  }
  if (i < j->hi && (i & 1)) { /* odd start: second half of a pair */
    store_value(j, i, normal_at(j->base, i));
    ++i;
  }
  for (; i + 1 < j->hi; i += 2) { /* whole pairs: one log/sqrt for both values */
    uint64_t p = i >> 1;
    double u1 = uniform01(j->base, 2 * p);
    double u2 = uniform01(j->base, 2 * p + 1);
    double rad = sqrt(-2.0 * log(u1));
    double th = 2.0 * GEN_PI * u2;
    store_value(j, i, rad * cos(th));
    store_value(j, i + 1, rad * sin(th));
  }
  if (i < j->hi) store_value(j, i, normal_at(j->base, i));
  return NULL;
}

static int run_jobs(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                    void* out, int kind, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n / 4096 + 1) nthreads = (int)(n / 4096 + 1);
  gen_job jobs[256];
  pthread_t tids[256];
  uint64_t base = stream_base(seed, stream);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].base = base;
    jobs[t].lo = n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].hi = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    jobs[t].mean = mean;
    jobs[t].std = std;
    jobs[t].out = out;
    jobs[t].kind = kind;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, gen_worker, &jobs[t]) != 0) break;
    started = t;
  }
  gen_worker(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) gen_worker(&jobs[t]); /* threads that failed to start */
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  return 0;
}

/* n normal values with the given mean and std, as raw bf16 bits. */
int moe_gen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                        uint16_t* out, int nthreads) {
  return run_jobs(seed, stream, n, mean, std, out, 0, nthreads);
}

/* n normal values with the given mean and std, as fp32. */
int moe_gen_normal_f32(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                       float* out, int nthreads) {
  return run_jobs(seed, stream, n, mean, std, out, 1, nthreads);
}

/* n raw 64-bit words r(0..n-1) of the stream (used for permutations). */
int moe_gen_u64(uint64_t seed, uint64_t stream, uint64_t n, uint64_t* out, int nthreads) {
  return run_jobs(seed, stream, n, 0.0, 0.0, out, 2, nthreads);
}
