/*
 * inputgen.c - seeded synthetic inputs shared by the oracle side and the
 * CUDA side of the tests and the benchmark.
 *
 * It holds none of the Command method's arithmetic: only random numbers.
 *
 * Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used counter-based: element
 * i of a stream is the (i+1)-th output of a SplitMix64 whose state starts at
 * the stream key, i.e. mix(key + (i + 1) * gamma). Every element depends only
 * on (seed, stream, i), so any split of the index range over threads gives
 * the same bytes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define IG_GAMMA 0x9e3779b97f4a7c15ull

/* SplitMix64 output function applied to a state value. */
static uint64_t ig_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

/* Key of stream `stream` under `seed`: the first output of a SplitMix64
 * seeded with seed ^ (stream * odd constant). */
uint64_t ig_stream_key(uint64_t seed, uint64_t stream) {
  return ig_mix((seed ^ (stream * 0xd1b54a32d192ed03ull)) + IG_GAMMA);
}

/* The i-th 64-bit output of a stream. */
uint64_t ig_bits(uint64_t key, uint64_t i) { return ig_mix(key + (i + 1) * IG_GAMMA); }

/* ---- distributions ----------------------------------------------------- */

enum { IG_U32 = 0, IG_UNIFORM_F32 = 1, IG_NORMAL_F32 = 2, IG_UNIFORM_BF16_TRUNC = 3 };

/* uniform in [0,1) with 24 random bits */
static double u24(uint64_t z) { return ldexp((double)(z >> 40), -24); }
/* uniform in (0,1] and [0,1) with 53 random bits */
static double u53_open0(uint64_t z) { return ldexp((double)((z >> 11) + 1), -53); }
static double u53(uint64_t z) { return ldexp((double)(z >> 11), -53); }

static float uniform_f32(uint64_t key, int64_t i, double lo, double hi) {
  return (float)(lo + (hi - lo) * u24(ig_bits(key, (uint64_t)i)));
}

/* Box-Muller: element i uses outputs 2i and 2i+1 of the stream. */
static float normal_f32(uint64_t key, int64_t i) {
  double u1 = u53_open0(ig_bits(key, 2 * (uint64_t)i));
  double u2 = u53(ig_bits(key, 2 * (uint64_t)i + 1));
  return (float)(sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2));
}

typedef struct {
  int kind;
  uint64_t key;
  double lo, hi;
  void* out;
  int64_t begin, end;
} ig_job;

static void run_job(const ig_job* j) {
  switch (j->kind) {
    case IG_U32: {
      uint32_t* o = (uint32_t*)j->out;
      for (int64_t i = j->begin; i < j->end; ++i) o[i] = (uint32_t)ig_bits(j->key, (uint64_t)i);
      break;
    }
    case IG_UNIFORM_F32: {
      float* o = (float*)j->out;
      for (int64_t i = j->begin; i < j->end; ++i) o[i] = uniform_f32(j->key, i, j->lo, j->hi);
      break;
    }
    case IG_NORMAL_F32: {
      float* o = (float*)j->out;
      for (int64_t i = j->begin; i < j->end; ++i) o[i] = normal_f32(j->key, i);
      break;
    }
    case IG_UNIFORM_BF16_TRUNC: {
      /* a binary32 uniform draw, truncated toward zero to its upper 16 bits */
      uint16_t* o = (uint16_t*)j->out;
      for (int64_t i = j->begin; i < j->end; ++i) {
        float f = uniform_f32(j->key, i, j->lo, j->hi);
        uint32_t u;
        memcpy(&u, &f, 4);
        o[i] = (uint16_t)(u >> 16);
      }
      break;
    }
  }
}

static void* thread_main(void* arg) {
  run_job((const ig_job*)arg);
  return NULL;
}

/* Fill out[0..n) with elements [0, n) of stream (seed, stream) drawn from
 * distribution `kind` (lo/hi used by the uniform kinds), on up to `threads`
 * threads. Returns 0, or -1 on a bad argument. */
int ig_fill(int kind, uint64_t seed, uint64_t stream, double lo, double hi, void* out,
            int64_t n, int threads) {
  if (kind < IG_U32 || kind > IG_UNIFORM_BF16_TRUNC || n < 0 || (n > 0 && !out)) return -1;
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if (n < (int64_t)threads * 65536) threads = 1;
  uint64_t key = ig_stream_key(seed, stream);
  ig_job jobs[64];
  pthread_t tid[64];
  int started[64];
  for (int t = 0; t < threads; ++t) {
    jobs[t].kind = kind;
    jobs[t].key = key;
    jobs[t].lo = lo;
    jobs[t].hi = hi;
    jobs[t].out = out;
    jobs[t].begin = n * t / threads;
    jobs[t].end = n * (t + 1) / threads;
    started[t] = 0;
  }
  for (int t = 1; t < threads; ++t)
    started[t] = pthread_create(&tid[t], NULL, thread_main, &jobs[t]) == 0;
  run_job(&jobs[0]);
  for (int t = 1; t < threads; ++t) {
    if (started[t])
      pthread_join(tid[t], NULL);
    else
      run_job(&jobs[t]);
  }
  return 0;
}
