/*
 * Seeded synthetic inputs for the top-k routed MoE feed-forward layer.
 *
 * This file holds only random-number generation: none of the layer's arithmetic
 * lives here.  Both the CPU oracle (through the tests) and the CUDA path (through
 * the tests, smoke check and benchmark) receive buffers produced by these
 * functions, so the two sides never generate their own inputs.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  The value for counter i of a
 * stream is the SplitMix64 finaliser applied to key + (i + 1) * GOLDEN, where
 * key is itself the finaliser applied to seed + (tensor_id + 1) * GOLDEN.  Any
 * element can therefore be produced on its own, which lets a test regenerate a
 * prefix of a batch or a single expert's weights.
 *
 * Normal samples: Box-Muller (Box & Muller, 1958) in double precision on the
 * pair (u1, u2) taken from counters 2p and 2p+1; element 2p takes r*cos, element
 * 2p+1 takes r*sin.  The double result is scaled, rounded to float, and (for
 * bf16 tensors) rounded again to bf16 with round-to-nearest-even.
 *
 * Compiled with -ffp-contract=off so x86-64 and aarch64 hosts round alike.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define TWO_PI 6.283185307179586476925286766559

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint32_t tensor_id) {
  return mix64(seed + ((uint64_t)tensor_id + 1ULL) * GOLDEN);
}

static inline uint64_t counter_bits(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1ULL) * GOLDEN);
}

/* uniform double in (0, 1] */
static inline double u01_open0(uint64_t b) { return ((double)(b >> 11) + 1.0) * 0x1.0p-53; }
/* uniform double in [0, 1) */
static inline double u01_open1(uint64_t b) { return (double)(b >> 11) * 0x1.0p-53; }

static inline double normal_at(uint64_t key, uint64_t n) {
  uint64_t p = n >> 1;
  double u1 = u01_open0(counter_bits(key, 2 * p));
  double u2 = u01_open1(counter_bits(key, 2 * p + 1));
  double r = sqrt(-2.0 * log(u1));
  double th = TWO_PI * u2;
  return (n & 1) ? r * sin(th) : r * cos(th);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint64_t key, start, begin, end;
  double std;
  int kind; /* 0: bf16 normal, 1: f32 normal, 2: f32 uniform [lo,hi), 3: i32 uniform [lo,hi) */
  double lo, hi;
  void* out;
} job_t;

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  uint64_t n = j->begin;
  if (j->kind <= 1) {
    /* normal samples come in Box-Muller pairs: produce both halves of a pair at once */
    while (n < j->end) {
      uint64_t c = j->start + n;
      uint64_t p = c >> 1;
      double u1 = u01_open0(counter_bits(j->key, 2 * p));
      double u2 = u01_open1(counter_bits(j->key, 2 * p + 1));
      double r = sqrt(-2.0 * log(u1));
      double th = TWO_PI * u2;
      double z[2] = {r * cos(th), r * sin(th)};
      for (uint64_t h = c & 1; h < 2 && n < j->end; ++h, ++n) {
        float v = (float)(j->std * z[h]);
        if (j->kind == 0) ((uint16_t*)j->out)[n] = f32_to_bf16_rne(v);
        else ((float*)j->out)[n] = v;
      }
    }
    return NULL;
  }
  for (; n < j->end; ++n) {
    uint64_t c = j->start + n;
    if (j->kind == 2) {
      ((float*)j->out)[n] = (float)(j->lo + (j->hi - j->lo) * u01_open1(counter_bits(j->key, c)));
    } else {
      uint64_t span = (uint64_t)(j->hi - j->lo);
      ((int32_t*)j->out)[n] = (int32_t)((int64_t)j->lo + (int64_t)(counter_bits(j->key, c) % span));
    }
  }
  return NULL;
}

static void fill(int kind, uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t count,
                 double std, double lo, double hi, void* out, int nthreads) {
  if (count == 0) return;
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > count / 65536 + 1) nthreads = (int)(count / 65536 + 1);
  job_t jobs[256];
  pthread_t th[256];
  uint64_t key = stream_key(seed, tensor_id);
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].key = key;
    jobs[i].start = start;
    jobs[i].begin = count * (uint64_t)i / (uint64_t)nthreads;
    jobs[i].end = count * (uint64_t)(i + 1) / (uint64_t)nthreads;
    jobs[i].std = std;
    jobs[i].kind = kind;
    jobs[i].lo = lo;
    jobs[i].hi = hi;
    jobs[i].out = out;
  }
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, run_job, &jobs[i]) != 0) break;
    started = i;
  }
  run_job(&jobs[0]);
  for (int i = started + 1; i < nthreads; ++i) run_job(&jobs[i]); /* threads that failed to start */
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
}

/* out[n] = bf16(float(std * N(0,1))) for counters start .. start+count-1 of (seed, tensor_id). */
void synth_normal_bf16(uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t count, double std,
                       uint16_t* out, int nthreads) {
  fill(0, seed, tensor_id, start, count, std, 0, 0, out, nthreads);
}

/* out[n] = float(std * N(0,1)). */
void synth_normal_f32(uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t count, double std,
                      float* out, int nthreads) {
  fill(1, seed, tensor_id, start, count, std, 0, 0, out, nthreads);
}

/* out[n] = float(lo + (hi - lo) * U[0,1)). */
void synth_uniform_f32(uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t count, double lo,
                       double hi, float* out, int nthreads) {
  fill(2, seed, tensor_id, start, count, 0, lo, hi, out, nthreads);
}

/* out[n] = lo + (bits mod (hi - lo)), an integer in [lo, hi). */
void synth_uniform_i32(uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t count, int64_t lo,
                       int64_t hi, int32_t* out, int nthreads) {
  if (hi <= lo) return;
  fill(3, seed, tensor_id, start, count, 0, (double)lo, (double)hi, out, nthreads);
}

/*
 * Zipf popularity bias: b[e] = coef * ln( (e+1)^(-s) / sum_{q=1..E} q^(-s) ).
 * Expert 0 is the most popular.  Computed in double, rounded to float.
 */
void synth_zipf_bias(int32_t E, double s, double coef, float* out) {
  double z = 0.0;
  for (int q = 1; q <= E; ++q) z += pow((double)q, -s);
  for (int e = 0; e < E; ++e) out[e] = (float)(coef * (-s * log((double)(e + 1)) - log(z)));
}

/*
 * Packed RL row: sequence lengths drawn in order from LogNormal(mu, sigma)
 * (normal counters of tensor_id), rounded to the nearest integer and clipped to
 * [lo, hi], appended until row_tokens tokens are filled; the last sequence is cut
 * at the row end.  Writes cu_seqlens[0..n] (cu_seqlens[0] = 0) and returns n, the
 * number of sequences, or -1 if max_seqs is too small.
 */
int32_t synth_packed_lengths(uint64_t seed, uint32_t tensor_id, double mu, double sigma, int32_t lo,
                             int32_t hi, int32_t row_tokens, int32_t* cu_seqlens, int32_t max_seqs) {
  uint64_t key = stream_key(seed, tensor_id);
  int32_t filled = 0, n = 0;
  cu_seqlens[0] = 0;
  for (uint64_t c = 0; filled < row_tokens; ++c) {
    if (n >= max_seqs) return -1;
    double len = exp(mu + sigma * normal_at(key, c));
    int64_t L = (int64_t)floor(len + 0.5);
    if (L < lo) L = lo;
    if (L > hi) L = hi;
    if (filled + L > row_tokens) L = row_tokens - filled;
    filled += (int32_t)L;
    cu_seqlens[++n] = filled;
  }
  return n;
}
