/*
 * Seeded, counter-based synthetic input generator.
 *
 * This module produces the random inputs (queries, subkeys, value rows) that
 * both the fp64 oracle and the CUDA path consume.  It holds none of the
 * product-key lookup arithmetic: it only turns (seed, tensor id, element
 * index) into numbers.
 *
 * Definition (so any other implementation can reproduce the bits):
 *   mix(z)       = SplitMix64 output finaliser (Steele, Lea & Flood 2014):
 *                  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                  z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   base(s, t)   = mix(mix(s) + t)                 (s = seed, t = tensor id)
 *   r_i          = mix(base + (i + 1) * 0x9E3779B97F4A7C15)
 *                  i.e. the (i+1)-th output of a SplitMix64 stream whose
 *                  state starts at base.
 *   normal_i     = sqrt(-2 ln u1) * cos(2 pi u2)   (Box-Muller, one output)
 *                  u1 = (hi32(r_i) + 0.5) / 2^32, u2 = (lo32(r_i) + 0.5) / 2^32
 *   uniform_i    = ((r_i >> 11) + 0.5) / 2^53
 * A value drawn "N(mean, var)" is (float)(mean + sqrt(var) * normal_i); a
 * bf16 value is that float rounded to nearest-even on its upper 16 bits.
 *
 * Work is split over POSIX threads by element range; the result does not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_base(uint64_t seed, uint64_t tensor_id) {
  return mix64(mix64(seed) + tensor_id);
}

static inline uint64_t draw(uint64_t base, uint64_t i) {
  return mix64(base + (i + 1) * SM64_GAMMA);
}

static inline double normal_of(uint64_t r) {
  const double two32 = 4294967296.0;
  double u1 = ((double)(r >> 32) + 0.5) / two32;
  double u2 = ((double)(r & 0xffffffffULL) + 0.5) / two32;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

static inline double uniform_of(uint64_t r) {
  return ((double)(r >> 11) + 0.5) / 9007199254740992.0;
}

static inline uint16_t bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- threads */

typedef struct {
  int kind; /* 0 normal f32, 1 normal bf16, 2 mixture bf16, 3 uniform f64 */
  uint64_t base, base2, base3;
  int64_t lo, hi, offset;
  double mean, sd;
  void *out;
  /* mixture */
  const double *cdf;
  int n_comp;
  int64_t row_len;
  double comp_sd;
  int32_t *comp_out;
} job_t;

static int pick_component(const double *cdf, int n_comp, double u) {
  for (int c = 0; c < n_comp; ++c)
    if (u < cdf[c]) return c;
  return n_comp - 1;
}

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  for (int64_t e = j->lo; e < j->hi; ++e) {
    uint64_t i = (uint64_t)(e + j->offset);
    switch (j->kind) {
      case 0:
        ((float *)j->out)[e] = (float)(j->mean + j->sd * normal_of(draw(j->base, i)));
        break;
      case 1:
        ((uint16_t *)j->out)[e] = bf16_rne((float)(j->mean + j->sd * normal_of(draw(j->base, i))));
        break;
      case 2: {
        /* element i = row * row_len + t; the row's component comes from the
           uniform stream base2 at the row index, its mean from stream base3
           at (component * row_len + t), its noise from stream base at i. */
        int64_t row = (int64_t)i / j->row_len, t = (int64_t)i % j->row_len;
        int c = pick_component(j->cdf, j->n_comp, uniform_of(draw(j->base2, (uint64_t)row)));
        double mu = normal_of(draw(j->base3, (uint64_t)c * (uint64_t)j->row_len + (uint64_t)t));
        double x = mu + j->comp_sd * normal_of(draw(j->base, i));
        ((uint16_t *)j->out)[e] = bf16_rne((float)x);
        if (j->comp_out && t == 0) j->comp_out[row - j->offset / j->row_len] = c;
        break;
      }
      case 3:
        ((double *)j->out)[e] = uniform_of(draw(j->base, i));
        break;
    }
  }
  return NULL;
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void run_parallel(job_t proto, int64_t n, int nthreads) {
  nthreads = resolve_threads(nthreads);
  if (n < 65536 || nthreads == 1) {
    proto.lo = 0;
    proto.hi = n;
    run_job(&proto);
    return;
  }
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  job_t jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  int launched = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].lo = (int64_t)t * per;
    jobs[t].hi = jobs[t].lo + per < n ? jobs[t].lo + per : n;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0) {
      run_job(&jobs[t]);
      th[t] = 0;
    }
    launched = t + 1;
  }
  for (int t = 0; t < launched; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ API */

/* Elements [offset, offset+n) of the N(mean, sd^2) stream (seed, tensor_id), as fp32. */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t offset, int64_t n,
                      double mean, double sd, float *out, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = 0;
  j.base = stream_base(seed, tensor_id);
  j.offset = offset;
  j.mean = mean;
  j.sd = sd;
  j.out = out;
  run_parallel(j, n, nthreads);
}

/* Same stream, each value rounded to bf16 (raw bits). */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, int64_t offset, int64_t n,
                       double mean, double sd, uint16_t *out, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = 1;
  j.base = stream_base(seed, tensor_id);
  j.offset = offset;
  j.mean = mean;
  j.sd = sd;
  j.out = out;
  run_parallel(j, n, nthreads);
}

/* Uniform(0,1) doubles from stream (seed, tensor_id). */
void synth_uniform_f64(uint64_t seed, uint64_t tensor_id, int64_t offset, int64_t n,
                       double *out, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = 3;
  j.base = stream_base(seed, tensor_id);
  j.offset = offset;
  j.out = out;
  run_parallel(j, n, nthreads);
}

/*
 * Gaussian-mixture rows, as bf16.  Rows are row_len long; rows
 * [offset/row_len, ...) are produced, n elements in all (offset and n must be
 * multiples of row_len).  Component weights are Zipf: p_c proportional to
 * (c+1)^-zipf_s for c = 0..n_comp-1.  Component means are N(0,1) per element
 * (stream tensor_id_mean), the row's component is drawn from the uniform
 * stream tensor_id_pick at the row index, and the value is
 * mean + comp_sd * N(0,1) (stream tensor_id_noise at the element index).
 * If comp_out is not NULL it receives each produced row's component.
 */
int synth_mixture_bf16(uint64_t seed, uint64_t tensor_id_noise, uint64_t tensor_id_mean,
                       uint64_t tensor_id_pick, int64_t row_len, int64_t offset, int64_t n,
                       int n_comp, double zipf_s, double comp_sd, uint16_t *out,
                       int32_t *comp_out, int nthreads) {
  if (row_len <= 0 || n_comp <= 0 || n_comp > 4096) return -1;
  if (offset % row_len || n % row_len) return -1;
  double *cdf = (double *)malloc(sizeof(double) * (size_t)n_comp);
  if (!cdf) return -2;
  double tot = 0.0;
  for (int c = 0; c < n_comp; ++c) tot += pow((double)(c + 1), -zipf_s);
  double acc = 0.0;
  for (int c = 0; c < n_comp; ++c) {
    acc += pow((double)(c + 1), -zipf_s) / tot;
    cdf[c] = acc;
  }
  cdf[n_comp - 1] = 1.0;
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = 2;
  j.base = stream_base(seed, tensor_id_noise);
  j.base2 = stream_base(seed, tensor_id_pick);
  j.base3 = stream_base(seed, tensor_id_mean);
  j.offset = offset;
  j.cdf = cdf;
  j.n_comp = n_comp;
  j.row_len = row_len;
  j.comp_sd = comp_sd;
  j.out = out;
  j.comp_out = comp_out;
  run_parallel(j, n, nthreads);
  free(cdf);
  return 0;
}

/* fp32 -> bf16 round-to-nearest-even, exposed for tests of the rounding rule. */
void synth_f32_to_bf16(const float *in, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_rne(in[i]);
}

uint64_t synth_draw_u64(uint64_t seed, uint64_t tensor_id, uint64_t i) {
  return draw(stream_base(seed, tensor_id), i);
}
