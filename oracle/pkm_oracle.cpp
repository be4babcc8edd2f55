// Plain, slow CPU oracle for the product-key memory (PKM) lookup forward pass.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file; only the tests, the package smoke check and the
// benchmark's CPU-baseline leg do.  It shares no code with the CUDA kernels.
//
// What it computes, with the passages it follows:
//   * Product-Key Memory, "Factorising the key space": a full key is the
//     concatenation (c1_a, c2_b) of one subkey from each half; its score
//     against q = (q1, q2) is q1.c1_a + q2.c2_b; the global top-k lies inside
//     top_k(half 1) x top_k(half 2), so k per-half winners per side, their k^2
//     pairwise sums and a top-k over those are exact.
//   * Product-Key Memory, code listing (forward): q.chunk(2) gives q1 = first
//     half, q2 = second half; flat index = i1 * n_keys + i2; the winners'
//     scores go through a softmax and weight an EmbeddingBag(mode="sum") read
//     of the value table.
//   * Memory Retrieval Mechanisms, "top-k retrieval" equations: alpha_j =
//     softmax over the k selected scores, r = sum_j alpha_j v_{i_j}.
// Readings where the pages are silent (all stated in the design notes):
//   ties -> lower subkey index per half and lower flat index overall; no
//   softmax temperature; several heads each score their own subkeys with their
//   own query slice, share one value table, and their reads are summed.
//
// Low-precision value table (the note after the code listing calls the
// value table "a good candidate for keeping in a lower precision"): rows of
// fp8 e4m3 codes with one fp32 scale per row.  e4m3 as defined by the OCP 8-bit
// floating point format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
// bits; exponent field 0 is subnormal (2^-6 * m/8); the all-ones pattern
// S.1111.111 is NaN and there are no infinities (largest finite 448).  The
// quantiser (a reading: the page fixes no recipe) takes per row
// scale = max(amax / 448, FLT_MIN) in fp32, amax = the row's largest |x|, and
// code = the e4m3 value nearest to x / scale (fp32 division), ties to the even
// mantissa, saturated to +-448.  The fp8 read dequantises exactly in double.
//
// Arithmetic: inputs are widened exactly to double (bf16 and fp32 are both
// subsets of double); every dot product is one sequential loop in double;
// the softmax uses std::exp after subtracting the largest selected score.
// Sorting uses std::sort with an explicit total order.  Parallelism is over
// independent (query, head) pairs only and never changes any arithmetic.
// Parity pins: every function here is pinned by tests (brute force over all
// n_keys^2 keys, closed forms, hand-worked cases); none is "parity unpinned".

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORC_F32 = 0, ORC_BF16 = 1 };

inline double widen(const void* base, int dtype, int64_t i) {
  if (dtype == ORC_F32) return (double)static_cast<const float*>(base)[i];
  uint32_t bits = (uint32_t) static_cast<const uint16_t*>(base)[i] << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

struct Cand {
  double score;
  int64_t flat;
};

// (score desc, flat asc): a strict total order on distinct flat indices.
inline bool cand_before(const Cand& x, const Cand& y) {
  if (x.score != y.score) return x.score > y.score;
  return x.flat < y.flat;
}

// s[a] = sum_t q[b,h,half*D/2 + t] * C[h,half,a,t], one sequential loop each.
void subkey_scores(const void* q, int qdt, const void* C, int cdt, int H, int d_q, int n,
                   int64_t b, int h, int half, std::vector<double>& s) {
  const int hd = d_q / 2;
  const int64_t qoff = ((int64_t)b * H + h) * d_q + (int64_t)half * hd;
  s.assign(n, 0.0);
  for (int a = 0; a < n; ++a) {
    const int64_t coff = (((int64_t)h * 2 + half) * n + a) * hd;
    double acc = 0.0;
    for (int t = 0; t < hd; ++t) acc += widen(q, qdt, qoff + t) * widen(C, cdt, coff + t);
    s[a] = acc;
  }
}

// Subkey indices of the top m scores, ordered by (score desc, index asc).
std::vector<int> half_topk(const std::vector<double>& s, int m) {
  std::vector<int> order(s.size());
  for (size_t a = 0; a < s.size(); ++a) order[a] = (int)a;
  std::sort(order.begin(), order.end(), [&](int x, int y) {
    if (s[x] != s[y]) return s[x] > s[y];
    return x < y;
  });
  order.resize(m);
  return order;
}

// All m x m sums of the two per-half lists, sorted.
std::vector<Cand> pair_candidates(const std::vector<double>& s1, const std::vector<int>& a1,
                                  const std::vector<double>& s2, const std::vector<int>& a2,
                                  int n) {
  std::vector<Cand> c;
  c.reserve(a1.size() * a2.size());
  for (int i : a1)
    for (int j : a2) c.push_back({s1[i] + s2[j], (int64_t)i * n + j});
  std::sort(c.begin(), c.end(), cand_before);
  return c;
}

inline double rel_gap(double hi, double lo) {
  double den = std::max(std::fabs(hi), std::fabs(lo));
  if (den == 0.0) return 0.0;
  return (hi - lo) / den;
}

int check_shape(int B, int H, int d_q, int n, int k) {
  if (B < 0 || H < 1 || d_q < 2 || (d_q & 1) || n < 1 || k < 1 || k > n) return -1;
  if ((int64_t)n * n > (int64_t)1 << 40) return -1;
  return 0;
}

}  // namespace

extern "C" {

// Lookup steps: per-half scoring, per-half top-k, k^2 merge, top-k, softmax.
//   q        [B, H, d_q]              (fp32 or bf16 bits)
//   subkeys  [H, 2, n, d_q/2]
//   idx      [B, H, k] int64 flat indices, (score desc, flat asc)
//   score    [B, H, k] double, the winners' scores (may be NULL)
//   w        [B, H, k] double softmax weights (may be NULL)
//   gap_k    [B, H] relative gap between the k-th and (k+1)-th best full key
//            (+inf when there is no (k+1)-th key) (may be NULL)
//   gap_in   [B, H] smallest relative gap between adjacent winners (+inf when
//            k == 1) (may be NULL)
//   counters [2] += subkey scores computed, k^2 merge candidates (may be NULL)
// Returns 0, or -1 for an invalid shape.
int oracle_lookup(const void* q, int qdt, const void* subkeys, int cdt, int B, int H, int d_q,
                  int n, int k, int64_t* idx, double* score, double* w, double* gap_k,
                  double* gap_in, long long* counters, int nthreads) {
  if (check_shape(B, H, d_q, n, k)) return -1;
  const int64_t pairs = (int64_t)B * H;
  long long n_scores = 0, n_cands = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : n_scores, n_cands)
#endif
  for (int64_t p = 0; p < pairs; ++p) {
    const int64_t b = p / H;
    const int h = (int)(p % H);
    std::vector<double> s1, s2;
    subkey_scores(q, qdt, subkeys, cdt, H, d_q, n, b, h, 0, s1);
    subkey_scores(q, qdt, subkeys, cdt, H, d_q, n, b, h, 1, s2);
    n_scores += 2LL * n;

    // The lookup itself: k winners per half, k^2 candidates, top-k.
    std::vector<int> a1 = half_topk(s1, k), a2 = half_topk(s2, k);
    std::vector<Cand> c = pair_candidates(s1, a1, s2, a2, n);
    n_cands += (long long)c.size();

    const double smax = c[0].score;
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += std::exp(c[j].score - smax);
    for (int j = 0; j < k; ++j) {
      idx[p * k + j] = c[j].flat;
      if (score) score[p * k + j] = c[j].score;
      if (w) w[p * k + j] = std::exp(c[j].score - smax) / z;
    }

    // Near-tie report (not part of the lookup): the (k+1)-th best full key
    // lies in top_{k+1}(half 1) x top_{k+1}(half 2) by the same argument.
    if (gap_k) {
      const int64_t N = (int64_t)n * n;
      if (N <= k) {
        gap_k[p] = INFINITY;
      } else {
        int m = std::min(k + 1, n);
        std::vector<int> e1 = half_topk(s1, m), e2 = half_topk(s2, m);
        std::vector<Cand> ce = pair_candidates(s1, e1, s2, e2, n);
        gap_k[p] = rel_gap(c[k - 1].score, ce[k].score);
      }
    }
    if (gap_in) {
      double g = INFINITY;
      for (int j = 0; j + 1 < k; ++j) g = std::min(g, rel_gap(c[j].score, c[j + 1].score));
      gap_in[p] = g;
    }
  }
  if (counters) {
    counters[0] += n_scores;
    counters[1] += n_cands;
  }
  return 0;
}

// Value read: out[b, :] = sum_h sum_j w[b,h,j] * V[idx[b,h,j], :], in double.
//   values [N, d_v] (fp32 or bf16 bits); out [B, d_v] double (overwritten).
// Returns 0, or -1 for a bad shape or an index outside [0, N).
int oracle_gather(const void* values, int vdt, int64_t N, int d_v, int B, int H, int k,
                  const int64_t* idx, const double* w, double* out, int nthreads) {
  if (B < 0 || H < 1 || k < 1 || d_v < 1 || N < 1) return -1;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(| : bad)
#endif
  for (int64_t b = 0; b < B; ++b) {
    double* o = out + b * d_v;
    for (int t = 0; t < d_v; ++t) o[t] = 0.0;
    for (int h = 0; h < H; ++h)
      for (int j = 0; j < k; ++j) {
        const int64_t e = (b * H + h) * k + j;
        const int64_t r = idx[e];
        if (r < 0 || r >= N) {
          bad = 1;
          continue;
        }
        for (int t = 0; t < d_v; ++t) o[t] += w[e] * widen(values, vdt, r * d_v + t);
      }
  }
  return bad ? -1 : 0;
}

// The whole forward pass: lookup then read (idx, w and out as above).
int oracle_forward(const void* q, int qdt, const void* subkeys, int cdt, const void* values,
                   int vdt, int B, int H, int d_q, int n, int d_v, int k, int64_t* idx, double* w,
                   double* out, int nthreads) {
  int rc = oracle_lookup(q, qdt, subkeys, cdt, B, H, d_q, n, k, idx, nullptr, w, nullptr,
                         nullptr, nullptr, nthreads);
  if (rc) return rc;
  return oracle_gather(values, vdt, (int64_t)n * n, d_v, B, H, k, idx, w, out, nthreads);
}

// ---------------------------------------------------------- fp8 value table

// The value of an e4m3 code, from the format's definition.
double oracle_e4m3_value(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// The e4m3 code nearest to x (ties to the even mantissa), saturated to the
// largest finite magnitude; NaN -> 0x7F.  Binary search over the 127
// non-negative finite codes, whose values increase with the code.
uint8_t oracle_e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 0x7E;  // value(lo) <= a < value(hi) after the search
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (oracle_e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  if (oracle_e4m3_value((uint8_t)hi) <= a) lo = hi;  // only when a == 448 exactly (handled above)
  const double vlo = oracle_e4m3_value((uint8_t)lo);
  if (vlo == a || lo == 0x7E) return sign | (uint8_t)lo;
  const double vhi = oracle_e4m3_value((uint8_t)(lo + 1));
  const double dlo = a - vlo, dhi = vhi - a;
  int c = lo;
  if (dhi < dlo || (dhi == dlo && ((lo + 1) & 1) == 0)) c = lo + 1;
  return sign | (uint8_t)c;
}

// Per-row quantisation of values [N, d_v] (fp32 or bf16 bits) into e4m3
// codes [N, d_v] and fp32 scales [N] (recipe in the header comment).
int oracle_quantize_fp8(const void* values, int vdt, int64_t N, int d_v, uint8_t* codes,
                        float* scales, int nthreads) {
  if (N < 1 || d_v < 1) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int64_t r = 0; r < N; ++r) {
    float amax = 0.0f;
    for (int t = 0; t < d_v; ++t) {
      const float x = (float)widen(values, vdt, r * d_v + t);  // exact: every input is a float
      amax = std::max(amax, std::fabs(x));
    }
    float scale = amax / 448.0f;
    if (!(scale >= FLT_MIN)) scale = FLT_MIN;
    scales[r] = scale;
    for (int t = 0; t < d_v; ++t) {
      const float x = (float)widen(values, vdt, r * d_v + t);
      codes[r * d_v + t] = oracle_e4m3_encode(x / scale);
    }
  }
  return 0;
}

// Value read from the fp8 table: out[b, :] = sum_h sum_j w[b,h,j] * scale[r] *
// value(code[r, :]) with r = idx[b,h,j], in double (each product is exact).
int oracle_gather_fp8(const uint8_t* codes, const float* scales, int64_t N, int d_v, int B, int H,
                      int k, const int64_t* idx, const double* w, double* out, int nthreads) {
  if (B < 0 || H < 1 || k < 1 || d_v < 1 || N < 1) return -1;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(| : bad)
#endif
  for (int64_t b = 0; b < B; ++b) {
    double* o = out + b * d_v;
    for (int t = 0; t < d_v; ++t) o[t] = 0.0;
    for (int h = 0; h < H; ++h)
      for (int j = 0; j < k; ++j) {
        const int64_t e = (b * H + h) * k + j;
        const int64_t r = idx[e];
        if (r < 0 || r >= N) {
          bad = 1;
          continue;
        }
        const double ws = w[e] * (double)scales[r];
        for (int t = 0; t < d_v; ++t) o[t] += ws * oracle_e4m3_value(codes[r * d_v + t]);
      }
  }
  return bad ? -1 : 0;
}

// ---------------------------------------------------------------- backward

// Gradients of the forward pass for a fixed selection (the top-k choices are
// not differentiated; only the selected scores and rows carry gradient, as
// in the code listing's autograd through topk, the softmax and the
// EmbeddingBag read).  Given dout [B, d_v]:
//   dV[r, :]   += sum over (b,h,j) with idx = r of w[b,h,j] * dout[b, :]
//   dw[b,h,j]   = dout[b, :] . V[idx[b,h,j], :]
//   ds[b,h,j]   = w[b,h,j] * (dw[b,h,j] - sum_l w[b,h,l] * dw[b,h,l])      (softmax)
//   each winner's score is s1[a1] + s2[a2] with a1 = idx / n, a2 = idx % n:
//   dq[b,h,0:D/2]   += ds * C[h,0,a1,:]      dC[h,0,a1,:] += ds * q[b,h,0:D/2]
//   dq[b,h,D/2:D]   += ds * C[h,1,a2,:]      dC[h,1,a2,:] += ds * q[b,h,D/2:D]
// in double.  dq [B,H,d_q] and dw [B,H,k] are overwritten; dC [H,2,n,d_q/2]
// and dV are added to: dV is [n^2, d_v], or with dv_slot given, one row per
// table row r whose dv_slot[r] >= 0 (at that row; other rows' sums are not
// formed).  Sequential over queries (the scatters).
int oracle_backward(const void* q, int qdt, const void* subkeys, int cdt, const void* values,
                    int vdt, int B, int H, int d_q, int n, int d_v, int k, const int64_t* idx,
                    const double* w, const double* dout, double* dw, double* dq, double* dC,
                    double* dV, const int64_t* dv_slot) {
  if (B < 0 || H < 1 || d_q < 2 || (d_q & 1) || n < 1 || k < 1 || d_v < 1) return -1;
  const int hd = d_q / 2;
  const int64_t N = (int64_t)n * n;
  std::vector<double> ds(k);
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      const int64_t e0 = (b * H + h) * k;
      double sw = 0.0;
      for (int j = 0; j < k; ++j) {
        const int64_t r = idx[e0 + j];
        if (r < 0 || r >= N) return -1;
        double acc = 0.0;
        for (int t = 0; t < d_v; ++t) acc += dout[b * d_v + t] * widen(values, vdt, r * d_v + t);
        dw[e0 + j] = acc;
        sw += w[e0 + j] * acc;
        // dv_slot (optional): the dV row each table row accumulates into, -1 for none
        const int64_t slot = dv_slot ? dv_slot[r] : r;
        if (slot >= 0)
          for (int t = 0; t < d_v; ++t) dV[slot * d_v + t] += w[e0 + j] * dout[b * d_v + t];
      }
      for (int j = 0; j < k; ++j) ds[j] = w[e0 + j] * (dw[e0 + j] - sw);
      double* dqb = dq + (b * H + h) * d_q;
      for (int t = 0; t < d_q; ++t) dqb[t] = 0.0;
      for (int j = 0; j < k; ++j) {
        const int64_t a[2] = {idx[e0 + j] / n, idx[e0 + j] % n};
        for (int half = 0; half < 2; ++half) {
          const int64_t crow = (((int64_t)h * 2 + half) * n + a[half]) * hd;
          for (int t = 0; t < hd; ++t) {
            dqb[half * hd + t] += ds[j] * widen(subkeys, cdt, crow + t);
            dC[crow + t] += ds[j] * widen(q, qdt, (b * H + h) * d_q + half * hd + t);
          }
        }
      }
    }
  return 0;
}

// ----------------------------------------------------------- query network

// Product-Key Memory, code listing: q = qnorm(query(x)) with query an
// nn.Linear(dim, F, bias=False) (weight [F, dim]) and qnorm an
// nn.BatchNorm1d(F), here in its inference form with running statistics:
//   z[b, f] = sum_t x[b, t] * W[f, t]                      (one sequential loop)
//   q[b, f] = (z[b, f] - mean[f]) / sqrt(var[f] + eps) * gamma[f] + beta[f]
// in double; x and W fp32 or bf16 bits.
int oracle_query_net(const void* x, int xdt, const void* w, int wdt, int B, int dim, int F,
                     const float* gamma, const float* beta, const float* mean, const float* var,
                     double eps, double* q, int nthreads) {
  if (B < 0 || dim < 1 || F < 1) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int64_t b = 0; b < B; ++b)
    for (int f = 0; f < F; ++f) {
      double z = 0.0;
      for (int t = 0; t < dim; ++t)
        z += widen(x, xdt, b * dim + t) * widen(w, wdt, (int64_t)f * dim + t);
      q[b * F + f] = (z - (double)mean[f]) / std::sqrt((double)var[f] + eps) * (double)gamma[f] +
                     (double)beta[f];
    }
  return 0;
}

// The query network in training mode: q = BatchNorm1d(x W^T) normalised by
// the statistics of the batch itself (Product-Key Memory, "Keeping the
// memory in use": the BatchNorm over the queries, computed on the batch, is
// a global constraint that spreads them over the key space; code listing:
// Linear(dim, F, bias=False) then BatchNorm1d).  Per feature f: the batch
// mean mu_f = sum_b z[b,f] / B and the biased variance var_f = sum_b (z[b,f]
// - mu_f)^2 / B (two passes), then q = (z - mu_f) / sqrt(var_f + eps) *
// gamma_f + beta_f.  mean_out / var_out (may be NULL) receive mu and var.
int oracle_query_net_batch(const void* x, int xdt, const void* w, int wdt, int B, int dim, int F,
                           const float* gamma, const float* beta, double eps, double* q,
                           double* mean_out, double* var_out, int nthreads) {
  if (B < 1 || dim < 1 || F < 1) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int64_t b = 0; b < B; ++b)
    for (int f = 0; f < F; ++f) {
      double z = 0.0;
      for (int t = 0; t < dim; ++t)
        z += widen(x, xdt, b * dim + t) * widen(w, wdt, (int64_t)f * dim + t);
      q[b * F + f] = z;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int f = 0; f < F; ++f) {
    double mu = 0.0;
    for (int64_t b = 0; b < B; ++b) mu += q[b * F + f];
    mu /= (double)B;
    double var = 0.0;
    for (int64_t b = 0; b < B; ++b) var += (q[b * F + f] - mu) * (q[b * F + f] - mu);
    var /= (double)B;
    const double inv = 1.0 / std::sqrt(var + eps);
    for (int64_t b = 0; b < B; ++b)
      q[b * F + f] = (q[b * F + f] - mu) * inv * (double)gamma[f] + (double)beta[f];
    if (mean_out) mean_out[f] = mu;
    if (var_out) var_out[f] = var;
  }
  return 0;
}

// Brute force over every full key: score(a, b') is ONE d_q-long dot product
// of q[b,h] with concat(C[h,0,a], C[h,1,b']); all n^2 keys sorted by
// (score desc, flat asc); first k kept.  Independent of the factorisation.
int oracle_brute_topk(const void* q, int qdt, const void* subkeys, int cdt, int B, int H,
                      int d_q, int n, int k, int64_t* idx, double* score, int nthreads) {
  if (check_shape(B, H, d_q, n, k)) return -1;
  const int hd = d_q / 2;
  const int64_t N = (int64_t)n * n;
  const int64_t pairs = (int64_t)B * H;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t p = 0; p < pairs; ++p) {
    const int64_t b = p / H;
    const int h = (int)(p % H);
    const int64_t qoff = (b * H + h) * d_q;
    std::vector<double> key(d_q);
    std::vector<Cand> all;
    all.reserve(N);
    for (int a = 0; a < n; ++a)
      for (int bb = 0; bb < n; ++bb) {
        for (int t = 0; t < hd; ++t) {
          key[t] = widen(subkeys, cdt, (((int64_t)h * 2 + 0) * n + a) * hd + t);
          key[hd + t] = widen(subkeys, cdt, (((int64_t)h * 2 + 1) * n + bb) * hd + t);
        }
        double acc = 0.0;
        for (int t = 0; t < d_q; ++t) acc += widen(q, qdt, qoff + t) * key[t];
        all.push_back({acc, (int64_t)a * n + bb});
      }
    std::partial_sort(all.begin(), all.begin() + k, all.end(), cand_before);
    for (int j = 0; j < k; ++j) {
      idx[p * k + j] = all[j].flat;
      if (score) score[p * k + j] = all[j].score;
    }
  }
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
