// Steps a1-a5 for fp32 queries and subkeys, on the CUDA cores.
//
// Product-Key Memory, "Factorising the key space": score each half of the
// query against its own subkey set, keep the top-k of each half, form the k^2
// separable sums s1 + s2 with flat index a1 * n_keys + a2, keep their top-k,
// and (code listing) softmax the winners.  This path serves small fp32
// problems (the tensor-core path takes bf16); it is plain and exact: one CTA
// per (query, head), fp32 FMA dot products, and every selection done by
// ranking, so ties follow the same total orders as everywhere else: (score
// desc, subkey asc) within a half and (score desc, flat asc) overall.
#include <float.h>
#include <stdint.h>

#include "pkm_internal.cuh"

namespace pkm {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
lookup_simt_kernel(const float* __restrict__ q, const float* __restrict__ subkeys, int H, int d_q,
                   int n, int k, int64_t* __restrict__ idx, float* __restrict__ w) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int hd = d_q / 2;
  float* s_q = reinterpret_cast<float*>(smem);         // [d_q]
  float* s_sc = s_q + d_q;                             // [2][n]
  float* s_tv = s_sc + 2 * n;                          // [2][k] per-half winners' scores
  int* s_ta = reinterpret_cast<int*>(s_tv + 2 * k);    // [2][k] per-half winners' subkeys
  float* s_cv = reinterpret_cast<float*>(s_ta + 2 * k);  // [k*k] candidate scores
  int* s_cf = reinterpret_cast<int*>(s_cv + k * k);      // [k*k] candidate flat indices
  float* s_ov = reinterpret_cast<float*>(s_cf + k * k);  // [k] output scores
  int* s_of = reinterpret_cast<int*>(s_ov + k);          // [k] output flats
  float* s_z = reinterpret_cast<float*>(s_of + k);       // softmax denominator

  const int64_t pair = blockIdx.x;  // b * H + h
  const int h = (int)(pair % H);
  const int tid = threadIdx.x;

  for (int t = tid; t < d_q; t += kThreads) s_q[t] = q[pair * d_q + t];
  __syncthreads();

  // a2: subkey scores of both halves.
  for (int e = tid; e < 2 * n; e += kThreads) {
    const int half = e / n, a = e - half * n;
    const float* c = subkeys + (((int64_t)h * 2 + half) * n + a) * hd;
    const float* qh = s_q + half * hd;
    float acc = 0.0f;
    for (int t = 0; t < hd; ++t) acc = fmaf(qh[t], c[t], acc);
    s_sc[e] = acc;
  }
  __syncthreads();

  // a3: per-half top-k by rank: rank(a) = #{a' : s[a'] > s[a] or (s[a'] == s[a] and a' < a)}.
  for (int e = tid; e < 2 * n; e += kThreads) {
    const int half = e / n, a = e - half * n;
    const float* s = s_sc + half * n;
    const float v = s[a];
    int rank = 0;
    for (int a2 = 0; a2 < n && rank < k; ++a2) rank += (s[a2] > v) || (s[a2] == v && a2 < a);
    if (rank < k) {
      s_tv[half * k + rank] = v;
      s_ta[half * k + rank] = a;
    }
  }
  __syncthreads();

  // a4: k^2 separable candidates and their top-k, (score desc, flat asc).
  const int kk = k * k;
  for (int c = tid; c < kk; c += kThreads) {
    const int i = c / k, j = c - i * k;
    s_cv[c] = s_tv[i] + s_tv[k + j];
    s_cf[c] = s_ta[i] * n + s_ta[k + j];
  }
  __syncthreads();
  for (int c = tid; c < kk; c += kThreads) {
    const float v = s_cv[c];
    const int f = s_cf[c];
    int rank = 0;
    for (int c2 = 0; c2 < kk && rank < k; ++c2)
      rank += (s_cv[c2] > v) || (s_cv[c2] == v && s_cf[c2] < f);
    if (rank < k) {
      s_ov[rank] = v;
      s_of[rank] = f;
    }
  }
  __syncthreads();

  // a5: softmax over the winners, largest first.
  if (tid == 0) {
    float z = 0.0f;
    for (int j = 0; j < k; ++j) z += expf(s_ov[j] - s_ov[0]);
    s_z[0] = z;
  }
  __syncthreads();
  for (int j = tid; j < k; j += kThreads) {
    idx[pair * k + j] = (int64_t)s_of[j];
    w[pair * k + j] = expf(s_ov[j] - s_ov[0]) / s_z[0];
  }
}

}  // namespace

cudaError_t launch_lookup_simt(const float* q, const float* subkeys, int B, int H, int d_q,
                               int n_keys, int k, int64_t* idx, float* w, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t smem = (size_t)d_q * 4 + (size_t)2 * n_keys * 4 + (size_t)4 * k * 4 +
                      (size_t)2 * k * k * 4 + (size_t)2 * k * 4 + 16;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(lookup_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t pairs = (int64_t)B * H;
  lookup_simt_kernel<<<(unsigned)pairs, kThreads, smem, stream>>>(q, subkeys, H, d_q, n_keys, k,
                                                                  idx, w);
  return cudaGetLastError();
}

}  // namespace pkm
