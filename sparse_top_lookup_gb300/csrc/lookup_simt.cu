// Steps a1-a5 on the CUDA cores: the path for fp32 queries and subkeys.
//
// Product-Key Memory, "Factorising the key space": score each half of the
// query against its own subkey set, keep the top-k of each half, form the k^2
// separable sums s1 + s2 with flat index a1 * n_keys + a2, keep their top-k,
// and (code listing) softmax the winners.  This path serves fp32 problems
// and bf16 ones with 32 < k <= 64 (the tensor-core path keeps lists of at most
// 32 per half); bf16 inputs are widened exactly.  It is plain and exact: one CTA
// per (query, head), fp32 FMA dot products, and every selection done by
// ranking, so ties follow the same total orders as everywhere else: (score
// desc, subkey asc) within a half and (score desc, flat asc) overall.  The
// dot products are fp32 FMA; the order of the additions inside one dot
// product is the lane-strided partial sums described at the scoring step.
#include <float.h>
#include <stdint.h>

#include "pkm_internal.cuh"

namespace pkm {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float load_elem(const float* p, int64_t i) { return p[i]; }
// bf16 (raw bits) widened exactly to fp32
__device__ __forceinline__ float load_elem(const uint16_t* p, int64_t i) {
  return __uint_as_float((uint32_t)p[i] << 16);
}

// Products of one 16-byte vector of subkey elements with the matching query
// elements, accumulated in element order.
__device__ __forceinline__ float dot16(const uint4& u, const float* qv, const float*) {
  float acc = 0.0f;
  acc = fmaf(__uint_as_float(u.x), qv[0], acc);
  acc = fmaf(__uint_as_float(u.y), qv[1], acc);
  acc = fmaf(__uint_as_float(u.z), qv[2], acc);
  acc = fmaf(__uint_as_float(u.w), qv[3], acc);
  return acc;
}
__device__ __forceinline__ float dot16(const uint4& u, const float* qv, const uint16_t*) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(w[i] << 16), qv[2 * i], acc);
    acc = fmaf(__uint_as_float(w[i] & 0xffff0000u), qv[2 * i + 1], acc);
  }
  return acc;
}
// Steps a1-a5 for one (query, head) pair, by the whole CTA.
template <typename TIn>
__device__ void lookup_pair(const TIn* __restrict__ q, const TIn* __restrict__ subkeys, int H,
                            int d_q, int n, int k, int64_t pair, int64_t* __restrict__ idx,
                            float* __restrict__ w, unsigned char* smem) {
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
  const int tid = threadIdx.x;
  const int h = (int)(pair % H);

  __syncthreads();  // shared data of a previous pair is no longer read
  for (int t = tid; t < d_q; t += kThreads) s_q[t] = load_elem(q, pair * d_q + t);
  __syncthreads();

  // a2: subkey scores of both halves.  When a subkey row is a whole number
  // of 16-byte vectors, one warp reads a row (coalesced), each lane takes every
  // 32nd vector and the lanes' partial sums are added with shuffles.  A warp
  // takes 8 rows at a time so their loads are in flight together.
  constexpr int EPV = 16 / (int)sizeof(TIn);
  if (hd % EPV == 0) {
    constexpr int R = 8;
    const int warp = tid >> 5, lane = tid & 31;
    const int nvec = hd / EPV;
    const int nwarps = kThreads / 32;
    for (int e0 = warp * R; e0 < 2 * n; e0 += nwarps * R) {
      float acc[R];
#pragma unroll
      for (int u = 0; u < R; ++u) acc[u] = 0.0f;
      for (int vi = lane; vi < nvec; vi += 32) {
        uint4 x[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
          const int e = e0 + u < 2 * n ? e0 + u : 2 * n - 1;  // in bounds, unused past the end
          const int half = e / n, a = e - half * n;
          x[u] = reinterpret_cast<const uint4*>(subkeys +
                                                (((int64_t)h * 2 + half) * n + a) * hd)[vi];
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
          const int e = e0 + u < 2 * n ? e0 + u : 2 * n - 1;
          acc[u] += dot16(x[u], s_q + (e / n) * hd + vi * EPV, subkeys);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < R; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
      if (lane == 0)
#pragma unroll
        for (int u = 0; u < R; ++u)
          if (e0 + u < 2 * n) s_sc[e0 + u] = acc[u];
    }
  } else {
    for (int e = tid; e < 2 * n; e += kThreads) {
      const int half = e / n, a = e - half * n;
      const int64_t c = (((int64_t)h * 2 + half) * n + a) * hd;
      const float* qh = s_q + half * hd;
      float acc = 0.0f;
      for (int t = 0; t < hd; ++t) acc = fmaf(qh[t], load_elem(subkeys, c + t), acc);
      s_sc[e] = acc;
    }
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

// CTA b handles the (query, head) pair b.
template <typename TIn>
__global__ void __launch_bounds__(kThreads)
lookup_simt_kernel(const TIn* __restrict__ q, const TIn* __restrict__ subkeys, int H, int d_q,
                   int n, int k, int64_t* __restrict__ idx, float* __restrict__ w) {
  extern __shared__ __align__(16) unsigned char smem[];
  lookup_pair(q, subkeys, H, d_q, n, k, (int64_t)blockIdx.x, idx, w, smem);
}

size_t simt_smem(int d_q, int n_keys, int k) {
  return (size_t)d_q * 4 + (size_t)2 * n_keys * 4 + (size_t)4 * k * 4 + (size_t)2 * k * k * 4 +
         (size_t)2 * k * 4 + 16;
}

}  // namespace

template <typename TIn>
cudaError_t launch_simt(const TIn* q, const TIn* subkeys, int B, int H, int d_q, int n_keys,
                        int k, int64_t* idx, float* w, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t smem = simt_smem(d_q, n_keys, k);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(lookup_simt_kernel<TIn>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t pairs = (int64_t)B * H;
  lookup_simt_kernel<TIn><<<(unsigned)pairs, kThreads, smem, stream>>>(q, subkeys, H, d_q,
                                                                       n_keys, k, idx, w);
  return cudaGetLastError();
}

cudaError_t launch_lookup_simt(const float* q, const float* subkeys, int B, int H, int d_q,
                               int n_keys, int k, int64_t* idx, float* w, cudaStream_t stream) {
  return launch_simt(q, subkeys, B, H, d_q, n_keys, k, idx, w, stream);
}

cudaError_t launch_lookup_simt_bf16(const uint16_t* q, const uint16_t* subkeys, int B, int H,
                                    int d_q, int n_keys, int k, int64_t* idx, float* w,
                                    cudaStream_t stream) {
  return launch_simt(q, subkeys, B, H, d_q, n_keys, k, idx, w, stream);
}

}  // namespace pkm
