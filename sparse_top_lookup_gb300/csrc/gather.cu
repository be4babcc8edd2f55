// Step a6: the weighted value read.
//
// Product-Key Memory (note after the code listing): the value table is read
// by an EmbeddingBag(mode="sum") with per-sample weights, so the k selected
// rows are gathered and weight-summed in one pass and the N x d table is
// never touched as a dense matrix.  Memory Retrieval Mechanisms (top-k
// retrieval): r = sum_j alpha_j v_{i_j}.  Here one bag holds the H*k rows a
// query selected over all its heads, so the per-head reads are summed.
//
// The kernel is HBM-bound: every byte of a selected row is read once, the
// arithmetic is one FMA per element.  One CTA owns one query (bag).  Each
// value row is split into 16-byte vectors and one thread owns one vector
// column, so a warp reads 512 contiguous bytes of a row; when a row has fewer
// vectors than the CTA has threads, the threads form row groups that take
// every G-th row and are reduced through shared memory at the end.  Loads are
// 16-byte non-coherent loads that bypass L1 (each row is used once per bag),
// unrolled eight rows deep so a thread keeps 128 bytes in flight.
//
// fp8 table (the note after the code listing: the value table is "a good
// candidate for keeping in a lower precision"): rows of e4m3 codes, one fp32
// scale per row stored after the codes.  A 16-byte vector then holds 16
// elements; the row's scale is folded into its staged weight, the codes are
// widened exactly (e4m3 -> f16 -> f32) and accumulated in fp32.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pkm_internal.cuh"

namespace pkm {
namespace {

constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Accumulate one 16-byte vector: 4 fp32, 8 bf16 or 16 fp8 e4m3 elements.
template <int VT>
struct VecAcc;

template <>
struct VecAcc<PKM_FP8_E4M3> {
  static constexpr int kElems = 16;
  __device__ __forceinline__ static void fma(float (&acc)[16], float wt, const uint4& v) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        // two codes -> two exact halves -> two floats (byte order = element order)
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            (__nv_fp8x2_storage_t)((u[i] >> (16 * hlf)) & 0xffffu), __NV_E4M3);
        const float2 f = __half22float2(__half2(hr));
        acc[4 * i + 2 * hlf] = fmaf(wt, f.x, acc[4 * i + 2 * hlf]);
        acc[4 * i + 2 * hlf + 1] = fmaf(wt, f.y, acc[4 * i + 2 * hlf + 1]);
      }
    }
  }
};

template <>
struct VecAcc<PKM_BF16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void fma(float (&acc)[8], float wt, const uint4& v) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wt, __uint_as_float(u[i] << 16), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wt, __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
    }
  }
};

template <>
struct VecAcc<PKM_F32> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void fma(float (&acc)[4], float wt, const uint4& v) {
    acc[0] = fmaf(wt, __uint_as_float(v.x), acc[0]);
    acc[1] = fmaf(wt, __uint_as_float(v.y), acc[1]);
    acc[2] = fmaf(wt, __uint_as_float(v.z), acc[2]);
    acc[3] = fmaf(wt, __uint_as_float(v.w), acc[3]);
  }
};

// grid: one CTA per bag.  block: vpr * groups threads.
// dynamic smem: rows_per_bag * (4 + 4) bytes, plus blockDim * E * 4 when groups > 1
// (kept small so these CTAs fit next to a running lookup kernel's CTA).
// scales: the fp8 table's row scales (null for fp32 / bf16 tables).
template <int VT>
__global__ void gather_kernel(const uint4* __restrict__ values, const float* __restrict__ scales,
                              int64_t N, int vpr, int groups, int rows_per_bag,
                              const int64_t* __restrict__ idx, const float* __restrict__ w,
                              float* __restrict__ out, int* __restrict__ status) {
  constexpr int E = VecAcc<VT>::kElems;
  extern __shared__ __align__(16) unsigned char smem[];
  int* s_row = reinterpret_cast<int*>(smem);
  float* s_w = reinterpret_cast<float*>(s_row + rows_per_bag);

  const int64_t bag = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t base = bag * rows_per_bag;

  // Stage the bag's row indices and weights.  An index outside [0, N) is
  // recorded and replaced by row 0 with weight 0, so every load stays inside
  // the table.
  for (int r = tid; r < rows_per_bag; r += blockDim.x) {
    int64_t row = idx[base + r];
    float wt = w[base + r];
    if (row < 0 || row >= N) {
      atomicExch(status, PKM_ERR_BAD_INDEX);
      row = 0;
      wt = 0.0f;
    }
    if (VT == PKM_FP8_E4M3) wt *= scales[row];
    s_row[r] = (int)row;
    s_w[r] = wt;
  }
  __syncthreads();

  const int g = tid / vpr;
  const int v = tid - g * vpr;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;

  const uint4* vbase = values + v;
  const int64_t stride = vpr;  // 16-byte vectors per value row
  int r = g;
  const int step = groups * kUnroll;
  for (; r + (kUnroll - 1) * groups < rows_per_bag; r += step) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) x[u] = ldg_stream(vbase + s_row[r + u * groups] * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) VecAcc<VT>::fma(acc, s_w[r + u * groups], x[u]);
  }
  for (; r < rows_per_bag; r += groups) {
    uint4 x = ldg_stream(vbase + s_row[r] * stride);
    VecAcc<VT>::fma(acc, s_w[r], x);
  }

  float* orow = out + bag * (int64_t)vpr * E;
  if (groups == 1) {
    float4* o4 = reinterpret_cast<float4*>(orow + v * E);
#pragma unroll
    for (int e = 0; e < E; e += 4) o4[e / 4] = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    return;
  }
  // Reduce the row groups: red[g][v][e].
  float* red = reinterpret_cast<float*>(smem + ((size_t)rows_per_bag * 8 + 15) / 16 * 16);
#pragma unroll
  for (int e = 0; e < E; ++e) red[(g * vpr + v) * E + e] = acc[e];
  __syncthreads();
  if (g == 0) {
    for (int gg = 1; gg < groups; ++gg)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += red[(gg * vpr + v) * E + e];
    float4* o4 = reinterpret_cast<float4*>(orow + v * E);
#pragma unroll
    for (int e = 0; e < E; e += 4) o4[e / 4] = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
  }
}

template <int VT>
cudaError_t launch_gather_vt(const void* values, int64_t N, int d_v, int B, int rows_per_bag,
                             const int64_t* idx, const float* w, float* out, int* status,
                             cudaStream_t stream) {
  constexpr int E = VecAcc<VT>::kElems;
  const int vpr = d_v / E;  // 16-byte vectors per row
  int groups = vpr >= 128 ? 1 : 128 / vpr;
  if (groups > rows_per_bag) groups = rows_per_bag > 0 ? rows_per_bag : 1;
  const int threads = vpr * groups;
  const size_t staged = (size_t)rows_per_bag * 8;
  const size_t red_off = (staged + 15) / 16 * 16;
  const size_t smem = groups > 1 ? red_off + (size_t)threads * E * 4 : staged;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gather_kernel<VT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // The loads bypass L1, so the SM can keep its maximum shared-memory split;
  // CTAs of this kernel then fit next to a running lookup kernel's CTA.
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaError_t e = cudaFuncSetAttribute(gather_kernel<VT>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    carveout_set = true;
  }
  // an fp8 table's row scales follow its N * d_v code bytes
  const float* scales =
      VT == PKM_FP8_E4M3
          ? reinterpret_cast<const float*>(static_cast<const unsigned char*>(values) + N * d_v)
          : nullptr;
  gather_kernel<VT><<<B, threads, smem, stream>>>(static_cast<const uint4*>(values), scales, N,
                                                  vpr, groups, rows_per_bag, idx, w, out, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const void* values, int value_dtype, int64_t N, int d_v, int B,
                          int rows_per_bag, const int64_t* idx, const float* w, float* out,
                          int* status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  if (value_dtype == PKM_FP8_E4M3)
    return launch_gather_vt<PKM_FP8_E4M3>(values, N, d_v, B, rows_per_bag, idx, w, out, status,
                                          stream);
  if (value_dtype == PKM_BF16)
    return launch_gather_vt<PKM_BF16>(values, N, d_v, B, rows_per_bag, idx, w, out, status,
                                      stream);
  return launch_gather_vt<PKM_F32>(values, N, d_v, B, rows_per_bag, idx, w, out, status, stream);
}

}  // namespace pkm
