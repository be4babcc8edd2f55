// The fp8 e4m3 value table: per-row quantisation of an fp32 or bf16 table.
//
// Product-Key Memory, note after the code listing: the value table is "a
// good candidate for keeping in a lower precision".  Layout (include/pkm.h):
// N rows of d_v e4m3 codes, then N fp32 row scales.  Recipe per row (the page
// fixes none): scale = max(amax / 448, FLT_MIN) with amax the row's largest
// magnitude, code = the e4m3 value nearest to x / scale (IEEE fp32 division,
// round to nearest even, saturated to +-448: the hardware conversion
// cvt.rn.satfinite).  One warp per row; this runs once per table, outside the
// lookup path.
#include <cuda_fp8.h>
#include <float.h>
#include <stdint.h>

#include "pkm_internal.cuh"

namespace pkm {
namespace {

template <bool kBf16>
__device__ __forceinline__ void load4(const void* values, int64_t e, float (&x)[4]) {
  if (kBf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(values) + e);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(values) + e);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
  }
}

template <bool kBf16>
__global__ void quantize_fp8_kernel(const void* __restrict__ values, int64_t N, int d_v,
                                    uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < N;
       r += warps) {
    const int64_t e0 = r * d_v;
    float amax = 0.0f;
    for (int c = 4 * lane; c < d_v; c += 128) {
      float x[4];
      load4<kBf16>(values, e0 + c, x);
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float scale = __fdiv_rn(amax, 448.0f);
    if (!(scale >= FLT_MIN)) scale = FLT_MIN;
    if (lane == 0) scales[r] = scale;
    for (int c = 4 * lane; c < d_v; c += 128) {
      float x[4];
      load4<kBf16>(values, e0 + c, x);
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        word |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], scale), __NV_SATFINITE, __NV_E4M3)
                << (8 * i);
      *reinterpret_cast<uint32_t*>(codes + e0 + c) = word;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* values, int value_dtype, int64_t N, int d_v, void* out,
                                cudaStream_t stream) {
  uint8_t* codes = static_cast<uint8_t*>(out);
  float* scales = reinterpret_cast<float*>(codes + N * d_v);
  const int threads = 256;  // 8 rows per CTA
  int64_t blocks = (N + 7) / 8;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  if (value_dtype == PKM_BF16)
    quantize_fp8_kernel<true><<<(unsigned)blocks, threads, 0, stream>>>(values, N, d_v, codes,
                                                                         scales);
  else
    quantize_fp8_kernel<false><<<(unsigned)blocks, threads, 0, stream>>>(values, N, d_v, codes,
                                                                          scales);
  return cudaGetLastError();
}

}  // namespace pkm

extern "C" int pkm_quantize_values_fp8(const void* values, int value_dtype, int64_t N, int d_v,
                                       void* out, void* stream) {
  if (!values || !out || N < 1 || d_v < 1) return PKM_ERR_INVALID;
  if (value_dtype != PKM_F32 && value_dtype != PKM_BF16) return PKM_ERR_UNSUPPORTED;
  if (d_v % 16) return PKM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(values) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
    return PKM_ERR_ALIGN;
  return pkm::launch_quantize_fp8(values, value_dtype, N, d_v, out,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKM_OK
             : PKM_ERR_CUDA;
}
