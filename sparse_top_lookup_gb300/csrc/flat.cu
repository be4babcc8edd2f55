// The flat exact top-k: the search that product keys replace, on the same
// GPU, as the baseline that measures what the factorisation saves.
//
// Memory Retrieval Mechanisms, top-k retrieval and its cost walk-through:
// score the query against every one of the N keys (O(N d)), keep the k best
// and take the softmax over them.  Product-Key Memory, "Factorising the key
// space": a full key is the concatenation of one subkey of each half, key
// (a, b) = [c1_a ; c2_b] with flat index a * n_keys + b, so the full key
// table is materialised from the subkeys and each of its N = n_keys^2 rows
// is scored as one d_q-long dot product (2 sqrt(N) subkey comparisons
// against N full-key ones).
//
//   full_keys_kernel     keys[h][a * n + b] = concat(C[h][0][a], C[h][1][b]),
//                        16-byte copies (an HBM write stream);
//   select_2sm_kernel    (flat form, lookup_2sm.cu) tcgen05 scoring of 256
//                        query rows per CTA pair against 256 full keys per
//                        chunk, the exact top-k of each row streamed through
//                        the register selection, softmax in its epilogue.
#include <cuda.h>
#include <stdint.h>

#include <algorithm>

#include "pkm_internal.cuh"
#include "tc_common.cuh"

namespace pkm {
namespace {

// One thread per 16 bytes of the full key table.
__global__ void full_keys_kernel(const uint4* __restrict__ subkeys, int n, int hd16,
                                 int64_t total, uint4* __restrict__ keys) {
  const int64_t row16 = 2 * (int64_t)hd16;  // 16-byte pieces of a full key
  const int64_t N = (int64_t)n * n;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / row16;  // h * N + flat
    const int p = (int)(t - r * row16);
    const int64_t h = r / N, f = r - h * N;
    const int half = p >= hd16;
    const int64_t sub = half ? f % n : f / n;
    keys[t] = subkeys[((h * 2 + half) * n + sub) * hd16 + (p - half * hd16)];
  }
}

}  // namespace

cudaError_t launch_full_keys(const uint16_t* subkeys, int H, int n_keys, int d_q, uint16_t* keys,
                             cudaStream_t stream) {
  if (d_q % 16) return cudaErrorInvalidValue;  // 16-byte pieces within each half
  const int hd16 = d_q / 2 / 8;
  const int64_t total = (int64_t)H * n_keys * n_keys * 2 * hd16;
  if (total == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)tc::sm_count() * 16);
  full_keys_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(subkeys), n_keys, hd16, total, reinterpret_cast<uint4*>(keys));
  return cudaGetLastError();
}

cudaError_t launch_flat_lookup(const uint16_t* q, const uint16_t* keys, int B, int H, int d_q,
                               int N, int k, int64_t* idx, float* w, int* status,
                               cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  if (k > kTcMaxK || k > N || d_q % 16) return cudaErrorInvalidValue;
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap mq, mk;
  {
    // q viewed as [B][H][1][d_q] (the selection kernel's half axis has one
    // entry), 64 x 128 boxes
    const cuuint64_t dims[4] = {(cuuint64_t)d_q, 1, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d_q * 2, (cuuint64_t)d_q * 2,
                                   (cuuint64_t)H * d_q * 2};
    const cuuint32_t box[4] = {64, 1, 1, 128};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // full keys [H][N][d_q], 64 x 128 boxes (each CTA of a pair loads 128 of
    // a chunk's 256 keys)
    const cuuint64_t dims[3] = {(cuuint64_t)d_q, (cuuint64_t)N, (cuuint64_t)H};
    const cuuint64_t strides[2] = {(cuuint64_t)d_q * 2, (cuuint64_t)N * d_q * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(keys), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return launch_select_2sm_flat(mq, mk, B, H, d_q, N, k, idx, w, status, stream);
}

}  // namespace pkm
