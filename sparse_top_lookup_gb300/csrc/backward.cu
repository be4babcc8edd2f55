// Backward pass of the lookup and read for a fixed selection.
//
// Product-Key Memory, code listing: autograd through the forward flows only
// through the selected scores (topk keeps values and indices), the softmax
// and the EmbeddingBag read; "Keeping the memory in use": only the selected
// value rows and subkeys receive gradient.  Given dout [B, d_v]:
//   dV[idx]   += w * dout[b]                     (scatter-add, duplicates summed)
//   dw         = dout[b] . V[idx]
//   ds         = w * (dw - sum_l w_l dw_l)       (softmax)
//   score = s1[a1] + s2[a2], a1 = idx / n, a2 = idx % n, s_i = q_i . C[h,i,a]:
//   dq_i[b,h]  = sum_a DS_i[b,h][a] * C[h,i,a,:]
//   dC[h,i,a] += sum_b DS_i[b,h][a] * q_i[b,h]
// where DS_i[b,h] is the [n_keys] row of ds summed per subkey of half i.
//
// Read part (dw and dV), grouped by value row so that each selected row of V
// and of dV crosses HBM once however many selections hit it (the gradient
// rows dout, B * d_v * 4 bytes, are re-read from L2 instead):
//   bucket_count_kernel    selections per bucket of 256 consecutive rows;
//   bucket_scan_kernel     bucket offsets, and the work items: each bucket's
//                          list cut into chunks of at most kChunk selections;
//   bucket_scatter_kernel  selection numbers into their bucket's list;
//   bucket_sort_kernel     one CTA per item: a counting sort of the chunk by
//                          row in shared memory, written back in place, and
//                          the chunk's pieces (up to kPiece selections of one
//                          row) appended to a global piece list;
//   row_grad_kernel        persistent, a warp per piece: the value row is read
//                          once for every dw of the piece and the dV row
//                          updated once: plain read-modify-write when the row
//                          has one piece in one item, vector atomic adds
//                          otherwise.
// Score part:
//   ds_rows_kernel         one warp per (query, head, half): softmax backward
//                          and the dense bf16 DS row (duplicates summed in
//                          shared memory);
//   two strided-batched cuBLAS GEMMs over the 2H (head, half) blocks (plain
//   library GEMMs, bf16 in, fp32 out): dq = DS C (overwrites) and dC += DS^T q.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "pkm_internal.cuh"
#include "tc_common.cuh"

namespace pkm {
namespace {

constexpr int kRowsPerBucket = 256;  // a row's place in its bucket fits a byte
constexpr int kChunk = 2048;         // selections one CTA sorts in shared memory
constexpr int kPiece = 8;            // selections of one row in one warp pass
constexpr int kReadWarps = 8;

__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Elements 4u .. 4u+3 of value row `row`, widened to fp32.
template <bool kBf16>
__device__ __forceinline__ void load4(const void* values, int64_t row, int d_v, int u,
                                      float (&x)[4]) {
  if (kBf16) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(
                              static_cast<const uint16_t*>(values) + row * d_v) + u);
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
  } else {
    const float4 v =
        __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(values) + row * d_v) + u);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
}

__global__ void bucket_count_kernel(const int64_t* __restrict__ idx, int E, int64_t N,
                                    int* __restrict__ bcount, float* __restrict__ dw,
                                    int* __restrict__ status) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    const int64_t r = idx[e];
    if (r < 0 || r >= N) {  // recorded; the selection contributes nothing
      atomicExch(status, PKM_ERR_BAD_INDEX);
      dw[e] = 0.0f;
      continue;
    }
    atomicAdd(&bcount[r / kRowsPerBucket], 1);
  }
}

// One CTA of 1024 threads: exclusive scans of the bucket sizes (list
// offsets, the scatter's cursors) and of their chunk counts (item numbers);
// item = (list start, length, bucket, bucket has a single item).
__global__ void __launch_bounds__(1024)
bucket_scan_kernel(const int* __restrict__ bcount, int nb, int* __restrict__ cursor,
                   int4* __restrict__ items, int* __restrict__ n_items) {
  __shared__ int s_w0[32], s_w1[32];
  __shared__ int s_carry0, s_carry1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry0 = s_carry1 = 0;
  __syncthreads();
  for (int base = 0; base < nb; base += 1024) {
    const int i = base + threadIdx.x;
    const int c = i < nb ? bcount[i] : 0;
    const int nc = (c + kChunk - 1) / kChunk;
    int x0 = c, x1 = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
      if (lane >= o) {
        x0 += y0;
        x1 += y1;
      }
    }
    if (lane == 31) {
      s_w0[warp] = x0;
      s_w1[warp] = x1;
    }
    __syncthreads();
    if (warp == 0) {
      int a0 = s_w0[lane], a1 = s_w1[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, a0, o),
                  y1 = __shfl_up_sync(0xffffffffu, a1, o);
        if (lane >= o) {
          a0 += y0;
          a1 += y1;
        }
      }
      s_w0[lane] = a0;
      s_w1[lane] = a1;
    }
    __syncthreads();
    const int off0 = s_carry0 + (warp ? s_w0[warp - 1] : 0) + x0 - c;
    const int off1 = s_carry1 + (warp ? s_w1[warp - 1] : 0) + x1 - nc;
    if (i < nb) {
      cursor[i] = off0;
      for (int j = 0; j < nc; ++j)
        items[off1 + j] = make_int4(off0 + j * kChunk, min(kChunk, c - j * kChunk), i, nc == 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_carry0 += s_w0[31];
      s_carry1 += s_w1[31];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_items = s_carry1;
}

__global__ void bucket_scatter_kernel(const int64_t* __restrict__ idx, int E, int64_t N,
                                      int* __restrict__ cursor, int* __restrict__ list) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    const int64_t r = idx[e];
    if (r < 0 || r >= N) continue;
    list[atomicAdd(&cursor[r / kRowsPerBucket], 1)] = e;
  }
}

// One CTA per item: the item's selections sorted by row (counting sort in
// shared memory) and written back in place; each row's run cut into pieces of
// at most kPiece, appended to the piece list as (row, first, m, atomic).
__global__ void __launch_bounds__(kReadWarps * 32)
bucket_sort_kernel(const int64_t* __restrict__ idx, const int4* __restrict__ items,
                   const int* __restrict__ n_items, int* __restrict__ list,
                   int4* __restrict__ pieces, int* __restrict__ n_pieces) {
  constexpr int R = kRowsPerBucket;
  __shared__ int s_e[kChunk];
  __shared__ unsigned char s_r[kChunk];
  __shared__ int s_cnt[R];
  __shared__ int s_start[R + 1];
  __shared__ int s_pstart[R + 1];
  __shared__ int s_base;
  if ((int)blockIdx.x >= *n_items) return;
  const int4 it = items[blockIdx.x];
  const int len = it.y;
  const int64_t row0 = (int64_t)it.z * R;
  const bool excl = it.w != 0;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < R; i += nt) s_cnt[i] = 0;
  __syncthreads();
  for (int i = tid; i < len; i += nt) {
    const int e = list[it.x + i];
    const int r = (int)(idx[e] - row0);
    s_e[i] = e;
    s_r[i] = (unsigned char)r;
    atomicAdd(&s_cnt[r], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scans of the row counts and of their piece counts
    int v[R / 32], p[R / 32], t0 = 0, t1 = 0;
#pragma unroll
    for (int j = 0; j < R / 32; ++j) {
      v[j] = s_cnt[lane * (R / 32) + j];
      p[j] = (v[j] + kPiece - 1) / kPiece;
      t0 += v[j];
      t1 += p[j];
    }
    int x0 = t0, x1 = t1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
      if (lane >= o) {
        x0 += y0;
        x1 += y1;
      }
    }
    int a0 = x0 - t0, a1 = x1 - t1;
#pragma unroll
    for (int j = 0; j < R / 32; ++j) {
      s_start[lane * (R / 32) + j] = a0;
      s_cnt[lane * (R / 32) + j] = a0;
      s_pstart[lane * (R / 32) + j] = a1;
      a0 += v[j];
      a1 += p[j];
    }
    if (lane == 31) {
      s_start[R] = a0;
      s_pstart[R] = a1;
      s_base = atomicAdd(n_pieces, a1);
    }
  }
  __syncthreads();
  for (int i = tid; i < len; i += nt) list[it.x + atomicAdd(&s_cnt[s_r[i]], 1)] = s_e[i];
  for (int r = tid; r < R; r += nt) {
    const int c = s_start[r + 1] - s_start[r];
    const int np = s_pstart[r + 1] - s_pstart[r];
    for (int q = 0; q < np; ++q)
      pieces[s_base + s_pstart[r] + q] =
          make_int4((int)(row0 + r), it.x + s_start[r] + q * kPiece, min(kPiece, c - q * kPiece),
                    !excl || np > 1);
  }
}

// Persistent; a warp per piece (row, first, m, atomic): the m <= kPiece
// selections list[first .. first+m) of one value row.  One pass over the
// row's 4-element units reads the value row once for all m dot products dw
// and adds sum_g w_g * dout[b_g] into the dV row, by plain read-modify-write
// (the warp owns the row) or by vector atomic adds.
template <bool kBf16>
__global__ void __launch_bounds__(kReadWarps * 32, 4)
row_grad_kernel(const void* __restrict__ values, int d_v, int HK, const float* __restrict__ w,
                const float* __restrict__ dout, const int* __restrict__ list,
                const int4* __restrict__ pieces, const int* __restrict__ n_pieces,
                float* __restrict__ dw, float* __restrict__ dvalues) {
  const int lane = threadIdx.x & 31;
  const int total = *n_pieces;
  const int nu = d_v >> 2;
  for (int p = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); p < total;
       p += (int)((gridDim.x * blockDim.x) >> 5)) {
    const int4 pc = pieces[p];
    const int64_t row = pc.x;
    const int m = pc.z;
    const bool atomic = pc.w != 0;
    const int my_e = lane < m ? list[pc.y + lane] : 0;
    float wt[kPiece], part[kPiece];
    int doff[kPiece];  // dout row of each selection, in 16-byte units
#pragma unroll
    for (int g = 0; g < kPiece; ++g) {
      const int e = __shfl_sync(0xffffffffu, my_e, g);
      wt[g] = g < m ? __ldg(w + e) : 0.0f;
      doff[g] = (e / HK) * nu;
      part[g] = 0.0f;
    }
    const float4* d4 = reinterpret_cast<const float4*>(dout);
    float4* dv = reinterpret_cast<float4*>(dvalues + row * d_v);
    for (int u = lane; u < nu; u += 32) {
      float x[4];
      load4<kBf16>(values, row, d_v, u, x);
      float4 acc = atomic ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : dv[u];
#pragma unroll
      for (int g = 0; g < kPiece; ++g) {
        if (g < m) {
          const float4 d = __ldg(d4 + doff[g] + u);
          part[g] = fmaf(d.x, x[0], part[g]);
          part[g] = fmaf(d.y, x[1], part[g]);
          part[g] = fmaf(d.z, x[2], part[g]);
          part[g] = fmaf(d.w, x[3], part[g]);
          acc.x = fmaf(wt[g], d.x, acc.x);
          acc.y = fmaf(wt[g], d.y, acc.y);
          acc.z = fmaf(wt[g], d.z, acc.z);
          acc.w = fmaf(wt[g], d.w, acc.w);
        }
      }
      if (atomic)
        red_add4(&dv[u].x, acc.x, acc.y, acc.z, acc.w);
      else
        dv[u] = acc;
    }
#pragma unroll
    for (int g = 0; g < kPiece; ++g) {
      if (g < m) {
        float v = part[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == g) dw[my_e] = v;
      }
    }
  }
}

// One warp per (query, head, half): ds_j = w_j (dw_j - sum_l w_l dw_l), then
// DS[(2h + half)][b][a] = sum of ds_j over the winners whose half-`half`
// subkey is a, as a dense bf16 row of n entries.  k <= 32 (one lane per
// winner); dynamic smem: n floats per warp.  A winner whose index is outside
// [0, n^2) adds nothing (gather_bwd_kernel records it).
__global__ void ds_rows_kernel(const int64_t* __restrict__ idx, const float* __restrict__ w,
                               const float* __restrict__ dw, int B, int H, int n, int k,
                               __nv_bfloat16* __restrict__ ds_rows) {
  extern __shared__ __align__(16) float s_row[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;  // (pair, half)
  if (item >= (int64_t)B * H * 2) return;  // whole warp
  const int64_t pair = item >> 1;
  const int half = (int)(item & 1);
  const int64_t b = pair / H;
  const int h = (int)(pair - b * H);
  float* row = s_row + wib * n;
  for (int a = lane; a < n; a += 32) row[a] = 0.0f;
  const float wj = lane < k ? w[pair * k + lane] : 0.0f;
  const float dwj = lane < k ? dw[pair * k + lane] : 0.0f;
  float sw = wj * dwj;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, o);
  __syncwarp();
  if (lane < k) {
    const int64_t f = idx[pair * k + lane];
    if (f >= 0 && f < (int64_t)n * n) {
      const int a = (int)(half == 0 ? f / n : f % n);
      atomicAdd(&row[a], wj * (dwj - sw));
    }
  }
  __syncwarp();
  __nv_bfloat16* out = ds_rows + ((int64_t)(2 * h + half) * B + b) * n;
  if ((n & 1) == 0) {  // rows start 4-byte aligned: pairs of entries
    for (int a = 2 * lane; a < n; a += 64)
      *reinterpret_cast<__nv_bfloat162*>(out + a) = __floats2bfloat162_rn(row[a], row[a + 1]);
  } else {
    for (int a = lane; a < n; a += 32) out[a] = __float2bfloat16_rn(row[a]);
  }
}

}  // namespace

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The read part's scratch, each array 256-byte aligned: the item and piece
// counts and the bucket sizes [nb] (cleared per call, one memset), scatter
// cursors [nb], the items [max_items], the bucketed selection numbers [E] and
// the pieces [E].
static void read_layout(int64_t N, int64_t E, size_t* off, int64_t* nb_out, int64_t* items_out) {
  const int64_t nb = (N + kRowsPerBucket - 1) / kRowsPerBucket;
  const int64_t items = std::min(nb, E) + E / kChunk + 1;
  off[0] = 0;                                   // n_items, n_pieces
  off[1] = off[0] + 256;                        // bcount
  off[2] = off[1] + align256(nb * 4);           // cursor
  off[3] = off[2] + align256(nb * 4);           // items
  off[4] = off[3] + align256(items * 16);       // list
  off[5] = off[4] + align256(E * 4);            // pieces
  off[6] = off[5] + align256(E * 16);           // end
  *nb_out = nb;
  *items_out = items;
}

size_t backward_read_workspace_bytes(int B, int H, int n_keys, int k) {
  size_t off[7];
  int64_t nb, items;
  read_layout((int64_t)n_keys * n_keys, (int64_t)B * H * k, off, &nb, &items);
  return off[6];
}

size_t backward_scores_workspace_bytes(int B, int H, int n_keys) {
  return (size_t)2 * H * B * n_keys * 2;
}

size_t backward_dw_bytes(int B, int H, int k) { return align256((size_t)B * H * k * 4); }

size_t backward_workspace_bytes(int B, int H, int n_keys, int k) {
  return backward_dw_bytes(B, H, k) + std::max(backward_read_workspace_bytes(B, H, n_keys, k),
                                               backward_scores_workspace_bytes(B, H, n_keys));
}

cudaError_t launch_backward_read(const void* values, int value_dtype, int B, int H, int n_keys,
                                 int d_v, int k, const int64_t* idx, const float* w,
                                 const float* dout, float* dw, float* dvalues, void* workspace,
                                 int* status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int64_t N = (int64_t)n_keys * n_keys, E = (int64_t)B * H * k;
  if (E > INT32_MAX || (int64_t)B * d_v / 4 > INT32_MAX) return cudaErrorInvalidValue;
  size_t off[7];
  int64_t nb, max_items;
  read_layout(N, E, off, &nb, &max_items);
  if (nb > INT32_MAX || max_items > INT32_MAX) return cudaErrorInvalidValue;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* n_items = reinterpret_cast<int*>(ws + off[0]);
  int* n_pieces = n_items + 1;
  int* bcount = reinterpret_cast<int*>(ws + off[1]);
  int* cursor = reinterpret_cast<int*>(ws + off[2]);
  int4* items = reinterpret_cast<int4*>(ws + off[3]);
  int* list = reinterpret_cast<int*>(ws + off[4]);
  int4* pieces = reinterpret_cast<int4*>(ws + off[5]);
  cudaError_t e = cudaMemsetAsync(ws, 0, off[2], stream);
  if (e != cudaSuccess) return e;
  const int sms = tc::sm_count();
  const int grid = (int)std::min<int64_t>((E + 255) / 256, (int64_t)sms * 8);
  bucket_count_kernel<<<grid, 256, 0, stream>>>(idx, (int)E, N, bcount, dw, status);
  bucket_scan_kernel<<<1, 1024, 0, stream>>>(bcount, (int)nb, cursor, items, n_items);
  bucket_scatter_kernel<<<grid, 256, 0, stream>>>(idx, (int)E, N, cursor, list);
  bucket_sort_kernel<<<(unsigned)max_items, kReadWarps * 32, 0, stream>>>(idx, items, n_items,
                                                                           list, pieces, n_pieces);
  // persistent: 4 CTAs of 8 warps per SM (64 registers a thread), a warp per piece
  const int grid2 = (int)std::min<int64_t>((E + kReadWarps - 1) / kReadWarps, (int64_t)sms * 4);
  if (value_dtype == PKM_BF16)
    row_grad_kernel<true><<<grid2, kReadWarps * 32, 0, stream>>>(values, d_v, H * k, w, dout,
                                                                 list, pieces, n_pieces, dw,
                                                                 dvalues);
  else
    row_grad_kernel<false><<<grid2, kReadWarps * 32, 0, stream>>>(values, d_v, H * k, w, dout,
                                                                  list, pieces, n_pieces, dw,
                                                                  dvalues);
  return cudaGetLastError();
}

cudaError_t launch_backward_scores(cublasHandle_t blas, const uint16_t* q,
                                   const uint16_t* subkeys, int B, int H, int d_q, int n_keys,
                                   int k, const int64_t* idx, const float* w, const float* dw,
                                   float* dq, float* dsubkeys, void* workspace,
                                   void* blas_workspace, size_t blas_workspace_bytes,
                                   cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  if (k > 32) return cudaErrorInvalidValue;
  __nv_bfloat16* ds = static_cast<__nv_bfloat16*>(workspace);
  // warps per block: up to 8 while their rows fit the default 48 KB; one
  // warp (up to 181 KB for the largest n) past that
  const size_t row_bytes = (size_t)n_keys * 4;
  const int wpb = (int)std::max<size_t>(1, std::min<size_t>(8, (48u << 10) / row_bytes));
  const size_t sm = wpb * row_bytes;
  cudaError_t e;
  if (sm > (48u << 10)) {
    e = cudaFuncSetAttribute(ds_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
  }
  const int64_t items = (int64_t)B * H * 2;
  ds_rows_kernel<<<(unsigned)((items + wpb - 1) / wpb), wpb * 32, sm, stream>>>(
      idx, w, dw, B, H, n_keys, k, ds);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // setting the stream puts cuBLAS back on its own workspace pool: hand it
  // the preallocated one again, so no call allocates
  if (cublasSetStream(blas, stream) != CUBLAS_STATUS_SUCCESS ||
      cublasSetWorkspace(blas, blas_workspace, blas_workspace_bytes) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorUnknown;
  const int hd = d_q / 2;
  const float one = 1.0f, zero = 0.0f;
  // dq (row-major [B][H*d_q], block (h, half) at column offset (2h + half) * hd):
  // column-major dq^T (hd x B) = C_half^T (hd x n) * DS^T (n x B)
  cublasStatus_t st = cublasGemmStridedBatchedEx(
      blas, CUBLAS_OP_N, CUBLAS_OP_N, hd, B, n_keys, &one, subkeys, CUDA_R_16BF, hd,
      (long long)n_keys * hd, ds, CUDA_R_16BF, n_keys, (long long)B * n_keys, &zero, dq,
      CUDA_R_32F, H * d_q, hd, 2 * H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  // dsubkeys (row-major [n][hd] per block) += DS^T q_half:
  // column-major dC^T (hd x n) += q_half^T (hd x B) * DS (B x n)
  st = cublasGemmStridedBatchedEx(
      blas, CUBLAS_OP_N, CUBLAS_OP_T, hd, n_keys, B, &one, q, CUDA_R_16BF, H * d_q, hd, ds,
      CUDA_R_16BF, n_keys, (long long)B * n_keys, &one, dsubkeys, CUDA_R_32F, hd,
      (long long)n_keys * hd, 2 * H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

}  // namespace pkm
