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
// where DS_i[b,h][a] is ds summed over the winners whose half-i subkey is a
// (nonzero for at most k subkeys).
//
// Read part (dw and dV), grouped by value row so that each selected row of V
// and of dV crosses HBM once however many selections hit it (the gradient
// rows dout, B * d_v * 4 bytes, are re-read from L2 instead):
//   bucket_count_kernel    selections per bucket of 256 consecutive rows
//                          (each selection's place in its bucket from the
//                          counting atomic);
//   bucket_scan_kernel     bucket offsets, and the work items: each bucket's
//                          list cut into chunks of at most kChunk selections;
//   bucket_scatter_kernel  selection numbers into their bucket's list (first
//                          slot + place, no atomics);
//   bucket_sort_kernel     one CTA per item: a counting sort of the chunk by
//                          row in shared memory, cut into pieces (up to
//                          kPiece selections of one row), each appended to a
//                          global list as a 64-byte record (row, count,
//                          whether the row is shared, and per selection its
//                          number, dout row and weight);
//   row_grad_kernel        persistent, 16 warps per SM; each warp walks its
//                          pieces in segments of kSegW columns through a
//                          private ring of shared-memory stages (4 to 6),
//                          every lane prefetching (cp.async) and then using
//                          only its own 4 columns of the value row, of the dV
//                          row (unless the row is shared) and of the
//                          selections' dout rows.  The value segment serves
//                          every dw of the piece, and the dV segment is
//                          written back once: a plain store when the row has
//                          one piece in one item, vector atomic adds otherwise.
// Score part, through the winning subkeys only (fp32 throughout):
//   ds_gather_kernel       one warp per (query, head): ds, DS per distinct
//                          winning subkey (winners sharing one summed in lane
//                          order), dq from those subkeys' rows (L2 gathers),
//                          and one (subkey, query, DS) contribution per
//                          distinct subkey, counted per (head, half, subkey)
//                          by an atomic add whose return is the
//                          contribution's place in its group; 8 row loads in
//                          flight per lane;
//   key_scan_kernel        the counts' offsets (one CTA);
//   key_scatter_kernel     the contributions grouped by subkey (offset +
//                          place, no atomics);
//   dsub_kernel            one warp per segment of 64 grouped contributions:
//                          each key's run in it sums DS * q_half rows (16 row
//                          loads in flight per lane, not kept in L1) and adds
//                          the sum to the key's dsubkeys row (vector atomic
//                          adds).
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "pkm_internal.cuh"
#include "tc_common.cuh"

namespace pkm {
namespace {

constexpr int kRowsPerBucket = 256;  // a row's place in its bucket fits a byte
constexpr int kChunk = 2048;         // selections one CTA sorts in shared memory
constexpr int kRec = 4;              // selections a piece record can hold
constexpr int kPiece = 4;            // selections of one row in one warp pass (<= kRec)
constexpr int kReadWarps = 8;        // warps of bucket_sort_kernel
constexpr int kSegW = 128;           // value-row columns per stage (4 per lane)
constexpr int kRgWarps = 8;          // warps per CTA of row_grad_kernel
constexpr int kRgCtas = 2;           // CTAs of row_grad_kernel per SM
// shared memory per warp (ring + metadata): two CTAs of 8 warps and their
// 1 KB reserves within an SM's 228 KB
constexpr int kRgWarpBytes = 113 * 1024 / kRgWarps;

// One piece of a row's selections (64 bytes): row; m | shared << 8; the
// row's slot in the sparse output; then per selection g < m its number e,
// its dout row b and its weight w.
struct alignas(16) PieceRec {
  int row, mf, slot, pad;
  int e[kRec];
  int b[kRec];
  float w[kRec];
};
static_assert(sizeof(PieceRec) == 64 && kRec == 4 && kPiece <= kRec, "piece record layout");

// f(std::integral_constant<int, m>) for the piece size m in 1 .. kPiece.
template <int M = 1, typename F>
__device__ __forceinline__ void with_piece_size(int m, F&& f) {
  if constexpr (M == kPiece) {
    f(std::integral_constant<int, M>{});
  } else {
    if (m == M)
      f(std::integral_constant<int, M>{});
    else
      with_piece_size<M + 1>(m, f);
  }
}

__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Selections per bucket, one thread per selection, whose place in its
// bucket's list is the count before it (the atomic add's return, kept in
// erank); with `bitmap` (the sparse output) also one bit per selected row.
__global__ void bucket_count_kernel(const int64_t* __restrict__ idx, int E, int64_t N,
                                    int* __restrict__ bcount, int* __restrict__ erank,
                                    uint32_t* __restrict__ bitmap, float* __restrict__ dw,
                                    int* __restrict__ status) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t r = idx[e];
  if (r < 0 || r >= N) {  // recorded; the selection contributes nothing
    atomicExch(status, PKM_ERR_BAD_INDEX);
    dw[e] = 0.0f;
    return;
  }
  erank[e] = atomicAdd(&bcount[r / kRowsPerBucket], 1);
  if (bitmap) atomicOr(&bitmap[r >> 5], 1u << (r & 31));
}

// One CTA of 1024 threads: exclusive scans of the bucket sizes (list
// offsets, the scatter's cursors), of their chunk counts (item numbers) and,
// with `bitmap`, of their distinct selected rows (each bucket's first slot
// in the sparse output; the total goes to *n_rows);
// item = (list start, length, bucket, bucket has a single item).
__global__ void __launch_bounds__(1024)
bucket_scan_kernel(const int* __restrict__ bcount, int nb, int* __restrict__ cursor,
                   int4* __restrict__ items, int* __restrict__ n_items,
                   const uint32_t* __restrict__ bitmap, int* __restrict__ rowoff,
                   int* __restrict__ n_rows) {
  constexpr int Q = 3;
  __shared__ int s_w[Q][32];
  __shared__ int s_carry[Q];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < Q) s_carry[threadIdx.x] = 0;
  __syncthreads();
  for (int base = 0; base < nb; base += 1024) {
    const int i = base + threadIdx.x;
    int v[Q];
    v[0] = i < nb ? bcount[i] : 0;
    v[1] = (v[0] + kChunk - 1) / kChunk;
    v[2] = 0;
    if (bitmap && i < nb) {
#pragma unroll
      for (int j = 0; j < kRowsPerBucket / 32; ++j)
        v[2] += __popc(bitmap[(int64_t)i * (kRowsPerBucket / 32) + j]);
    }
    int x[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) x[q] = v[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int y = __shfl_up_sync(0xffffffffu, x[q], o);
        if (lane >= o) x[q] += y;
      }
    }
    if (lane == 31) {
#pragma unroll
      for (int q = 0; q < Q; ++q) s_w[q][warp] = x[q];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        int a = s_w[q][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, a, o);
          if (lane >= o) a += y;
        }
        s_w[q][lane] = a;
      }
    }
    __syncthreads();
    int off[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) off[q] = s_carry[q] + (warp ? s_w[q][warp - 1] : 0) + x[q] - v[q];
    if (i < nb) {
      cursor[i] = off[0];
      if (bitmap) rowoff[i] = off[2];
      for (int j = 0; j < v[1]; ++j)
        items[off[1] + j] =
            make_int4(off[0] + j * kChunk, min(kChunk, v[0] - j * kChunk), i, v[1] == 1);
    }
    __syncthreads();
    if (threadIdx.x < Q) s_carry[threadIdx.x] += s_w[threadIdx.x][31];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *n_items = s_carry[1];
    if (bitmap) *n_rows = s_carry[2];
  }
}

// Each selection to its bucket's first slot plus its place (no atomics).
__global__ void bucket_scatter_kernel(const int64_t* __restrict__ idx, int E, int64_t N,
                                      const int* __restrict__ cursor,
                                      const int* __restrict__ erank, int* __restrict__ list) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t r = idx[e];
  if (r < 0 || r >= N) return;
  list[cursor[r / kRowsPerBucket] + erank[e]] = (int)e;
}

// One CTA per item: the item's selections sorted by row (counting sort in
// shared memory); each row's run cut into pieces of at most kPiece, each
// appended to the piece list as a PieceRec.
__global__ void __launch_bounds__(kReadWarps * 32)
bucket_sort_kernel(const int64_t* __restrict__ idx, const float* __restrict__ w, int HK,
                   const int4* __restrict__ items, const int* __restrict__ n_items,
                   const int* __restrict__ list, PieceRec* __restrict__ pieces,
                   int* __restrict__ n_pieces, const uint32_t* __restrict__ bitmap,
                   const int* __restrict__ rowoff, int64_t* __restrict__ rows_out,
                   int* __restrict__ zero_list, int* __restrict__ n_zero) {
  constexpr int R = kRowsPerBucket;
  __shared__ int s_e[kChunk];
  __shared__ int s_sorted[kChunk];
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
  for (int i = tid; i < len; i += nt) s_sorted[atomicAdd(&s_cnt[s_r[i]], 1)] = s_e[i];
  __syncthreads();
  const int npieces = s_pstart[R];
  for (int q = tid; q < npieces; q += nt) {
    int lo = 0, hi = R;  // row of piece q: s_pstart[lo] <= q < s_pstart[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pstart[mid] <= q)
        lo = mid;
      else
        hi = mid;
    }
    const int first = s_start[lo] + (q - s_pstart[lo]) * kPiece;
    const int m = min(kPiece, s_start[lo + 1] - first);
    const bool shared = !excl || s_pstart[lo + 1] - s_pstart[lo] > 1;
    int e[kRec], b[kRec];
    float wt[kRec];
#pragma unroll
    for (int g = 0; g < kRec; ++g) {
      e[g] = g < m ? s_sorted[first + g] : 0;
      b[g] = e[g] / HK;
      wt[g] = g < m ? __ldg(w + e[g]) : 0.0f;
    }
    // the sparse output: the row's slot is the bucket's first slot plus the
    // selected rows below it in the bucket (bitmap); the row's first piece in
    // this item lists it, and a shared row's slot is cleared before any
    // piece adds to it
    int slot = 0;
    if (bitmap) {
      const uint32_t* bw = bitmap + (int64_t)it.z * (R / 32);
      slot = rowoff[it.z];
      for (int j = 0; j < (lo >> 5); ++j) slot += __popc(bw[j]);
      slot += __popc(bw[lo >> 5] & ((1u << (lo & 31)) - 1u));
      if (q == s_pstart[lo]) {
        rows_out[slot] = row0 + lo;
        if (shared) zero_list[atomicAdd(n_zero, 1)] = slot;
      }
    }
    int4* out = reinterpret_cast<int4*>(pieces + s_base + q);
    out[0] = make_int4((int)(row0 + lo), m | (shared ? 1 << 8 : 0), slot, 0);
    out[1] = make_int4(e[0], e[1], e[2], e[3]);
    out[2] = make_int4(b[0], b[1], b[2], b[3]);
    out[3] = make_int4(__float_as_int(wt[0]), __float_as_int(wt[1]), __float_as_int(wt[2]),
                       __float_as_int(wt[3]));
  }
}

// Sparse output: the slots of shared rows (several pieces add to them) are
// cleared first; a slot listed twice is cleared twice.
__global__ void zero_rows_kernel(const int* __restrict__ zero_list, const int* __restrict__ n_zero,
                                 int d_v, float* __restrict__ grad_rows) {
  const int nz = *n_zero;
  const int nu = d_v >> 2;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < (int64_t)nz * nu;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t slot = zero_list[t / nu];
    reinterpret_cast<float4*>(grad_rows + slot * d_v)[t % nu] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Asynchronous copies global -> shared with an L2 cache policy (createpolicy):
// the streamed value and dV rows are marked evict-first, the dout rows (re-read
// for every selection) evict-last, so that dout stays in L2.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2;" ::"r"(dst), "l"(src),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_global_stream(float* p, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Per stage, written by lane 0 when the stage is issued: the piece's row,
// m | shared << 8, the segment's first column, whether it is the piece's
// last segment, and per selection its number and weight.
struct alignas(16) StageMeta {
  int row, mf, c0, last;
  int e[kRec];
  float w[kRec];
  int pad[4];
};

// A stage of row_grad_kernel: the value segment ([lane][8 bytes] for bf16,
// [lane][16 bytes] for fp32), the dV segment ([lane][16 bytes]; the dense
// output only) and kPiece dout segments ([lane][16 bytes]); as many stages
// per warp as its share of shared memory holds (more for the sparse output,
// which reads no dV segment, so more copies are in flight).
template <bool kBf16, bool kSparse>
struct RgLayout {
  static constexpr int kVStride = kBf16 ? 8 : 16;
  static constexpr int kDvOff = 32 * kVStride;
  static constexpr int kDoutOff = kDvOff + (kSparse ? 0 : 512);
  static constexpr int kStage = kDoutOff + 512 * kPiece;
  static constexpr int kS0 = kRgWarpBytes / (kStage + (int)sizeof(StageMeta));
  static constexpr int kStages = kS0 > 8 ? 8 : kS0;
  static_assert(kStages >= 3, "row_grad ring too shallow");
};

// One lane's 4 columns of one segment for a piece of M selections: dot
// products into part, sum_g w_g * dout[b_g] added to the dV columns (read
// from the stage, or 0 for atomic adds).
template <int M, bool kBf16, bool kSparse>
__device__ __forceinline__ void seg_compute(const unsigned char* st, int lane,
                                            const float (&wt)[kRec], float (&part)[kRec],
                                            bool copied, bool shared, float* drow,
                                            uint64_t pol_stream) {
  using Lay = RgLayout<kBf16, kSparse>;
  float x[4];
  if (kBf16) {
    const uint2 v = *reinterpret_cast<const uint2*>(st + lane * Lay::kVStride);
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
  } else {
    const float4 v = *reinterpret_cast<const float4*>(st + lane * 16);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
  float4 acc = !kSparse && copied ? *reinterpret_cast<const float4*>(st + Lay::kDvOff + lane * 16)
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
  for (int g = 0; g < M; ++g) {
    const float4 d =
        *reinterpret_cast<const float4*>(st + Lay::kDoutOff + 512 * g + lane * 16);
    part[g] = fmaf(d.x, x[0], part[g]);
    part[g] = fmaf(d.y, x[1], part[g]);
    part[g] = fmaf(d.z, x[2], part[g]);
    part[g] = fmaf(d.w, x[3], part[g]);
    acc.x = fmaf(wt[g], d.x, acc.x);
    acc.y = fmaf(wt[g], d.y, acc.y);
    acc.z = fmaf(wt[g], d.z, acc.z);
    acc.w = fmaf(wt[g], d.w, acc.w);
  }
  if (shared)
    red_add4(drow, acc.x, acc.y, acc.z, acc.w);
  else
    st_global_stream(drow, acc, pol_stream);
}

// The copies of one lane's 4 columns (column col of row `row`) of a segment
// into the stage at shared address st (the stage's first byte).
template <int M, bool kBf16, bool kSparse>
__device__ __forceinline__ void seg_issue(uint32_t st, int lane, const void* values,
                                          const float* out_rows, const float* dout, int64_t row,
                                          int64_t dst_row, int d_v, int col, const int (&b)[kRec],
                                          bool copy_dv, uint64_t pol_stream, uint64_t pol_keep) {
  using Lay = RgLayout<kBf16, kSparse>;
  const int64_t off = row * d_v + col;
  if (kBf16)
    cp_async8(st + lane * Lay::kVStride, static_cast<const uint16_t*>(values) + off, pol_stream);
  else
    cp_async16(st + lane * Lay::kVStride, static_cast<const float*>(values) + off, pol_stream);
  if (!kSparse && copy_dv)
    cp_async16(st + Lay::kDvOff + lane * 16, out_rows + dst_row * d_v + col, pol_stream);
#pragma unroll
  for (int g = 0; g < M; ++g)
    cp_async16(st + Lay::kDoutOff + 512 * g + lane * 16, dout + (int64_t)b[g] * d_v + col,
               pol_keep);
}

// Persistent, kRgWarps warps per CTA, kRgCtas CTAs per SM.  Warp gw of GW takes
// pieces gw, gw + GW, ...; each piece is walked in segments of kSegW
// columns, one stage each, S - 1 stages ahead of the one computed.
// Records are fetched 32 at a time (one per lane) and broadcast by shuffles.
// Lane l copies and uses columns c0 + 4l .. c0 + 4l + 3 of the segment only,
// so a lane waits for its own copies (cp.async groups) and no data crosses
// lanes except the dw sums.
template <bool kBf16, bool kSparse>
__global__ void __launch_bounds__(kRgWarps * 32, kRgCtas)
row_grad_kernel(const void* __restrict__ values, int d_v, const float* __restrict__ dout,
                const PieceRec* __restrict__ pieces, const int* __restrict__ n_pieces,
                float* __restrict__ dw, float* __restrict__ out_rows) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Lay = RgLayout<kBf16, kSparse>;
  constexpr int S = Lay::kStages;
  constexpr int kStageBytes = Lay::kStage;
  constexpr bool sparse = kSparse;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* ring = smem + warp * S * kStageBytes;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + kRgWarps * S * kStageBytes) + warp * S;
  const uint32_t ring_s = tc::smem_u32(ring);
  const int total = *n_pieces;
  const int GW = gridDim.x * kRgWarps, gw = blockIdx.x * kRgWarps + warp;
  const int np = gw < total ? (total - gw + GW - 1) / GW : 0;
  const int nseg = (d_v + kSegW - 1) / kSegW;
  const int ntask = np * nseg;
  const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();

  int4 r0 = make_int4(0, 0, 0, 0), r1 = r0, r2 = r0, r3 = r0;  // this lane's record
  int win = -32;                                                // first piece of the window
  int pj = -1, ps = 0;                                          // task being issued
  // the piece being issued: its value row, its output row (the value row
  // itself, or its slot in the sparse output), size, flags and dout rows
  int irow = 0, idst = 0, im = 0, ishared = 0, ib[kRec] = {0, 0, 0, 0};
  int issued = 0;

  auto issue = [&]() {
    if (issued < ntask) {
      if (ps == 0) {  // a new piece: its record from the lane that holds it
        ++pj;
        if (pj >= win + 32) {
          win = pj;
          if (win + lane < np) {
            const int4* rp =
                reinterpret_cast<const int4*>(pieces + gw + (int64_t)GW * (win + lane));
            r0 = rp[0];
            r1 = rp[1];
            r2 = rp[2];
            r3 = rp[3];
          }
        }
        const int hl = pj - win;
        irow = __shfl_sync(0xffffffffu, r0.x, hl);
        idst = sparse ? __shfl_sync(0xffffffffu, r0.z, hl) : irow;
        const int mf = __shfl_sync(0xffffffffu, r0.y, hl);
        im = mf & 0xff;
        ishared = mf >> 8;
        ib[0] = __shfl_sync(0xffffffffu, r2.x, hl);
        ib[1] = __shfl_sync(0xffffffffu, r2.y, hl);
        ib[2] = __shfl_sync(0xffffffffu, r2.z, hl);
        ib[3] = __shfl_sync(0xffffffffu, r2.w, hl);
        const int e0 = __shfl_sync(0xffffffffu, r1.x, hl), e1 = __shfl_sync(0xffffffffu, r1.y, hl);
        const int e2 = __shfl_sync(0xffffffffu, r1.z, hl), e3 = __shfl_sync(0xffffffffu, r1.w, hl);
        const int w0 = __shfl_sync(0xffffffffu, r3.x, hl), w1 = __shfl_sync(0xffffffffu, r3.y, hl);
        const int w2 = __shfl_sync(0xffffffffu, r3.z, hl), w3 = __shfl_sync(0xffffffffu, r3.w, hl);
        if (lane == 0) {  // the piece's selections, for every stage of the piece
          int4* ep = reinterpret_cast<int4*>(meta + issued % S);
          ep[1] = make_int4(e0, e1, e2, e3);
          ep[2] = make_int4(w0, w1, w2, w3);
        }
      } else if (lane == 0) {
        const int4* prev = reinterpret_cast<const int4*>(meta + (issued + S - 1) % S);
        int4* ep = reinterpret_cast<int4*>(meta + issued % S);
        ep[1] = prev[1];
        ep[2] = prev[2];
      }
      const int st = issued % S;
      const int c0 = ps * kSegW;
      // the dV segment is read (and rewritten) only for an owned row of the
      // dense output; shared rows and the sparse output start from zero
      const bool copy_dv = !sparse && !ishared;
      if (lane == 0)
        reinterpret_cast<int4*>(meta + st)[0] =
            make_int4(idst, im | (ishared << 8) | (copy_dv ? 1 << 9 : 0), c0, ps == nseg - 1);
      const int col = c0 + 4 * lane;
      if (col < d_v) {
        const uint32_t dst = ring_s + st * kStageBytes;
        with_piece_size(im, [&](auto mc) {
          seg_issue<decltype(mc)::value, kBf16, kSparse>(dst, lane, values, out_rows, dout, irow,
                                                         idst, d_v, col, ib, copy_dv, pol_stream,
                                                         pol_keep);
        });
      }
      if (++ps == nseg) ps = 0;
      ++issued;
    }
    cp_async_commit();  // one group per slot of the ring, empty ones included
    __syncwarp();
  };

  float part[kRec] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < S - 1; ++i) issue();
  for (int t = 0; t < ntask; ++t) {
    issue();
    cp_async_wait<S - 1>();  // this lane's copies of task t have landed
    const int st = t % S;
    const int4 h = reinterpret_cast<const int4*>(meta + st)[0];
    const int m = h.y & 0xff;
    const bool shared = ((h.y >> 8) & 1) != 0, copied = ((h.y >> 9) & 1) != 0;
    const int col = h.z + 4 * lane;
    if (col < d_v) {
      const float4 wv = reinterpret_cast<const float4*>(meta + st)[2];
      const float wt[kRec] = {wv.x, wv.y, wv.z, wv.w};
      const unsigned char* base = ring + st * kStageBytes;
      float* drow = out_rows + (int64_t)h.x * d_v + col;
      with_piece_size(m, [&](auto mc) {
        seg_compute<decltype(mc)::value, kBf16, kSparse>(base, lane, wt, part, copied, shared,
                                                         drow, pol_stream);
      });
    }
    if (h.w) {  // the piece's last segment: its dw
      const int4 ev = reinterpret_cast<const int4*>(meta + st)[1];
      const int es[kRec] = {ev.x, ev.y, ev.z, ev.w};
#pragma unroll
      for (int g = 0; g < kPiece; ++g) {
        if (g < m) {
          float v = part[g];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == g) dw[es[g]] = v;
        }
        part[g] = 0.0f;
      }
    }
    __syncwarp();  // the stage's metadata is read before it is reissued
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------ score part
//
// Through the selected pairs only: a winner j of (b, h) has flat index
// a_j * n + c_j and score q1 . C1[a_j] + q2 . C2[c_j], so its score gradient
// ds_j = w_j (dw_j - sum_l w_l dw_l) reaches dq1 through C1[a_j], dq2
// through C2[c_j], and C1[a_j] (C2[c_j]) through q1 (q2).  Winners sharing a
// subkey are summed first (DS, fp32).
constexpr uint32_t kNoKey = 0xffffffffu;
constexpr int kMaxChunks = 4;  // 256-wide chunks of a half-query: d_q / 2 <= 1024
constexpr int kGatherLoads = 8;  // 16-byte row loads a lane of ds_gather has in flight
constexpr int kDsubLoads = 16;   // the same for dsub_kernel
constexpr int kDsubSeg = 64;     // sorted contributions per dsub_kernel work item

// A 16-byte load of read-only data that is not kept in L1 (each query row
// serves one contribution of a group).
__device__ __forceinline__ uint4 ld_nc_no_l1(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc[c][0..8) += s[r] * row[r][c * 256 + lane * 8 .. +8) summed over the R
// bf16 rows (columns at or past hd skipped); every load is issued before the
// first multiply-add.  kNoL1: the rows bypass L1 (subkey rows, re-read by the
// queries an SM holds, are better kept there).
template <int NC, int R, bool kNoL1>
__device__ __forceinline__ void fma_rows(const uint16_t* const (&row)[R], const float (&s)[R],
                                         int hd, int lane, float (&acc)[NC][8]) {
  uint4 u[R][NC];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d0 = c * 256 + lane * 8;
      u[r][c] = d0 >= hd   ? make_uint4(0, 0, 0, 0)
                : kNoL1    ? ld_nc_no_l1(row[r] + d0)
                           : *reinterpret_cast<const uint4*>(row[r] + d0);
    }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const uint32_t uw[4] = {u[r][c].x, u[r][c].y, u[r][c].z, u[r][c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[c][2 * e] = fmaf(s[r], __uint_as_float(uw[e] << 16), acc[c][2 * e]);
        acc[c][2 * e + 1] = fmaf(s[r], __uint_as_float(uw[e] & 0xffff0000u), acc[c][2 * e + 1]);
      }
    }
}

// One warp per (query, head).  Lane j holds winner j.  dq (overwritten) from
// the distinct winning subkeys' rows; each (subkey, query, DS) contribution
// to dsubkeys goes to slot ((pair * 2 + half) * k + lane) (kNoKey where lane
// j is not the first winner of its subkey), with its place among its key's
// contributions (the count before it), key (h * 2 + half) * n + subkey.
// NC: 256-wide chunks of a half-query (hd <= NC * 256).
template <int NC>
__global__ void __launch_bounds__(256)
ds_gather_kernel(const uint16_t* __restrict__ subkeys, const int64_t* __restrict__ idx,
                 const float* __restrict__ w, const float* __restrict__ dw, int B, int H, int hd,
                 int n, int k, float* __restrict__ dq, uint32_t* __restrict__ ekey,
                 uint32_t* __restrict__ erank, float* __restrict__ eds,
                 int* __restrict__ kcount) {
  constexpr int R = kGatherLoads / NC;
  const int lane = threadIdx.x & 31;
  const int64_t pair = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (pair >= (int64_t)B * H) return;  // whole warp
  const int64_t b = pair / H;
  const int h = (int)(pair - b * H);
  const int64_t N = (int64_t)n * n;
  int64_t f = -1;
  float wj = 0.0f, dwj = 0.0f;
  if (lane < k) {
    f = idx[pair * k + lane];
    wj = w[pair * k + lane];
    dwj = dw[pair * k + lane];
  }
  const bool valid = f >= 0 && f < N;  // an index outside the table contributes nothing
  float sw = wj * dwj;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, o);
  const float ds = valid ? wj * (dwj - sw) : 0.0f;
  const int d_q = 2 * hd;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    // the winner's subkey in this half (lanes without one get distinct -1 - lane)
    const int a = valid ? (int)(half == 0 ? f / n : f % n) : -1 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, a);
    const bool first = (same & ((1u << lane) - 1u)) == 0u;
    // DS: the sum over winners sharing the subkey, in lane order
    float sum = 0.0f;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      const float v = __shfl_sync(0xffffffffu, ds, l);
      sum += ((same >> l) & 1u) ? v : 0.0f;
    }
    const bool lead = first && valid;
    // the dsubkeys contribution; its count's return is first needed after
    // the row gathers below
    const uint32_t key = (uint32_t)((h * 2 + half) * n + (lead ? a : 0));
    int rank = 0;
    if (lead) rank = atomicAdd(&kcount[key], 1);
    // dq of this half: the distinct subkeys' rows, 8 dimensions per lane and
    // 256-wide chunk, R rows per step (past the last: weight 0 on row 0)
    float acc[NC][8];
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[c][e] = 0.0f;
    const uint16_t* ctab = subkeys + (size_t)(h * 2 + half) * n * hd;
    unsigned m = __ballot_sync(0xffffffffu, lead);
#pragma unroll 1
    while (m) {
      const uint16_t* row[R];
      float sL[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int L = m ? __ffs(m) - 1 : 0;
        const int aL = __shfl_sync(0xffffffffu, a, L);
        const float v = __shfl_sync(0xffffffffu, sum, L);
        row[r] = ctab + (size_t)(m ? aL : 0) * hd;
        sL[r] = m ? v : 0.0f;
        m &= m - 1u;
      }
      fma_rows<NC, R, false>(row, sL, hd, lane, acc);
    }
    float* out = dq + pair * d_q + half * hd;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d0 = c * 256 + lane * 8;
      if (d0 < hd) {
        reinterpret_cast<float4*>(out + d0)[0] =
            make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
        reinterpret_cast<float4*>(out + d0)[1] =
            make_float4(acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
      }
    }
    if (lane < k) {
      const int64_t slot = (pair * 2 + half) * k + lane;
      ekey[slot] = lead ? key : kNoKey;
      erank[slot] = (uint32_t)rank;
      eds[slot] = sum;
    }
  }
}

// Exclusive scan of the per-key counts into koff [K + 1] (one CTA of 1024
// threads, 4096 counts per coalesced pass).
__global__ void __launch_bounds__(1024)
key_scan_kernel(const int* __restrict__ kcount, int K, int* __restrict__ koff) {
  __shared__ int warp_sums[32];
  __shared__ int s_carry;
  const int t = threadIdx.x;
  if (t == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < K; base += 4096) {
    const int i0 = base + t * 4;
    int v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = i0 + j < K ? kcount[i0 + j] : 0;
    const int local = v[0] + v[1] + v[2] + v[3];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if ((t & 31) >= o) incl += y;
    }
    if ((t & 31) == 31) warp_sums[t >> 5] = incl;
    __syncthreads();
    if (t < 32) {
      int x = warp_sums[t];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (t >= o) x += y;
      }
      warp_sums[t] = x;
    }
    __syncthreads();
    int run = s_carry + incl - local + ((t >> 5) ? warp_sums[(t >> 5) - 1] : 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i0 + j < K) koff[i0 + j] = run;
      run += v[j];
    }
    __syncthreads();
    if (t == 1023) s_carry = run;
    __syncthreads();
  }
  if (t == 0) koff[K] = s_carry;
}

// The contributions grouped by key, each at its key's offset plus its place
// (order within a key: the order of the count's atomic adds), as one record
// (key, query, DS bits, 0); the query of slot s is s / (2 k H).
__global__ void key_scatter_kernel(const uint32_t* __restrict__ ekey,
                                   const uint32_t* __restrict__ erank,
                                   const float* __restrict__ eds, int64_t S, int64_t per_query,
                                   const int* __restrict__ koff, uint4* __restrict__ rec) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < S;
       s += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t key = ekey[s];
    if (key == kNoKey) continue;
    const int pos = koff[key] + (int)erank[s];
    rec[pos] = make_uint4(key, (uint32_t)(s / per_query), __float_as_uint(eds[s]), 0u);
  }
}

// dsubkeys from the grouped contributions, one warp per segment of kDsubSeg
// of them (grid-stride): each run of one key (h, half, subkey) in the
// segment sums DS * q_half[b] over its contributions (fp32 fma) and adds the
// sum to the key's dsubkeys row (vector atomic adds: a key's contributions
// may span several segments).
template <int NC>
__global__ void __launch_bounds__(256)
dsub_kernel(const uint16_t* __restrict__ q, const int* __restrict__ koff, int K,
            const uint4* __restrict__ rec, int H, int hd, int n, float* __restrict__ dsubkeys) {
  constexpr int R = kDsubLoads / NC;
  const int lane = threadIdx.x & 31;
  const int total = koff[K];
  const int d_q = 2 * hd;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
#pragma unroll 1
  for (int seg = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); seg * kDsubSeg < total;
       seg += nwarps) {
    const int s1 = min(total, (seg + 1) * kDsubSeg);
#pragma unroll 1
    for (int e = seg * kDsubSeg; e < s1;) {
      const uint32_t key = rec[e].x;
      const int re = min(s1, koff[key + 1]);
      const int hh = (int)key / n;  // h * 2 + half
      const int h = hh >> 1, half = hh & 1;
      float acc[NC][8];
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[c][i] = 0.0f;
      // R contributions per step (past the run's end: weight 0 on its first row)
      const int rs = e;
#pragma unroll 1
      for (; e < re; e += R) {
        const uint16_t* row[R];
        float sv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const bool in = e + r < re;
          const uint4 c = rec[in ? e + r : rs];
          const uint32_t b = c.y;
          sv[r] = in ? __uint_as_float(c.z) : 0.0f;
          row[r] = q + ((size_t)b * H + h) * d_q + half * hd;
        }
        fma_rows<NC, R, true>(row, sv, hd, lane, acc);
      }
      e = re;
      float* out = dsubkeys + (size_t)key * hd;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int d0 = c * 256 + lane * 8;
        if (d0 < hd) {
          red_add4(out + d0, acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
          red_add4(out + d0 + 4, acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
        }
      }
    }
  }
}

}  // namespace

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The read part's scratch, each array 256-byte aligned: the item, piece and
// zero-list counts, the bucket sizes [nb] and the selected-row bitmap
// [nb * 8 words] (these three cleared per call, one memset), the scatter
// cursors [nb], the buckets' first sparse-output slots [nb], the items
// [max_items], the bucketed selection numbers [E], the piece records [E] and
// the sparse output's slots to clear [E].
enum { kOffHead, kOffCount, kOffBitmap, kOffCursor, kOffRowOff, kOffItems, kOffList, kOffPieces,
       kOffZero, kOffEnd };
static void read_layout(int64_t N, int64_t E, size_t* off, int64_t* nb_out, int64_t* items_out) {
  const int64_t nb = (N + kRowsPerBucket - 1) / kRowsPerBucket;
  const int64_t items = std::min(nb, E) + E / kChunk + 1;
  off[kOffHead] = 0;
  off[kOffCount] = off[kOffHead] + 256;
  off[kOffBitmap] = off[kOffCount] + align256(nb * 4);
  off[kOffCursor] = off[kOffBitmap] + align256(nb * (kRowsPerBucket / 32) * 4);
  off[kOffRowOff] = off[kOffCursor] + align256(nb * 4);
  off[kOffItems] = off[kOffRowOff] + align256(nb * 4);
  off[kOffList] = off[kOffItems] + align256(items * 16);
  off[kOffPieces] = off[kOffList] + align256(E * 4);
  off[kOffZero] = off[kOffPieces] + align256(E * sizeof(PieceRec));
  off[kOffEnd] = off[kOffZero] + align256(E * 4);
  *nb_out = nb;
  *items_out = items;
}

size_t backward_read_workspace_bytes(int B, int H, int n_keys, int k) {
  size_t off[kOffEnd + 1];
  int64_t nb, items;
  read_layout((int64_t)n_keys * n_keys, (int64_t)B * H * k, off, &nb, &items);
  return off[kOffEnd];
}

// The score part's scratch: per key (h, half, subkey) its count and offset
// (K + 1); per slot (query, head, half, winner) a key, the place among its
// key's contributions and DS; then the contributions grouped by key (one
// 16-byte record each).
static void scores_layout(int B, int H, int n_keys, int k, size_t* off) {
  const size_t K = (size_t)2 * H * n_keys, S = (size_t)B * H * 2 * k;
  off[0] = 0;                                 // kcount [K]
  off[1] = off[0] + align256(K * 4);          // koff [K + 1]
  off[2] = off[1] + align256((K + 1) * 4);    // ekey [S]
  off[3] = off[2] + align256(S * 4);          // erank [S]
  off[4] = off[3] + align256(S * 4);          // eds [S]
  off[5] = off[4] + align256(S * 4);          // rec [S]
  off[6] = off[5] + align256(S * 16);
}

size_t backward_scores_workspace_bytes(int B, int H, int n_keys, int k) {
  size_t off[7];
  scores_layout(B, H, n_keys, k, off);
  return off[6];
}

size_t backward_dw_bytes(int B, int H, int k) { return align256((size_t)B * H * k * 4); }

size_t backward_workspace_bytes(int B, int H, int n_keys, int k) {
  return backward_dw_bytes(B, H, k) + std::max(backward_read_workspace_bytes(B, H, n_keys, k),
                                               backward_scores_workspace_bytes(B, H, n_keys, k));
}

cudaError_t launch_backward_read(const void* values, int value_dtype, int B, int H, int n_keys,
                                 int d_v, int k, const int64_t* idx, const float* w,
                                 const float* dout, float* dw, float* dvalues, int64_t* rows_out,
                                 float* grad_rows, int* n_rows, void* workspace, int* status,
                                 cudaStream_t stream) {
  const bool sparse = rows_out != nullptr;
  const int64_t N = (int64_t)n_keys * n_keys, E = (int64_t)B * H * k;
  if (E > INT32_MAX || (int64_t)B * d_v / 4 > INT32_MAX) return cudaErrorInvalidValue;
  size_t off[kOffEnd + 1];
  int64_t nb, max_items;
  read_layout(N, E, off, &nb, &max_items);
  if (nb > INT32_MAX || max_items > INT32_MAX) return cudaErrorInvalidValue;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* n_items = reinterpret_cast<int*>(ws + off[kOffHead]);
  int* n_pieces = n_items + 1;
  int* n_zero = n_items + 2;
  int* bcount = reinterpret_cast<int*>(ws + off[kOffCount]);
  uint32_t* bitmap = sparse ? reinterpret_cast<uint32_t*>(ws + off[kOffBitmap]) : nullptr;
  int* cursor = reinterpret_cast<int*>(ws + off[kOffCursor]);
  int* rowoff = reinterpret_cast<int*>(ws + off[kOffRowOff]);
  int4* items = reinterpret_cast<int4*>(ws + off[kOffItems]);
  int* list = reinterpret_cast<int*>(ws + off[kOffList]);
  PieceRec* pieces = reinterpret_cast<PieceRec*>(ws + off[kOffPieces]);
  int* zero_list = reinterpret_cast<int*>(ws + off[kOffZero]);
  cudaError_t e =
      cudaMemsetAsync(ws, 0, sparse ? off[kOffCursor] : off[kOffBitmap], stream);
  if (e != cudaSuccess) return e;
  if (sparse) {  // no row selected yet
    e = cudaMemsetAsync(n_rows, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
  }
  if (B == 0) return cudaSuccess;
  const int sms = tc::sm_count();
  // the places of the selections in their buckets, between the count and the
  // scatter, in the piece records' region (written only by the sort after)
  int* erank = reinterpret_cast<int*>(ws + off[kOffPieces]);
  const unsigned eblocks = (unsigned)((E + 255) / 256);
  bucket_count_kernel<<<eblocks, 256, 0, stream>>>(idx, (int)E, N, bcount, erank, bitmap, dw,
                                                   status);
  bucket_scan_kernel<<<1, 1024, 0, stream>>>(bcount, (int)nb, cursor, items, n_items, bitmap,
                                             rowoff, n_rows);
  bucket_scatter_kernel<<<eblocks, 256, 0, stream>>>(idx, (int)E, N, cursor, erank, list);
  bucket_sort_kernel<<<(unsigned)max_items, kReadWarps * 32, 0, stream>>>(
      idx, w, H * k, items, n_items, list, pieces, n_pieces, bitmap, rowoff, rows_out, zero_list,
      n_zero);
  if (sparse)
    zero_rows_kernel<<<sms * 4, 256, 0, stream>>>(zero_list, n_zero, d_v, grad_rows);
  float* out_rows = sparse ? grad_rows : dvalues;
  auto launch = [&](auto kernel, int stages, int stage_bytes) {
    const size_t sm = (size_t)kRgWarps * stages * (stage_bytes + sizeof(StageMeta));
    // two CTAs per SM need the whole shared-memory carveout
    cudaError_t e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)sm);
    if (e2 == cudaSuccess)
      e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
    if (e2 != cudaSuccess) return e2;
    kernel<<<kRgCtas * sms, kRgWarps * 32, sm, stream>>>(values, d_v, dout, pieces, n_pieces, dw,
                                                         out_rows);
    return cudaSuccess;
  };
  if (value_dtype == PKM_BF16)
    e = sparse ? launch(row_grad_kernel<true, true>, RgLayout<true, true>::kStages,
                        RgLayout<true, true>::kStage)
               : launch(row_grad_kernel<true, false>, RgLayout<true, false>::kStages,
                        RgLayout<true, false>::kStage);
  else
    e = sparse ? launch(row_grad_kernel<false, true>, RgLayout<false, true>::kStages,
                        RgLayout<false, true>::kStage)
               : launch(row_grad_kernel<false, false>, RgLayout<false, false>::kStages,
                        RgLayout<false, false>::kStage);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_backward_scores(const uint16_t* q, const uint16_t* subkeys, int B, int H,
                                   int d_q, int n_keys, int k, const int64_t* idx, const float* w,
                                   const float* dw, float* dq, float* dsubkeys, void* workspace,
                                   cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int hd = d_q / 2;
  if (k > 32 || hd > 256 * kMaxChunks || hd % 8) return cudaErrorInvalidValue;
  size_t off[7];
  scores_layout(B, H, n_keys, k, off);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* kcount = reinterpret_cast<int*>(ws + off[0]);
  int* koff = reinterpret_cast<int*>(ws + off[1]);
  uint32_t* ekey = reinterpret_cast<uint32_t*>(ws + off[2]);
  uint32_t* erank = reinterpret_cast<uint32_t*>(ws + off[3]);
  float* eds = reinterpret_cast<float*>(ws + off[4]);
  uint4* rec = reinterpret_cast<uint4*>(ws + off[5]);
  const int K = 2 * H * n_keys;
  const int64_t S = (int64_t)B * H * 2 * k;
  cudaError_t e = cudaMemsetAsync(kcount, 0, (size_t)K * 4, stream);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (int64_t)B * H;
  const unsigned g_pairs = (unsigned)((pairs + 7) / 8);
  const int sms = tc::sm_count();
  const int nc = (hd + 255) / 256;
  auto run = [&](auto nc_tag) {
    constexpr int NC = decltype(nc_tag)::value;
    ds_gather_kernel<NC><<<g_pairs, 256, 0, stream>>>(subkeys, idx, w, dw, B, H, hd, n_keys, k,
                                                      dq, ekey, erank, eds, kcount);
    key_scan_kernel<<<1, 1024, 0, stream>>>(kcount, K, koff);
    // one thread per slot: each is a chain of two dependent loads
    key_scatter_kernel<<<(unsigned)((S + 255) / 256), 256, 0, stream>>>(
        ekey, erank, eds, S, (int64_t)2 * k * H, koff, rec);
    int per_sm = 0;  // a persistent grid: the CTAs that fit at once
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dsub_kernel<NC>, 256, 0) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    dsub_kernel<NC><<<sms * per_sm, 256, 0, stream>>>(q, koff, K, rec, H, hd, n_keys,
                                                      dsubkeys);
  };
  if (nc <= 1)
    run(std::integral_constant<int, 1>{});
  else if (nc <= 2)
    run(std::integral_constant<int, 2>{});
  else
    run(std::integral_constant<int, 4>{});
  return cudaGetLastError();
}

}  // namespace pkm
