// Step a6: the weighted value read.
//
// Product-Key Memory (note after the code listing): the value table is read
// by an EmbeddingBag(mode="sum") with per-sample weights, so the k selected
// rows are gathered and weight-summed in one pass and the N x d table is
// never touched as a dense matrix.  Memory Retrieval Mechanisms (top-k
// retrieval): r = sum_j alpha_j v_{i_j}.  Here one bag holds the H*k rows a
// query selected over all its heads, so the per-head reads are summed.
//
// The read is HBM-bound: every byte of a selected row is read once, the
// arithmetic is one FMA per element.  Two forms:
//   gather_bulk_kernel (rows of 512-byte multiples up to 8 KB): one
//     persistent CTA per SM streams whole rows into a shared-memory ring by
//     bulk copies (described above the kernel); an SM keeps far more bytes in
//     flight this way than with per-thread loads, whose misses in flight
//     hold an SM near 45 GB/s;
//   gather_kernel (other widths): one CTA owns one query (bag).  Each value
//     row is split into 16-byte vectors and one thread owns one vector
//     column, so a warp reads 512 contiguous bytes of a row; when a row has
//     fewer vectors than the CTA has threads, the threads form row groups
//     that take every G-th row and are reduced through shared memory at the
//     end.  Loads are 16-byte non-coherent loads that bypass L1 (each row is
//     used once per bag), unrolled eight rows deep.
// Both accumulate in fp32 (the bulk form in row order within a bag).
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
#include "tc_common.cuh"

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
// (kept small, so many CTAs fit on an SM).
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

// Bulk-copy form (one persistent CTA per SM): value rows stream into a
// shared-memory ring as whole-row bulk copies (cp.async.bulk, the SM's copy
// engine), up to ~200 KB in flight per SM.  The CTA holds `teams` teams;
// team t is an independent pipeline over bags (g * gridDim.x + blockIdx.x) *
// teams + t, g = 0, 1, ...:
//   producer  warp t: stages its bags' indices and weights (and, for an fp8
//             table, the selected rows' scales) in shared memory by cp.async
//             ahead of use; for each batch of kBatch rows, lane j waits for
//             the team's next batch slot to be free, stores row j's weight
//             beside its ring slot and issues one bulk copy of the row; the
//             batch completes on one barrier;
//   consumers vpr threads (whole warps), one 16-byte column of the rows each:
//             per batch one wait, then weight * row accumulated in fp32 over
//             the batch's rows, in row order; each warp then frees the slot.
// Every wait is bounded (2 s); on time-out the kernel records
// PKM_ERR_TIMEOUT, stops, and waits (bounded) for the copies in flight
// before it returns.
constexpr int kBatch = 8;            // rows per batch (one barrier)
constexpr int kBulkMaxTeams = 8;
constexpr int kBulkConsumers = 512;  // consumer threads per CTA at most
constexpr int kBulkThreads = 768;    // producer warps + consumers per CTA at most

template <int VT>
__global__ void __launch_bounds__(kBulkThreads, 1)
gather_bulk_kernel(const unsigned char* __restrict__ values, const float* __restrict__ scales,
                   int64_t N, int row_bytes, int rows_per_bag, int B, int teams, int nbs,
                   const int64_t* __restrict__ idx, const float* __restrict__ w,
                   float* __restrict__ out, int* __restrict__ status, int stall) {
  using namespace tc;
  constexpr int E = VecAcc<VT>::kElems;
  constexpr bool kFp8 = VT == PKM_FP8_E4M3;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  const int vpr = row_bytes / 16;
  const int cpb = (rows_per_bag + kBatch - 1) / kBatch;  // batches per bag
  const int bslots = teams * nbs;                         // batch slots, nbs per team
  const int rpb = rows_per_bag;
  // ring [bslots * kBatch][row_bytes]; then 8-byte items: full and empty
  // barriers per batch slot, staged indices [teams][3][rpb]; then 4-byte
  // items: row weights [bslots * kBatch], batch slot uses [bslots], staged
  // weights [teams][3][rpb], staged fp8 scales [teams][2][rpb]
  unsigned char* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)bslots * kBatch * row_bytes);
  int64_t* st_idx = reinterpret_cast<int64_t*>(bars + 2 * bslots);
  float* slot_w = reinterpret_cast<float*>(st_idx + (size_t)teams * 3 * rpb);
  int* last_use = reinterpret_cast<int*>(slot_w + bslots * kBatch);
  float* st_w = reinterpret_cast<float*>(last_use + bslots);
  float* st_sc = st_w + (size_t)teams * 3 * rpb;
  const uint32_t bar_full0 = smem_u32(bars), bar_empty0 = smem_u32(bars + bslots);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < bslots; ++i) {
      mbar_init(bar_full0 + 8u * i, kBatch);                 // one arrival per producer lane
      mbar_init(bar_empty0 + 8u * i, (uint32_t)(vpr / 32));  // one per consumer warp
      last_use[i] = -1;
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const Ctl ctl{&s_abort, status};
  auto bag_of = [&](int64_t g, int t) { return (g * gridDim.x + blockIdx.x) * (int64_t)teams + t; };

  if (warp < teams && stall) {
    // (stall: a test of the bounded waits; no copy is issued, so every
    // consumer's first wait runs out, the kernel records PKM_ERR_TIMEOUT and
    // every warp returns)
  } else if (warp < teams) {
    // ------------------------------------------------------------ producer
    const int t = warp;
    int64_t* my_idx = st_idx + (size_t)t * 3 * rpb;  // [3][rpb], bag g in buffer g % 3
    float* my_w = st_w + (size_t)t * 3 * rpb;
    float* my_sc = st_sc + (size_t)t * 2 * rpb;       // [2][rpb], bag g in buffer g % 2
    auto stage_rows = [&](int64_t g) {               // indices and weights of bag g
      const int64_t bag = bag_of(g, t);
      if (bag >= B) return;
      const int buf = (int)(g % 3);
      for (int j = lane; j < rpb; j += 32) {
        cp_async8(smem_u32(my_idx + buf * rpb + j), idx + bag * rpb + j);
        cp_async4(smem_u32(my_w + buf * rpb + j), w + bag * rpb + j);
      }
    };
    auto stage_scales = [&](int64_t g) {  // fp8 row scales of bag g (its indices have landed)
      if constexpr (kFp8) {
        if (bag_of(g, t) >= B) return;
        for (int j = lane; j < rpb; j += 32) {
          const int64_t r = my_idx[(g % 3) * rpb + j];
          cp_async4(smem_u32(my_sc + (g & 1) * rpb + j), scales + (r >= 0 && r < N ? r : 0));
        }
      }
    };
    stage_rows(0);
    stage_rows(1);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    stage_scales(0);
    cp_async_commit();
    bool ok = true;
    uint32_t bq = 0, ph = 0;  // the team's next batch slot and its use parity
    for (int64_t g = 0; ok && bag_of(g, t) < B; ++g) {
      // what was staged one bag ago has landed: bag g's scales, bag g+1's rows
      cp_async_wait<0>();
      __syncwarp();
      stage_rows(g + 2);
      stage_scales(g + 1);
      cp_async_commit();
      const int rb = (int)(g % 3) * rpb, sb = (int)(g & 1) * rpb;
      for (int c = 0; ok && c < cpb; ++c) {
        const uint32_t bb = (uint32_t)t * nbs + bq;
        const uint32_t full = bar_full0 + 8u * bb;
        if (lane < kBatch) {
          // slot bb's previous use was this team's batch nbs batches ago,
          // issued earlier, so the team's consumers free it
          if (!wait_phase(bar_empty0 + 8u * bb, ph ^ 1u, ctl)) {
            ok = false;
          } else {
            const int j = c * kBatch + lane;
            if (lane == 0) last_use[bb] = (int)ph;
            if (j < rpb) {
              int64_t row = my_idx[rb + j];
              float wt = my_w[rb + j];
              if (row < 0 || row >= N) {
                atomicExch(status, PKM_ERR_BAD_INDEX);
                row = 0;
                wt = 0.0f;
              } else if (kFp8) {
                wt *= my_sc[sb + j];
              }
              const uint32_t rs = bb * kBatch + lane;  // ring slot of the row
              slot_w[rs] = wt;
              mbar_expect_tx(full, (uint32_t)row_bytes);
              bulk_load(smem_u32(ring + (size_t)rs * row_bytes), values + row * row_bytes,
                        (uint32_t)row_bytes, full);
            } else {
              mbar_arrive(full);  // past the bag's end: arrival only
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (++bq == (uint32_t)nbs) {
          bq = 0;
          ph ^= 1u;
        }
      }
    }
    cp_async_wait<0>();  // no staging copy outlives the CTA
    if (!ok) {
      // only a batch slot's last use can still be in flight (each use waits
      // for the previous one to be consumed): let those copies land
      __syncwarp();
      for (int i = t * nbs + lane; i < (t + 1) * nbs; i += 32)
        if (last_use[i] >= 0) wait_phase_drain(bar_full0 + 8u * i, (uint32_t)last_use[i] & 1u);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = threadIdx.x - 32 * teams;
    const int t = ct / vpr, v = ct - (ct / vpr) * vpr;
    bool ok = true;
    uint32_t bq = 0, ph = 0;
    for (int64_t g = 0; ok && bag_of(g, t) < B; ++g) {
      const int64_t bag = bag_of(g, t);
      float acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.0f;
      for (int c = 0; c < cpb; ++c) {
        const uint32_t bb = (uint32_t)t * nbs + bq;
        if (!__all_sync(0xffffffffu, wait_phase(bar_full0 + 8u * bb, ph, ctl))) {
          ok = false;
          break;
        }
        const int nr = rpb - c * kBatch < kBatch ? rpb - c * kBatch : kBatch;
        const unsigned char* base = ring + (size_t)bb * kBatch * row_bytes + v * 16;
        const float* wb = slot_w + bb * kBatch;
        uint4 x[kBatch];
        float wt[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (u < nr) {
            x[u] = *reinterpret_cast<const uint4*>(base + (size_t)u * row_bytes);
            wt[u] = wb[u];
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (u < nr) VecAcc<VT>::fma(acc, wt[u], x[u]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty0 + 8u * bb);
        if (++bq == (uint32_t)nbs) {
          bq = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      float4* o4 = reinterpret_cast<float4*>(out + bag * (int64_t)vpr * E + v * E);
#pragma unroll
      for (int e = 0; e < E; e += 4)
        o4[e / 4] = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    }
  }
  __syncthreads();
}

// Shape of the bulk form for a row of vpr 16-byte vectors: the most teams
// (a power of two) whose staging and two batch slots each fit, or false when
// the row does not suit it (teams must be whole warps).
bool bulk_shape(int vpr, int rows_per_bag, int& teams, int& nbs, size_t& smem) {
  if (vpr % 32 || vpr > kBulkConsumers || rows_per_bag < 1) return false;
  const size_t budget = 220u * 1024u;
  const size_t per_batch = kBatch * ((size_t)vpr * 16 + 4) + 8 * 2 + 4;
  int tm = 1;
  while (tm * 2 <= kBulkMaxTeams && tm * 2 * vpr <= kBulkConsumers &&
         tm * 2 * (32 + vpr) <= kBulkThreads)
    tm *= 2;
  for (teams = tm; teams >= 1; teams /= 2) {
    const size_t staging = (size_t)teams * rows_per_bag * (3 * (8 + 4) + 2 * 4);
    if (staging + 2 * per_batch * teams > budget) continue;
    nbs = (int)((budget - staging) / (per_batch * teams));
    smem = per_batch * teams * nbs + staging;
    return true;
  }
  return false;
}

template <int VT>
cudaError_t launch_gather_vt(const void* values, int64_t N, int d_v, int B, int rows_per_bag,
                             const int64_t* idx, const float* w, float* out, int* status,
                             int ctas, bool stall, cudaStream_t stream) {
  constexpr int E = VecAcc<VT>::kElems;
  const int vpr = d_v / E;  // 16-byte vectors per row
  // an fp8 table's row scales follow its N * d_v code bytes
  const float* scales =
      VT == PKM_FP8_E4M3
          ? reinterpret_cast<const float*>(static_cast<const unsigned char*>(values) + N * d_v)
          : nullptr;
  int teams = 0, nbs = 0;
  size_t bulk_smem = 0;
  if (ctas > 0 && bulk_shape(vpr, rows_per_bag, teams, nbs, bulk_smem)) {
    static size_t smem_set = 0;
    if (bulk_smem > smem_set) {
      cudaError_t e = cudaFuncSetAttribute(
          gather_bulk_kernel<VT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bulk_smem);
      if (e != cudaSuccess) return e;
      smem_set = bulk_smem;
    }
    const int64_t want = ((int64_t)B + teams - 1) / teams;
    const int grid = want < ctas ? (int)want : ctas;
    gather_bulk_kernel<VT><<<grid, teams * (32 + vpr), bulk_smem, stream>>>(
        static_cast<const unsigned char*>(values), scales, N, vpr * 16, rows_per_bag, B, teams,
        nbs, idx, w, out, status, stall ? 1 : 0);
    return cudaGetLastError();
  }
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
  // The loads bypass L1, so the SM can keep its maximum shared-memory split.
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaError_t e = cudaFuncSetAttribute(gather_kernel<VT>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    carveout_set = true;
  }
  gather_kernel<VT><<<B, threads, smem, stream>>>(static_cast<const uint4*>(values), scales, N,
                                                  vpr, groups, rows_per_bag, idx, w, out, status);
  return cudaGetLastError();
}

}  // namespace

bool gather_bulk_ok(int value_dtype, int d_v, int rows_per_bag) {
  const int esz = value_dtype == PKM_FP8_E4M3 ? 1 : value_dtype == PKM_BF16 ? 2 : 4;
  int teams, ns;
  size_t smem;
  return (int64_t)d_v * esz % 16 == 0 && bulk_shape(d_v * esz / 16, rows_per_bag, teams, ns, smem);
}

cudaError_t launch_gather(const void* values, int value_dtype, int64_t N, int d_v, int B,
                          int rows_per_bag, const int64_t* idx, const float* w, float* out,
                          int* status, cudaStream_t stream, int ctas, bool stall) {
  if (B == 0) return cudaSuccess;
  if (value_dtype == PKM_FP8_E4M3)
    return launch_gather_vt<PKM_FP8_E4M3>(values, N, d_v, B, rows_per_bag, idx, w, out, status,
                                          ctas, stall, stream);
  if (value_dtype == PKM_BF16)
    return launch_gather_vt<PKM_BF16>(values, N, d_v, B, rows_per_bag, idx, w, out, status, ctas,
                                      stall, stream);
  return launch_gather_vt<PKM_F32>(values, N, d_v, B, rows_per_bag, idx, w, out, status, ctas,
                                   stall, stream);
}

}  // namespace pkm
