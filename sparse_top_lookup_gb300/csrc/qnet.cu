// The query network ahead of the lookup: q = BatchNorm1d(x W^T).
//
// Product-Key Memory, code listing (module setup and forward): the query is
// an nn.Linear(dim, dim, bias=False) of the layer input followed by an
// nn.BatchNorm1d, a global constraint on the query distribution ("Keeping
// the memory in use").  With H heads of width d_q the Linear maps dim -> F =
// H * d_q features (one head in the listing).  The listing leaves the
// BatchNorm mode open; both are built:
//   inference form: per feature f, q = (z - mean[f]) / sqrt(var[f] + eps) *
//     gamma[f] + beta[f] with the running statistics, folded into
//     q = z * scale[f] + shift[f] (bn_fold_kernel);
//   training form: mean[f] and the biased variance var[f] of z over the
//     batch itself.  A first GEMM pass (kStats) writes, per 32-row block and
//     feature, the block's mean and its sum of squared deviations from it
//     (warp transpose-reduce in the epilogue; z is not stored); the blocks
//     are joined by the law of total variance (bn_batch_finalize_kernel)
//     into scale / shift; the GEMM runs again with
//     them (the same tiles and MMA order: identical z).
//
// GEMM z = x W^T on the tcgen05 tensor cores, bf16 in, fp32 accumulate, one
// persistent CTA per SM over 128 x 256 output tiles:
//   warp 0      TMA producer: 128x64 slabs of x and 256x64 slabs of W
//               (128-byte swizzle) into a 4-stage ring of 48 KB stages;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=256, K=16) into one of two 256-column accumulators,
//               so tile t+1 is multiplied while tile t is written out;
//   warps 2..5  epilogue, one thread per output row (its TMEM lane): fp32
//               accumulators -> z * scale + shift -> bf16 (nearest even) ->
//               64-byte row segments in global memory.
// Every mbarrier wait is bounded like the lookup kernel's.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "pkm_internal.cuh"
#include "tc_common.cuh"

namespace pkm {
namespace {

using namespace tc;

constexpr int QM = 128;   // rows per tile (MMA M)
constexpr int QN = 256;   // features per tile (MMA N)
constexpr int QK = 64;    // bf16 per k-slab: one 128-byte swizzle row
constexpr int QSTAGES = 4;
constexpr int QA_BYTES = QM * QK * 2;  // 16 KiB
constexpr int QB_BYTES = QN * QK * 2;  // 32 KiB
constexpr int QSTAGE_BYTES = QA_BYTES + QB_BYTES;
constexpr int QSMEM = QSTAGES * QSTAGE_BYTES + 1024;  // + alignment slack
// the two-SM form: per CTA an x slab and half (128 rows) of the W slab
constexpr int Q2STAGES = 6;
constexpr int Q2STAGE_BYTES = QA_BYTES + QB_BYTES / 2;  // 32 KiB
constexpr int Q2SMEM = Q2STAGES * Q2STAGE_BYTES + 1024;
static_assert(Q2SMEM <= 227 * 1024, "two-SM query network shared memory");
constexpr int QTHREADS = 192;

// The 32-row blocks' (mean m_b, squared-deviation sum M_b, row count n_b)
// joined by the law of total variance, in two passes over the blocks: mu =
// sum_b n_b m_b / B, then M = sum_b (M_b + n_b (m_b - mu)^2) and var = M / B
// (biased; every term of the second sum is >= 0, so nothing cancels).  A CTA
// takes 32 consecutive features (one per lane: coalesced reads) and its 32
// warps split the blocks, four independent loads in flight per thread; fp32
// with four accumulators per thread, joined in shared memory.  scale / shift fold gamma and beta as in bn_fold_kernel;
// batch_mean / batch_var may be NULL.
constexpr int kFinWarps = 32;

__global__ void __launch_bounds__(kFinWarps * 32)
bn_batch_finalize_kernel(const float* __restrict__ part_mean, const float* __restrict__ part_m2,
                         int B, int F, const float* __restrict__ gamma,
                         const float* __restrict__ beta, float eps, float* __restrict__ scale,
                         float* __restrict__ shift, float* __restrict__ batch_mean,
                         float* __restrict__ batch_var) {
  __shared__ float s_part[kFinWarps][4][32];
  __shared__ float s_mu[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int f = blockIdx.x * 32 + lane;
  const bool in = f < F;
  const int blocks = (B + 31) / 32;
  auto count = [&](int k) { return (float)min(32, B - 32 * k); };
  // pass 1: sum_b n_b m_b (blocks wid + kFinWarps * (4 i + r) to accumulator r)
  float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int k0 = wid; k0 < blocks; k0 += 4 * kFinWarps) {
    float m[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int k = k0 + r * kFinWarps;
      m[r] = in && k < blocks ? part_mean[(size_t)k * F + f] : 0.0f;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int k = k0 + r * kFinWarps;
      if (k < blocks) a[r] = fmaf(count(k), m[r], a[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) s_part[wid][r][lane] = a[r];
  __syncthreads();
  if (wid == 0) {
    float t = 0.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float u = 0.0f;
#pragma unroll
      for (int w = 0; w < kFinWarps; ++w) u += s_part[w][r][lane];
      t += u;
    }
    s_mu[lane] = t / (float)B;
  }
  __syncthreads();
  const float mu = s_mu[lane];
  // pass 2: sum_b (M_b + n_b (m_b - mu)^2)
#pragma unroll
  for (int r = 0; r < 4; ++r) a[r] = 0.0f;
  for (int k0 = wid; k0 < blocks; k0 += 4 * kFinWarps) {
    float m[4], q[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int k = k0 + r * kFinWarps;
      const bool ok = in && k < blocks;
      m[r] = ok ? part_mean[(size_t)k * F + f] : mu;
      q[r] = ok ? part_m2[(size_t)k * F + f] : 0.0f;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int k = k0 + r * kFinWarps;
      const float d = m[r] - mu;
      if (k < blocks) a[r] += fmaf(count(k) * d, d, q[r]);
    }
  }
  __syncthreads();  // pass 1's partial sums have been read
#pragma unroll
  for (int r = 0; r < 4; ++r) s_part[wid][r][lane] = a[r];
  __syncthreads();
  if (wid == 0 && in) {
    float M = 0.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float u = 0.0f;
#pragma unroll
      for (int w = 0; w < kFinWarps; ++w) u += s_part[w][r][lane];
      M += u;
    }
    const float var = M / (float)B;
    const float sc = gamma[f] / sqrtf(var + eps);
    scale[f] = sc;
    shift[f] = fmaf(-mu, sc, beta[f]);
    if (batch_mean) batch_mean[f] = mu;
    if (batch_var) batch_var[f] = var;
  }
}

__global__ void bn_fold_kernel(const float* __restrict__ gamma, const float* __restrict__ beta,
                               const float* __restrict__ mean, const float* __restrict__ var,
                               float eps, int F, float* __restrict__ scale,
                               float* __restrict__ shift) {
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= F) return;
  const float s = __fdiv_rn(gamma[f], __fsqrt_rn(var[f] + eps));
  scale[f] = s;
  shift[f] = fmaf(-mean[f], s, beta[f]);
}

// Sum over the warp's 32 lanes of each of 32 values: on return lane j holds
// the sum of every lane's a[j] (31 shuffles: each step halves the values a
// lane holds, the pair of lanes keeping complementary halves).
__device__ __forceinline__ float transpose_sum32(float (&a)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = up ? a[i] : a[i + off];
      const float keep = up ? a[i + off] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return a[0];
}

// The epilogue of one 128 x 256 output tile (row tile tm, feature tile tn),
// whose accumulators are at TMEM address taddr (this thread's lane, column
// 0): q = z * scale + shift in bf16, or (kStats) column statistics instead of
// q: for the 32 rows of the warp (block tm * 4 + quad) and each feature f, the
// mean of the block's rows inside the batch and the sum of their squared
// deviations from it, at part_mean / part_m2 [block][F].
template <bool kStats>
__device__ __forceinline__ void qnet_tile_out(uint32_t taddr, int tm, int tn, int quad, int row,
                                              int lane, int B, int F,
                                              const float* __restrict__ scale,
                                              const float* __restrict__ shift,
                                              __nv_bfloat16* __restrict__ q,
                                              float* __restrict__ part_mean,
                                              float* __restrict__ part_m2) {
  const int b = tm * QM + row;
  for (int g = 0; g < QN; g += 32) {
    const int c0 = tn * QN + g;
    if (c0 >= F) break;  // F is a multiple of 32: a group is all in or all out
    float v[32];
    tmem_ld32(taddr + g, v);
    if constexpr (kStats) {
      const bool in = b < B;
      const int nb = __popc(__ballot_sync(0xffffffffu, in));  // the block's rows in the batch
      if (nb == 0) continue;  // warp-uniform: a block past the batch writes nothing
      float a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] = in ? v[j] : 0.0f;
      const float mean = transpose_sum32(a, lane) / (float)nb;  // column c0 + lane
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        // every lane takes part in the broadcast, in the block or not
        const float mj = __shfl_sync(0xffffffffu, mean, j);
        const float d = in ? v[j] - mj : 0.0f;
        a[j] = d * d;
      }
      const float m2 = transpose_sum32(a, lane);
      const size_t o = (size_t)(tm * 4 + quad) * F + c0 + lane;
      part_mean[o] = mean;
      part_m2[o] = m2;
      continue;
    }
    const float4* sc4 = reinterpret_cast<const float4*>(scale + c0);
    const float4* sh4 = reinterpret_cast<const float4*>(shift + c0);
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 a = sc4[j], t = sh4[j];
      const __nv_bfloat162 lo =
          __floats2bfloat162_rn(fmaf(v[4 * j], a.x, t.x), fmaf(v[4 * j + 1], a.y, t.y));
      const __nv_bfloat162 hi =
          __floats2bfloat162_rn(fmaf(v[4 * j + 2], a.z, t.z), fmaf(v[4 * j + 3], a.w, t.w));
      packed[2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
      packed[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
    }
    if (b < B) {
      uint4* dst = reinterpret_cast<uint4*>(q + (size_t)b * F + c0);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
    }
  }
}

// One CTA per tile (a batch of at most one 128-row tile, or the pair form
// unavailable): persistent over 128 x 256 output tiles.
template <bool kStats>
__global__ void __launch_bounds__(QTHREADS, 1)
qnet_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            int B, int F, int dim, const float* __restrict__ scale,
            const float* __restrict__ shift, __nv_bfloat16* __restrict__ q,
            float* __restrict__ part_mean, float* __restrict__ part_m2,
            int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * QSTAGES + 4 + 1];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int tm_count = (B + QM - 1) / QM, tn_count = (F + QN - 1) / QN;
  const int slot = (int)blockIdx.x, slots = (int)gridDim.x;
  const int tiles = tm_count * tn_count;
  const int mine = slot < tiles ? (tiles - 1 - slot) / slots + 1 : 0;
  if (mine == 0) return;
  const int kb_count = (dim + QK - 1) / QK;

  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t tiles_u32 = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar_full = [&](uint32_t s) { return bar0 + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bar0 + 8u * (QSTAGES + s); };
  auto bar_tfull = [&](uint32_t b) { return bar0 + 8u * (2 * QSTAGES + b); };
  auto bar_tempty = [&](uint32_t b) { return bar0 + 8u * (2 * QSTAGES + 2 + b); };
  const uint32_t bar_done = bar0 + 8u * (2 * QSTAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < QSTAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull(b), 1);
      mbar_init(bar_tempty(b), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar_done, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  const Ctl ctl{&s_abort, status};
  auto tile_of = [&](int i, int& tm, int& tn) {
    const int t = slot + i * slots;
    tm = t / tn_count;
    tn = t - tm * tn_count;
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; ok && i < mine; ++i) {
        int tm, tn;
        tile_of(i, tm, tn);
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const uint32_t s = it % QSTAGES, ph = (it / QSTAGES) & 1u;
          if (!wait_phase(bar_empty(s), ph ^ 1u, ctl)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar_full(s), QSTAGE_BYTES);
          const uint32_t dst = tiles_u32 + s * QSTAGE_BYTES;
          tma_load_2d(dst, &tmap_x, kb * QK, tm * QM, bar_full(s));
          tma_load_2d(dst + QA_BYTES, &tmap_w, kb * QK, tn * QN, bar_full(s));
        }
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        const uint32_t first = it > (uint32_t)QSTAGES ? it - QSTAGES : 0u;
        for (uint32_t j = first; j < it; ++j) wait_phase_drain(bar_full(j % QSTAGES), (j / QSTAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(QM, QN);
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; ok && i < mine; ++i) {
        const uint32_t buf = i & 1u, use = i >> 1;
        if (!wait_phase(bar_tempty(buf), (use & 1u) ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * QN;
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const uint32_t s = it % QSTAGES, ph = (it / QSTAGES) & 1u;
          if (!wait_phase(bar_full(s), ph, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sw128_desc(tiles_u32 + s * QSTAGE_BYTES);
          const uint64_t b_desc = sw128_desc(tiles_u32 + s * QSTAGE_BYTES + QA_BYTES);
#pragma unroll
          for (int kk = 0; kk < QK / 16; ++kk)
            tc_mma(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc, (kb | kk) != 0);
          tc_commit(bar_empty(s));
        }
        if (!ok) break;
        tc_commit(bar_tfull(buf));
      }
      tc_commit(bar_done);
      wait_phase_drain(bar_done, 0);
    }
  } else {
    // ------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    for (int i = 0; i < mine; ++i) {
      int tm, tn;
      tile_of(i, tm, tn);
      const uint32_t buf = i & 1u, use = i >> 1;
      if (!__all_sync(0xffffffffu, wait_phase(bar_tfull(buf), use & 1u, ctl))) break;
      tc_fence_after();
      qnet_tile_out<kStats>(lane_addr + buf * QN, tm, tn, quad, row, lane, B, F, scale, shift, q,
                            part_mean, part_m2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
  }
}

// The two-SM form (batches of at least two row tiles): clusters of two CTAs
// on row tiles 2p and 2p + 1 of one feature tile issue one MMA of M = 256
// rows (128 in each CTA) and N = 256 features, each CTA loading its own x
// slab and half (128 rows) of the W slab, so for the same MMA work an SM
// receives 32 KB per k-slab instead of 48 KB.  As in the two-SM selection
// kernel: both CTAs' copies complete on the leader CTA's full barrier, whose
// producer expects both CTAs' bytes; the leader's MMA warp issues
// tcgen05.mma.cta_group::2 and commits to both CTAs' barriers; the epilogue
// warps of both CTAs hand a TMEM buffer back on the leader's barrier; TMEM is
// allocated and freed jointly.  A CTA whose row tile is past the batch loads
// zero-filled x rows for its partner's sake and stores nothing.
template <bool kStats>
__global__ void __launch_bounds__(QTHREADS, 1)
qnet2_kernel(const __grid_constant__ CUtensorMap tmap_x,
             const __grid_constant__ CUtensorMap tmap_w_half, int B, int F, int dim,
             const float* __restrict__ scale, const float* __restrict__ shift,
             __nv_bfloat16* __restrict__ q, float* __restrict__ part_mean,
             float* __restrict__ part_m2, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * Q2STAGES + 4 + 1];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int tm_count = (B + QM - 1) / QM, tn_count = (F + QN - 1) / QN;
  const uint32_t rank = cluster_ctarank();
  const int slot = (int)(blockIdx.x >> 1), slots = (int)(gridDim.x >> 1);
  const int tiles = (tm_count + 1) / 2 * tn_count;
  const int mine = slot < tiles ? (tiles - 1 - slot) / slots + 1 : 0;
  if (mine == 0) return;  // both CTAs of the cluster alike
  const int kb_count = (dim + QK - 1) / QK;

  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t tiles_u32 = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar_full = [&](uint32_t s) { return bar0 + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bar0 + 8u * (Q2STAGES + s); };
  auto bar_tfull = [&](uint32_t b) { return bar0 + 8u * (2 * Q2STAGES + b); };
  auto bar_tempty = [&](uint32_t b) { return bar0 + 8u * (2 * Q2STAGES + 2 + b); };
  const uint32_t bar_done = bar0 + 8u * (2 * Q2STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Q2STAGES; ++s) {
      mbar_init(bar_full(s), 1);   // leader: its producer's expect_tx (both CTAs' bytes)
      mbar_init(bar_empty(s), 1);  // the leader's MMA commit, multicast to both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull(b), 1);   // the leader's MMA commit, multicast
      mbar_init(bar_tempty(b), 8);  // leader: four epilogue warps of each CTA
    }
    mbar_init(bar_done, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates, jointly for the pair
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  const uint32_t tmem = s_tmem_base;
  const Ctl ctl{&s_abort, status};
  // the cluster's tile i: pair tile (row tiles 2p, 2p + 1) and feature tile
  auto tile_of = [&](int i, int& tp, int& tn) {
    const int t = slot + i * slots;
    tp = t / tn_count;
    tn = t - tp * tn_count;
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; ok && i < mine; ++i) {
        int tp, tn;
        tile_of(i, tp, tn);
        const int row0 = (2 * tp + (int)rank) * QM;
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const uint32_t s = it % Q2STAGES, ph = (it / Q2STAGES) & 1u;
          if (!wait_phase_cluster(bar_empty(s), ph ^ 1u, ctl)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(bar_full(s), 2u * Q2STAGE_BYTES);
          const uint32_t dst = tiles_u32 + s * Q2STAGE_BYTES;
          const uint32_t fb = mapa_shared(bar_full(s), 0);
          tma_load_2d_cg2(dst, &tmap_x, kb * QK, row0, fb);
          tma_load_2d_cg2(dst + QA_BYTES, &tmap_w_half, kb * QK, tn * QN + (int)rank * (QN / 2),
                          fb);
        }
      }
      // the leader's last releases of this CTA's stages land before it exits
      if (ok) {
        const uint32_t first = it > (uint32_t)Q2STAGES ? it - Q2STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_phase_drain(bar_empty(j % Q2STAGES), (j / Q2STAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = idesc_bf16(2 * QM, QN);
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; ok && i < mine; ++i) {
        const uint32_t buf = i & 1u, use = i >> 1;
        if (!wait_phase_cluster(bar_tempty(buf), (use & 1u) ^ 1u, ctl)) break;
        tc_fence_after();
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const uint32_t s = it % Q2STAGES, ph = (it / Q2STAGES) & 1u;
          if (!wait_phase_cluster(bar_full(s), ph, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sw128_desc(tiles_u32 + s * Q2STAGE_BYTES);
          const uint64_t b_desc = sw128_desc(tiles_u32 + s * Q2STAGE_BYTES + QA_BYTES);
#pragma unroll
          for (int kk = 0; kk < QK / 16; ++kk)
            tc_mma_cg2(tmem + buf * QN, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                       (kb | kk) != 0);
          tc_commit_cg2_mc(bar_empty(s), 3);  // the stage is free again in both CTAs
        }
        if (!ok) break;
        tc_commit_cg2_mc(bar_tfull(buf), 3);  // the tile's sums are in both TMEMs
      }
      // every issued MMA completes before TMEM is released
      tc_commit_cg2_mc(bar_done, 1);
      wait_phase_drain(bar_done, 0);
    }
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    for (int i = 0; i < mine; ++i) {
      int tp, tn;
      tile_of(i, tp, tn);
      const uint32_t buf = i & 1u, use = i >> 1;
      if (!__all_sync(0xffffffffu, wait_phase_cluster(bar_tfull(buf), use & 1u, ctl))) break;
      tc_fence_after();
      qnet_tile_out<kStats>(lane_addr + buf * QN, 2 * tp + (int)rank, tn, quad, row, lane, B, F,
                            scale, shift, q, part_mean, part_m2);
      // tile written: hand the TMEM buffer back to the leader's MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_tempty(buf), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  // the leader's MMAs (which write both CTAs' TMEM and read both CTAs'
  // stages) are complete, and no CTA still arrives on the other's barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_bn_fold(const float* gamma, const float* beta, const float* mean,
                           const float* var, float eps, int F, float* scale, float* shift,
                           cudaStream_t stream) {
  bn_fold_kernel<<<(F + 255) / 256, 256, 0, stream>>>(gamma, beta, mean, var, eps, F, scale,
                                                      shift);
  return cudaGetLastError();
}

namespace {

// The GEMM z = x W^T with either epilogue: q = z * scale + shift (bf16), or
// (kStats) the per-block column statistics.
template <bool kStats>
cudaError_t launch_qnet_gemm(const uint16_t* x, const uint16_t* w, int B, int dim, int F,
                             const float* scale, const float* shift, uint16_t* q,
                             float* part_mean, float* part_m2, int* status, cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap mx, mw, mwh;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)dim, (cuuint64_t)B};
    const cuuint64_t strides[1] = {(cuuint64_t)dim * 2};
    const cuuint32_t box[2] = {QK, QM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)dim, (cuuint64_t)F};
    const cuuint64_t strides[1] = {(cuuint64_t)dim * 2};
    const cuuint32_t box[2] = {QK, QN};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    // the same view in half-slab boxes (128 rows): each CTA of the two-SM
    // form loads its half of each W slab
    const cuuint32_t hbox[2] = {QK, QN / 2};
    if (enc(&mwh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims, strides,
            hbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int tm_count = (B + QM - 1) / QM, tn_count = (F + QN - 1) / QN;
  auto q16 = reinterpret_cast<__nv_bfloat16*>(q);
  // the two-SM form when there are at least two row tiles
  if (tm_count >= 2) {
    auto kernel = qnet2_kernel<kStats>;
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Q2SMEM);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(QTHREADS);
    cfg.dynamicSmemBytes = Q2SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_clusters = 0;
    if (!max_clusters) {
      cfg.gridDim = dim3(2 * (sm_count() / 2));
      cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    }
    const int pair_tiles = (tm_count + 1) / 2 * tn_count;
    cfg.gridDim = dim3(2 * (pair_tiles < max_clusters ? pair_tiles : max_clusters));
    return cudaLaunchKernelEx(&cfg, kernel, mx, mwh, B, F, dim, scale, shift, q16, part_mean,
                              part_m2, status);
  }
  auto kernel = qnet_kernel<kStats>;
  static bool attr_set1 = false;
  if (!attr_set1) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QSMEM);
    if (e != cudaSuccess) return e;
    attr_set1 = true;
  }
  const int tiles = tm_count * tn_count;
  const int grid = tiles < sm_count() ? tiles : sm_count();
  kernel<<<grid, QTHREADS, QSMEM, stream>>>(mx, mw, B, F, dim, scale, shift, q16, part_mean,
                                           part_m2, status);
  return cudaGetLastError();
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

cudaError_t launch_qnet(const uint16_t* x, const uint16_t* w, int B, int dim, int F,
                        const float* scale, const float* shift, uint16_t* q, int* status,
                        cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_qnet_gemm<false>(x, w, B, dim, F, scale, shift, q, nullptr, nullptr, status,
                                 stream);
}

size_t qnet_batch_workspace_bytes(int B, int F) {
  const size_t blocks = ((size_t)B + 31) / 32;
  return 2 * align256(blocks * F * 4) + 2 * align256((size_t)F * 4);
}

cudaError_t launch_qnet_batch(const uint16_t* x, const uint16_t* w, int B, int dim, int F,
                              const float* gamma, const float* beta, float eps, void* workspace,
                              uint16_t* q, float* batch_mean, float* batch_var, int* status,
                              cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t blocks = ((size_t)B + 31) / 32;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* part_mean = reinterpret_cast<float*>(ws);
  float* part_m2 = reinterpret_cast<float*>(ws + align256(blocks * F * 4));
  float* scale = reinterpret_cast<float*>(ws + 2 * align256(blocks * F * 4));
  float* shift = scale + align256((size_t)F * 4) / 4;
  cudaError_t e = launch_qnet_gemm<true>(x, w, B, dim, F, nullptr, nullptr, nullptr, part_mean,
                                         part_m2, status, stream);
  if (e != cudaSuccess) return e;
  bn_batch_finalize_kernel<<<(F + 31) / 32, kFinWarps * 32, 0, stream>>>(
      part_mean, part_m2, B, F, gamma, beta, eps, scale, shift, batch_mean, batch_var);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_qnet_gemm<false>(x, w, B, dim, F, scale, shift, q, nullptr, nullptr, status,
                                 stream);
}

}  // namespace pkm

namespace {
// device status word for pkm_query_net calls that pass none
__device__ int g_qnet_status;

bool qnet_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

extern "C" int pkm_bn_fold(const float* gamma, const float* beta, const float* running_mean,
                           const float* running_var, float eps, int F, float* scale, float* shift,
                           void* stream) {
  if (!gamma || !beta || !running_mean || !running_var || !scale || !shift || F < 1)
    return PKM_ERR_INVALID;
  return pkm::launch_bn_fold(gamma, beta, running_mean, running_var, eps, F, scale, shift,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKM_OK
             : PKM_ERR_CUDA;
}

extern "C" size_t pkm_query_net_batch_workspace_bytes(int B, int F) {
  if (B < 0 || F < 1) return 0;
  return pkm::qnet_batch_workspace_bytes(B, F);
}

extern "C" int pkm_query_net_batch(const void* x, const void* weight, int B, int dim, int F,
                                   const float* gamma, const float* beta, float eps,
                                   void* workspace, void* q, float* batch_mean, float* batch_var,
                                   int* status, void* stream) {
  if (B < 0 || dim < 1 || F < 1 || !(eps >= 0.0f)) return PKM_ERR_INVALID;
  if (dim % 16 || F % 32) return PKM_ERR_UNSUPPORTED;
  if ((int64_t)(B + 31) / 32 * F > INT32_MAX) return PKM_ERR_RANGE;
  if (B == 0) return PKM_OK;
  if (!x || !weight || !gamma || !beta || !workspace || !q) return PKM_ERR_INVALID;
  if (!qnet_aligned16(x) || !qnet_aligned16(weight) || !qnet_aligned16(workspace) ||
      !qnet_aligned16(q))
    return PKM_ERR_ALIGN;
  int* st = status;
  if (!st) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qnet_status) != cudaSuccess) return PKM_ERR_CUDA;
    st = static_cast<int*>(p);
  }
  return pkm::launch_qnet_batch(static_cast<const uint16_t*>(x),
                                static_cast<const uint16_t*>(weight), B, dim, F, gamma, beta, eps,
                                workspace, static_cast<uint16_t*>(q), batch_mean, batch_var, st,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKM_OK
             : PKM_ERR_CUDA;
}

extern "C" int pkm_query_net(const void* x, const void* weight, int B, int dim, int F,
                             const float* scale, const float* shift, void* q, int* status,
                             void* stream) {
  if (B < 0 || dim < 1 || F < 1) return PKM_ERR_INVALID;
  if (dim % 16 || F % 32) return PKM_ERR_UNSUPPORTED;
  if (B == 0) return PKM_OK;
  if (!x || !weight || !scale || !shift || !q) return PKM_ERR_INVALID;
  if (!qnet_aligned16(x) || !qnet_aligned16(weight) || !qnet_aligned16(scale) ||
      !qnet_aligned16(shift) || !qnet_aligned16(q))
    return PKM_ERR_ALIGN;
  int* st = status;
  if (!st) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qnet_status) != cudaSuccess) return PKM_ERR_CUDA;
    st = static_cast<int*>(p);
  }
  return pkm::launch_qnet(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(weight), B,
                          dim, F, scale, shift, static_cast<uint16_t*>(q), st,
                          static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKM_OK
             : PKM_ERR_CUDA;
}
