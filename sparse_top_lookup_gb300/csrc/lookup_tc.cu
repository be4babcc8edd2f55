// Steps a1-a5 for bf16 queries and subkeys: subkey scoring on the tcgen05
// tensor cores with the whole selection fused into the epilogue.
//
// Product-Key Memory, "Factorising the key space": a full key is a pair of
// subkeys, one per query half, and its score is q1.c1_a + q2.c2_b; the
// global top-k lies inside top_k(half 1) x top_k(half 2), so per-half top-k
// lists, their k^2 pairwise sums and a final top-k are exact.  Code listing
// (forward): q.chunk(2) halves, per-half `q_i @ subkeys[i].T` then topk, k^2
// sums with flat index i1 * n_keys + i2, topk, softmax.
//
// One CTA owns 128 queries x one head at a time (persistent over tiles):
//   warp 0      TMA producer: 128x64 query slabs and NCx64 subkey slabs
//               (bf16, 128-byte swizzle) into a 3-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=NC<=256, K=16, fp32 accumulate) into one of two
//               TMEM buffers, so scoring chunk c+1 overlaps the epilogue of c;
//   warps 2..5  epilogue, one thread per query row (= TMEM lane): reads its
//               row's scores 32 columns at a time with tcgen05.ld and keeps
//               an exact running top-KL list in registers (ties: lower subkey
//               index first, since columns arrive in increasing order), then
//               merges the two halves' lists and applies the softmax.
// Scores never leave the SM.  Every mbarrier wait is bounded; on time-out
// the kernel records PKM_ERR_TIMEOUT, stops issuing work, waits (bounded) for
// its own copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "pkm_internal.cuh"

namespace pkm {
namespace {

constexpr int BM = 128;             // query rows per tile (MMA M)
constexpr int BK = 64;              // bf16 elements per k-slab: one 128-byte swizzle row
constexpr int NCMAX = 256;          // subkeys per chunk (MMA N)
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;     // 16 KiB
constexpr int B_BYTES = NCMAX * BK * 2;  // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SLOTS = 32;                       // per-row queue / list slots
constexpr int AREA_BYTES = SLOTS * BM * 8;      // [slot][row] fp32 scores + int32 indices
constexpr int SMEM_TILES = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = SMEM_TILES + 2 * AREA_BYTES + 1024;  // + alignment slack
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row swizzle atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------- bounded waits

struct Ctl {
  volatile int* abort;
  int* status;
};

// Waits for the phase of the given parity; false on time-out or abort.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*ctl.abort) return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      *ctl.abort = 1;
      atomicExch(ctl.status, PKM_ERR_TIMEOUT);
      return false;
    }
  }
}

// Teardown wait: ignores the abort flag, still bounded.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > WAIT_LIMIT_NS) return;
}

// ---------------------------------------------------- selection helpers

// Insert (x, xi) into V (sorted descending, KL entries) with payload I.  A
// new entry goes after existing equal scores, so arrival order breaks ties.
// Every position is computed independently from the old list.
template <int KL>
__device__ __forceinline__ void insert_sorted(float (&V)[KL], int (&I)[KL], float x, int xi) {
#pragma unroll
  for (int i = KL - 1; i >= 1; --i) {
    const bool gi = x > V[i];
    const bool gp = x > V[i - 1];
    V[i] = gp ? V[i - 1] : (gi ? x : V[i]);
    I[i] = gp ? I[i - 1] : (gi ? xi : I[i]);
  }
  const bool g0 = x > V[0];
  V[0] = g0 ? x : V[0];
  I[0] = g0 ? xi : I[0];
}

// Fold 32 new scores (columns col0 .. col0+31, increasing) into the row's
// running top-KL.  Scores above the current KL-th are queued in this row's
// column of shared memory (order kept), then the warp inserts queue entries
// in lock-step; lanes whose queue is shorter insert -inf, a no-op.
template <int KL>
__device__ __forceinline__ void select_group(float (&V)[KL], int (&I)[KL], const float (&v)[32],
                                             int col0, float* qv, int* qi, int row) {
  const float T = V[KL - 1];
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (v[j] > T) {
      qv[cnt * BM + row] = v[j];
      qi[cnt * BM + row] = col0 + j;
      ++cnt;
    }
  }
  const int m = __reduce_max_sync(0xffffffffu, cnt);
  for (int t = 0; t < m; ++t) {
    float x = -INFINITY;
    int xi = 0;
    if (t < cnt) {
      x = qv[t * BM + row];
      xi = qi[t * BM + row];
    }
    insert_sorted<KL>(V, I, x, xi);
  }
}

// ---------------------------------------------------------------- kernel

template <int KL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
lookup_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_c,
                 int B, int H, int n, int k, int NC, int nch, int kb_count,
                 int64_t* __restrict__ idx, float* __restrict__ w, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * STAGES + 5];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t tiles_u32 = smem_u32(smem);
  float* q_val = reinterpret_cast<float*>(smem + SMEM_TILES);  // queue, then half-2 list
  int* q_idx = reinterpret_cast<int*>(smem + SMEM_TILES + SLOTS * BM * 4);
  float* l1_val = reinterpret_cast<float*>(smem + SMEM_TILES + AREA_BYTES);  // half-1 list
  int* l1_idx = reinterpret_cast<int*>(smem + SMEM_TILES + AREA_BYTES + SLOTS * BM * 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar_full = [&](uint32_t s) { return bar0 + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto bar_tfull = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + b); };
  auto bar_tempty = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t bar_done = bar0 + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  const Ctl ctl{&s_abort, status};

  const int row_tiles = (B + BM - 1) / BM;
  const int tiles = row_tiles * H;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint32_t tx = (uint32_t)(A_BYTES + NC * BK * 2);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
        const int rt = tile / H, h = tile - (tile / H) * H;
        for (int half = 0; ok && half < 2; ++half)
          for (int ch = 0; ok && ch < nch; ++ch)
            for (int kb = 0; kb < kb_count; ++kb) {
              const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
              if (!wait_phase(bar_empty(s), ph ^ 1u, ctl)) {
                ok = false;
                break;
              }
              mbar_expect_tx(bar_full(s), tx);
              const uint32_t a_dst = tiles_u32 + s * STAGE_BYTES;
              tma_load_4d(a_dst, &tmap_q, kb * BK, half, h, rt * BM, bar_full(s));
              tma_load_3d(a_dst + A_BYTES, &tmap_c, kb * BK, ch * NC, h * 2 + half, bar_full(s));
              ++it;
            }
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) wait_phase_drain(bar_full(j % STAGES), (j / STAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, NC);
      uint32_t it = 0, cc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x)
        for (int half = 0; ok && half < 2; ++half)
          for (int ch = 0; ok && ch < nch; ++ch, ++cc) {
            const uint32_t buf = cc & 1u, use = cc >> 1;
            if (!wait_phase(bar_tempty(buf), (use & 1u) ^ 1u, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + buf * NCMAX;
            for (int kb = 0; kb < kb_count; ++kb, ++it) {
              const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
              if (!wait_phase(bar_full(s), ph, ctl)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t a_desc = sw128_desc(tiles_u32 + s * STAGE_BYTES);
              const uint64_t b_desc = sw128_desc(tiles_u32 + s * STAGE_BYTES + A_BYTES);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                tc_mma(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc, (kb | kk) != 0);
              tc_commit(bar_empty(s));  // frees the stage once these MMAs have read it
            }
            if (!ok) break;
            tc_commit(bar_tfull(buf));  // chunk complete in TMEM
          }
      // all issued MMAs complete before TMEM is released
      tc_commit(bar_done);
      wait_phase_drain(bar_done, 0);
    }
  } else {
    // ---------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    uint32_t cc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
      const int rt = tile / H, h = tile - (tile / H) * H;
      for (int half = 0; ok && half < 2; ++half) {
        float V[KL];
        int I[KL];
#pragma unroll
        for (int i = 0; i < KL; ++i) {
          V[i] = -INFINITY;
          I[i] = 0;
        }
        for (int ch = 0; ch < nch; ++ch, ++cc) {
          const uint32_t buf = cc & 1u, use = cc >> 1;
          // every lane observes the phase; the warp leaves together on failure
          if (!__all_sync(0xffffffffu, wait_phase(bar_tfull(buf), use & 1u, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int g = 0; g < NC / 32; ++g) {
            float v[32];
            tmem_ld32(lane_addr + buf * NCMAX + g * 32, v);
            const int col0 = ch * NC + g * 32;
            if (col0 + 32 > n) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= n) v[j] = -INFINITY;
            }
            select_group<KL>(V, I, v, col0, q_val, q_idx, row);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(buf));
        }
        if (!ok) break;
        float* dv = half == 0 ? l1_val : q_val;
        int* di = half == 0 ? l1_idx : q_idx;
#pragma unroll
        for (int i = 0; i < KL; ++i) {
          dv[i * BM + row] = V[i];
          di[i * BM + row] = I[i];
        }
      }
      if (!ok) break;

      // a4: the k^2 merge as a frontier walk.  Row i of the candidate grid
      // (list-1 entry i paired with every list-2 entry) is already sorted, so
      // the next winner is the best of the rows' current heads; the t-th
      // winner can only come from rows 0..t (each earlier row head beats it).
      float fv[KL];
      int ff[KL], fp[KL];
      {
        const float s2 = q_val[row];
        const int a2 = q_idx[row];
#pragma unroll
        for (int i = 0; i < KL; ++i) {
          fv[i] = l1_val[i * BM + row] + s2;
          ff[i] = l1_idx[i * BM + row] * n + a2;
          fp[i] = 0;
        }
      }
      const int b = rt * BM + row;
      const bool live = b < B;
      int64_t* ip = idx + ((int64_t)b * H + h) * k;
      float* wp = w + ((int64_t)b * H + h) * k;
      float ov[KL];
#pragma unroll
      for (int t = 0; t < KL; ++t) {
        float bv = fv[0];
        int bf = ff[0], bi = 0, bp = fp[0];
#pragma unroll
        for (int i = 1; i <= t; ++i) {
          const bool better = fv[i] > bv || (fv[i] == bv && ff[i] < bf);
          bv = better ? fv[i] : bv;
          bf = better ? ff[i] : bf;
          bi = better ? i : bi;
          bp = better ? fp[i] : bp;
        }
        ov[t] = bv;
        if (live && t < k) ip[t] = (int64_t)bf;
        const int np = bp + 1;
        float nv = -INFINITY;
        int nf = 0;
        if (np < KL) {
          nv = l1_val[bi * BM + row] + q_val[np * BM + row];
          nf = l1_idx[bi * BM + row] * n + q_idx[np * BM + row];
        }
#pragma unroll
        for (int i = 0; i <= t; ++i) {
          if (i == bi) {
            fv[i] = nv;
            ff[i] = nf;
            fp[i] = np;
          }
        }
      }
      // a5: softmax over the k winners (largest first).
      float z = 0.0f;
#pragma unroll
      for (int t = 0; t < KL; ++t)
        if (t < k) z += expf(ov[t] - ov[0]);
      if (live) {
#pragma unroll
        for (int t = 0; t < KL; ++t)
          if (t < k) wp[t] = expf(ov[t] - ov[0]) / z;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int KL>
cudaError_t launch_kl(const CUtensorMap& mq, const CUtensorMap& mc, int B, int H, int n, int k,
                      int NC, int nch, int kbc, int64_t* idx, float* w, int* status,
                      cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(lookup_tc_kernel<KL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int tiles = (B + BM - 1) / BM * H;
  const int grid = tiles < sm_count() ? tiles : sm_count();
  lookup_tc_kernel<KL><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(mq, mc, B, H, n, k, NC, nch, kbc,
                                                                  idx, w, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lookup_tc(const uint16_t* q, const uint16_t* subkeys, int B, int H, int d_q,
                             int n_keys, int k, int64_t* idx, float* w, int* status,
                             cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int hd = d_q / 2;
  const int NC = n_keys >= NCMAX ? NCMAX : (n_keys + 31) / 32 * 32;
  const int nch = (n_keys + NC - 1) / NC;
  const int kbc = (hd + BK - 1) / BK;

  CUtensorMap mq, mc;
  {
    // q viewed as [B][H][2][hd]: innermost first.
    const cuuint64_t dims[4] = {(cuuint64_t)hd, 2, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)d_q * 2,
                                   (cuuint64_t)H * d_q * 2};
    const cuuint32_t box[4] = {BK, 1, 1, BM};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // subkeys viewed as [H*2][n][hd].
    const cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)n_keys, (cuuint64_t)H * 2};
    const cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)n_keys * hd * 2};
    const cuuint32_t box[3] = {BK, (cuuint32_t)NC, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(subkeys), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (k <= 16)
    return launch_kl<16>(mq, mc, B, H, n_keys, k, NC, nch, kbc, idx, w, status, stream);
  return launch_kl<32>(mq, mc, B, H, n_keys, k, NC, nch, kbc, idx, w, status, stream);
}

}  // namespace pkm
