// Steps a1-a3 for bf16 queries and subkeys on SM pairs: subkey scoring with
// two-SM tcgen05 MMAs, the per-half exact top-KL selection fused into the
// epilogue.
//
// Product-Key Memory, "Factorising the key space": a full key is a pair of
// subkeys, one per query half, scored q1.c1_a + q2.c2_b; the global top-k
// lies inside top_k(half 1) x top_k(half 2).  Code listing (forward):
// q.chunk(2), per-half `q_i @ subkeys[i].T` and topk.  This kernel computes
// the per-half scores and top-KL lists; lookup_merge.cu forms the k^2 sums.
//
// What bounds the scoring on GB300 is the bytes each SM receives through
// TMA: a one-SM MMA of M = 128 query rows needs a 128-row subkey slab for
// every 128 rows of queries.  Here the two CTAs of a cluster run one MMA of
// M = 256 rows (128 per CTA) and N = 256 keys, each CTA loading its own 128
// query rows and HALF of the subkey slab (128 keys), so a subkey byte feeds
// twice the rows.
//
// A work unit is (256-query pair tile, head, half); clusters are persistent
// over units.  Per CTA:
//   warp 0     TMA producer: 128x64 query slab + 128x64 subkey half-slab per
//              stage (bf16, 128-byte swizzle), 32 KB stages; completions are
//              signalled on the leader CTA's barrier (cta_group::2 form),
//              whose producer expects both CTAs' bytes.
//   warp 1     allocates TMEM jointly with the peer (512 columns: two 256-
//              column score buffers); in the leader CTA (rank 0) lane 0
//              issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and
//              commits to both CTAs' barriers.
//   epilogue   one or two sets of four warps, one thread per query row (its
//              TMEM lane).  Two sets (the default) own one TMEM buffer each
//              and take every other unit, so the selection work of two
//              units overlaps; one set reads both buffers in turn.
// Selection per row (exact top-KL of the half's n scores): scores above a
// threshold are appended to a log in shared memory; folds sort the log into
// the register-resident best KL (values and columns), empty it and raise
// the threshold to the KL-th value (helpers below).
// Every mbarrier wait is bounded; on time-out the kernel records
// PKM_ERR_TIMEOUT, stops issuing, and both CTAs meet at the final cluster
// barrier before TMEM is freed.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "pkm_internal.cuh"
#include "select_net.cuh"
#include "tc_common.cuh"

namespace pkm {
namespace {

using namespace tc;

constexpr int BM = 128;                 // query rows per CTA (TMEM lanes)
constexpr int NP = 256;                 // keys per chunk: the pair MMA's N
constexpr int NH = NP / 2;              // keys of a chunk loaded by each CTA
constexpr int BK = 64;                  // bf16 elements per k-slab (one 128-byte swizzle row)
constexpr int A_BYTES = BM * BK * 2;    // 16 KiB
constexpr int B_BYTES = NH * BK * 2;    // 16 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TBUFS = 2;
constexpr uint32_t TMEM_COLS = TBUFS * NP;  // 512: all of TMEM
constexpr int LOG_CAP = 64;                 // log slots per row
constexpr int LOG_STEP = BM * 8;            // bytes from one slot of a row to the next
constexpr int LOG_BYTES = LOG_CAP * LOG_STEP;

// Epilogue forms.  kEpiOneSet: four warps read both TMEM buffers in turn
// (the MMA fills one while they read the other), 5 tile stages.
// kEpiTwoSets: two sets of four warps own one buffer each and take every
// other unit, so two units' selection work overlaps; 3 tile stages leave
// room for the second log.
constexpr int kEpiOneSet = 1, kEpiTwoSets = 2;

template <int kEpi>
struct Shape2 {
  static constexpr int kStages = kEpi == kEpiTwoSets ? 3 : 5;
  static constexpr int kSets = kEpi == kEpiTwoSets ? 2 : 1;  // epilogue warp sets
  static constexpr int kThreads = 64 + kSets * 128;
  static constexpr int kTiles = kStages * STAGE_BYTES;
  static constexpr int kSmem = kTiles + kSets * LOG_BYTES + 1024;  // + alignment slack
  static_assert(kSmem <= 227 * 1024, "two-SM selection kernel shared memory");
};

// ---------------------------------------------------- selection helpers
//
// Per row, the selection state is V / C: the values and columns of the best
// KL scores folded so far, sorted by value (registers), and a log of newer
// candidates in shared memory: 8-byte entries (score bits, column) in
// [slot][row] layout (a warp's 32 rows fall in distinct banks), filled from
// both ends (bottom slots [0, nA) and top slots [tB, LOG_CAP)).  A fold
// sorts the log's entries into V / C and empties the log; the KL-th value
// becomes the threshold, and later scores are logged only when above it
// (their columns are higher than every logged one, so a later equal score
// could never be selected).  Appends use byte offsets oA (next free bottom
// slot) and oB (next free top slot) from the row's slot 0.
//
// The sorting networks compare values only; equal neighbours are then put
// in column order by a few transposition passes, run only by rows that hold
// equal values.  With both of its inputs in (score desc, column asc) order,
// the step of a merge that decides which entries stay compares columns on
// equal scores too, so the cut is exact.

struct RowLog {
  uint2* e;  // [capacity][BM]
  int row;
  __device__ __forceinline__ uint2& at(int s) const { return e[s * BM + row]; }
};

__device__ __forceinline__ void st_shared_v2(uint32_t addr, float v, uint32_t col) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "f"(v), "r"(col) : "memory");
}

// Append the scores v[0..7] (columns c0 .. c0+7) that are above thr: even
// ones at the bottom end, odd ones at the top end.  Every store address is
// formed (plain adds, the two ends independent) before the first store, so
// no store waits for an address update.
__device__ __forceinline__ void append8(uint32_t lrow, uint32_t& oA, uint32_t& oB,
                                        const float* v, float thr, uint32_t c0) {
  uint32_t ad[8];
  uint32_t a = oA, b = oB;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t step = v[j] > thr ? (uint32_t)LOG_STEP : 0u;
    if (j & 1) {
      ad[j] = b;
      b -= step;
    } else {
      ad[j] = a;
      a += step;
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (v[j] > thr) st_shared_v2(lrow + ad[j], v[j], c0 + (uint32_t)j);
  oA = a;
  oB = b;
}

// Fold the log's entries into V / C and empty the log: blocks of 16 entries
// (entry i < nA is bottom slot i, the rest top slots tB + i - nA), each
// sorted and merged in.  Raises the threshold to the KL-th value and counts
// the values held (nv, at most KL).  Warp-uniform loop; lanes without
// entries fold -inf.
template <int KL, int CAP = LOG_CAP>
__device__ __forceinline__ void fold_log(const RowLog& L, uint32_t& oA, uint32_t& oB,
                                         float (&V)[KL], uint32_t (&C)[KL], float& thr, int& nv) {
  const int nA = (int)(oA / LOG_STEP);
  const int tB = (int)(oB / LOG_STEP) + 1;
  const int cnt = nA + (CAP - tB);
#pragma unroll 1
  for (int b0 = 0; __any_sync(0xffffffffu, cnt > b0); b0 += 16) {
    float Bv[16];
    uint32_t Bc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = b0 + j;
      const int sl = i < nA ? i : tB + i - nA;
      const uint2 t = L.at(i < cnt ? sl : 0);  // in bounds, read unconditionally
      Bv[j] = i < cnt ? __uint_as_float(t.x) : -INFINITY;
      Bc[j] = t.y;
    }
    sort_desc_payload<16>(Bv, Bc);
    order_ties<16>(Bv, Bc);
    merge_top_payload<KL, 16>(V, C, Bv, Bc);
  }
  nv = min(KL, nv + cnt);
  if (V[KL - 1] > -INFINITY) thr = fmaxf(thr, V[KL - 1]);
  oA = 0;
  oB = (uint32_t)(CAP - 1) * LOG_STEP;
}

// 16 TMEM columns of this thread's lane into registers; the empty asm after
// the wait keeps every use of the values below it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    asm volatile("" : "+r"(r[i]));
    v[i] = __uint_as_float(r[i]);
  }
}

// ---------------------------------------------------------------- kernel

// Cluster c (CTAs 2c, 2c+1; rank 0 leads) takes pair units c + i * clusters.
// Pair unit u: half u & 1, pair tile (u >> 1) / H, head (u >> 1) % H; CTA
// rank r holds query rows 256 * tile + 128 * r + [0, 128).
//
// kFlat: the flat exact top-k that the factorisation replaces (Memory
// Retrieval Mechanisms, top-k retrieval: score all keys, keep the k best).
// The columns are the n = n_keys^2 full keys of a head (tmap_c over
// [H][n][d_q]; the query map's half axis has one entry), unit u is pair tile
// u / H, head u % H, and each row's best k (score desc, flat index asc) go
// with their softmax to out_idx / out_w [B][H][k].  Run without a threshold
// hint: the selection is exact with nothing to retry.
template <int KL, int kEpi, bool kFlat>
__global__ void __launch_bounds__(Shape2<kEpi>::kThreads, 1)
select_2sm_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_c, int B, int H, int n, int nch,
                  int kb_count, float hint_z, float* __restrict__ list_v,
                  unsigned short* __restrict__ list_c, int64_t* __restrict__ out_idx,
                  float* __restrict__ out_w, int k, int* __restrict__ status, int stall,
                  int* __restrict__ clear_words, int clear_count) {
  constexpr int STAGES = Shape2<kEpi>::kStages, SETS = Shape2<kEpi>::kSets;
  constexpr int SMEM_TILES = Shape2<kEpi>::kTiles;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * STAGES + 2 * TBUFS + 1];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  // the call's retry bookkeeping starts clear: the merge after this kernel
  // counts into it (every CTA helps, also one without units)
  if (clear_words)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < clear_count;
         i += gridDim.x * blockDim.x)
      clear_words[i] = 0;
  const uint32_t rank = cluster_ctarank();
  const int slot = (int)(blockIdx.x >> 1);
  const int slots = (int)(gridDim.x >> 1);
  const int pair_tiles = (B + 2 * BM - 1) / (2 * BM);
  const int units = pair_tiles * H * (kFlat ? 1 : 2);
  const int mine = slot < units ? (units - 1 - slot) / slots + 1 : 0;
  if (mine == 0) return;  // both CTAs of the cluster alike

  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t tiles_u32 = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar_full = [&](uint32_t s) { return bar0 + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto bar_tfull = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + b); };
  auto bar_tempty = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + TBUFS + b); };
  const uint32_t bar_done = bar0 + 8u * (2 * STAGES + 2 * TBUFS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);   // leader: its producer's expect_tx (both CTAs' bytes)
      mbar_init(bar_empty(s), 1);  // the leader's MMA commit, multicast to both CTAs
    }
    for (int b = 0; b < TBUFS; ++b) {
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
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  const uint32_t tmem = s_tmem_base;
  const Ctl ctl{&s_abort, status};

  auto unit_at = [&](int i) { return slot + i * slots; };
  // unit u -> (half, pair tile, head)
  auto decode = [&](int u, int& half, int& pt, int& h) {
    half = kFlat ? 0 : (u & 1);
    const int hu = kFlat ? u : (u >> 1);
    pt = hu / H;
    h = hu - pt * H;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // (stall: a test of the bounded waits; nothing is loaded, the leader's
    // MMA wait runs out and every warp returns; no copy is ever in flight)
    if (lane == 0 && !stall) {
      uint32_t it = 0;
      bool ok = true;
      for (int i0 = 0; ok && i0 < mine; i0 += SETS)
        for (int ch = 0; ok && ch < nch; ++ch)
          for (int st = 0; ok && st < SETS && i0 + st < mine; ++st) {
            int half, pt, h;
            decode(unit_at(i0 + st), half, pt, h);
            const int row0 = pt * 2 * BM + (int)rank * BM;
            for (int kb = 0; kb < kb_count; ++kb, ++it) {
              const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
              if (!wait_phase_cluster(bar_empty(s), ph ^ 1u, ctl)) {
                ok = false;
                break;
              }
              // the leader expects both CTAs' bytes; each CTA's copies land
              // in its own stage and complete on the leader's barrier
              if (rank == 0) mbar_expect_tx(bar_full(s), 2u * STAGE_BYTES);
              const uint32_t dst = tiles_u32 + s * STAGE_BYTES;
              const uint32_t fb = mapa_shared(bar_full(s), 0);
              tma_load_4d_cg2(dst, &tmap_q, kb * BK, half, h, row0, fb);
              tma_load_3d_cg2(dst + A_BYTES, &tmap_c, kb * BK, ch * NP + (int)rank * NH,
                              kFlat ? h : h * 2 + half, fb);
            }
          }
      // the leader's last releases of this CTA's stages land before it exits
      if (ok) {
        const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_phase_drain(bar_empty(j % STAGES), (j / STAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = idesc_bf16(2 * BM, NP);
      uint32_t it = 0, cnt[SETS] = {};
      bool ok = true;
      for (int i0 = 0; ok && i0 < mine; i0 += SETS)
        for (int ch = 0; ok && ch < nch; ++ch)
          for (int st = 0; ok && st < SETS && i0 + st < mine; ++st) {
            // two sets: set st owns buffer st; one set: its chunks alternate
            const uint32_t buf = SETS == 2 ? (uint32_t)st : cnt[st] % TBUFS;
            const uint32_t use = SETS == 2 ? cnt[st] : cnt[st] / TBUFS;
            ++cnt[st];
            if (!wait_phase_cluster(bar_tempty(buf), (use & 1u) ^ 1u, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int kb = 0; kb < kb_count; ++kb, ++it) {
              const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
              if (!wait_phase_cluster(bar_full(s), ph, ctl)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t a_desc = sw128_desc(tiles_u32 + s * STAGE_BYTES);
              const uint64_t b_desc = sw128_desc(tiles_u32 + s * STAGE_BYTES + A_BYTES);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                tc_mma_cg2(tmem + buf * NP, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                           (kb | kk) != 0);
              tc_commit_cg2_mc(bar_empty(s), 3);  // the stage is free again in both CTAs
            }
            if (!ok) break;
            tc_commit_cg2_mc(bar_tfull(buf), 3);  // the chunk's scores are in both TMEMs
          }
      // every issued MMA completes before TMEM is released
      tc_commit_cg2_mc(bar_done, 1);
      wait_phase_drain(bar_done, 0);
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int set = (warp - 2) >> 2;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const RowLog L{reinterpret_cast<uint2*>(smem + SMEM_TILES + set * LOG_BYTES), row};
    const uint32_t lrow = smem_u32(&L.at(0));  // the row's slot 0
    const int need = KL < n ? KL : n;          // valid entries a full list holds
    uint32_t cnt = 0;                          // chunks of this set consumed so far
    bool ok = true;
    for (int i = set; ok && i < mine; i += SETS) {
      int half, pt, h;
      decode(unit_at(i), half, pt, h);
      float thr = -INFINITY;  // a score is logged when it is > thr
      float V[KL];
      uint32_t C[KL];
#pragma unroll
      for (int i2 = 0; i2 < KL; ++i2) {
        V[i2] = -INFINITY;
        C[i2] = 0u;
      }
      int nv = 0;  // values held in V (at most KL)
      uint32_t oA = 0, oB = (uint32_t)(LOG_CAP - 1) * LOG_STEP;
      // one step per 16 columns of the unit, then a last step that only
      // folds: the fold has a single call site (code size)
      constexpr int kGroups = NP / 16;
      const int steps = nch * kGroups;
      uint32_t base = 0, buf = 0;
#pragma unroll 1
      for (int st = 0; st <= steps; ++st) {
        // before each group, room for 16 more entries (8 per end)
        if (__any_sync(0xffffffffu, st == steps || oB < oA + 15u * LOG_STEP))
          fold_log<KL, LOG_CAP>(L, oA, oB, V, C, thr, nv);
        if (st == steps) break;
        const int ch = st / kGroups, g = (st - ch * kGroups) * 16;
        if (g == 0) {
          buf = SETS == 2 ? (uint32_t)set : cnt % TBUFS;
          const uint32_t use = SETS == 2 ? cnt : cnt / TBUFS;
          ok = __all_sync(0xffffffffu, wait_phase_cluster(bar_tfull(buf), use & 1u, ctl));
          if (!ok) break;
          tc_fence_after();
          base = lane_addr + buf * NP;
          if (ch == 0 && n > LOG_CAP && hint_z > -INFINITY) {
            // threshold hint: mean + z * spread of the chunk's scores
            // (columns >= n score exactly 0: zero-filled subkeys)
            float a1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
            for (int g2 = 0; g2 < NP; g2 += 16) {
              float v[16];
              tmem_ld16(base + g2, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                a1[j & 3] += v[j];
                a2[j & 3] = fmaf(v[j], v[j], a2[j & 3]);
              }
            }
            const float s1 = (a1[0] + a1[1]) + (a1[2] + a1[3]);
            const float s2 = (a2[0] + a2[1]) + (a2[2] + a2[3]);
            const float m = (float)(n < NP ? n : NP);
            const float mu = s1 / m;
            const float sd = sqrtf(fmaxf(s2 / m - mu * mu, 0.0f));
            thr = nextafterf(fmaf(hint_z, sd, mu), -INFINITY);  // v > thr <=> v >= hint
          }
        }
        float v[16];
        tmem_ld16(base + g, v);
        const int c0 = ch * NP + g;
        if (c0 + 16 > n) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j >= n) v[j] = -INFINITY;
        }
        append8(lrow, oA, oB, v, thr, (uint32_t)c0);
        append8(lrow, oA, oB, v + 8, thr, (uint32_t)c0 + 8u);
        if (g == NP - 16) {
          // chunk consumed: hand the TMEM buffer back to the leader's MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_tempty(buf), 0));
          ++cnt;
        }
      }
      if (!ok) break;
      const int b = pt * 2 * BM + (int)rank * BM + row;
      if constexpr (kFlat) {
        // the k best full keys and their softmax (V[0] is the largest)
        if (b < B) {
          const size_t off = ((size_t)b * H + h) * k;
          float z = 0.0f;
#pragma unroll
          for (int r = 0; r < KL; ++r)
            if (r < k) z += expf(V[r] - V[0]);
          const float inv_z = 1.0f / z;
#pragma unroll
          for (int r = 0; r < KL; ++r)
            if (r < k) {
              out_idx[off + r] = (int64_t)C[r];
              out_w[off + r] = expf(V[r] - V[0]) * inv_z;
            }
        }
        continue;
      }
      // the half's list by (score desc, subkey asc) to global memory.  A list
      // with fewer than `need` entries (the hint was above the row's KL-th
      // score) is marked by the subkey 0xffff in its first slot and selected
      // again by the retry pass.
      if (b < B) {
        const size_t off = (((size_t)b * H + h) * 2 + half) * KL;
        float4* gv = reinterpret_cast<float4*>(list_v + off);
        uint4* gc = reinterpret_cast<uint4*>(list_c + off);
#pragma unroll
        for (int i2 = 0; i2 < KL; i2 += 4)
          gv[i2 / 4] = make_float4(V[i2], V[i2 + 1], V[i2 + 2], V[i2 + 3]);
#pragma unroll
        for (int i2 = 0; i2 < KL; i2 += 8) {
          uint32_t wv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            wv[q] = (C[i2 + 2 * q] & 0xffffu) | (C[i2 + 2 * q + 1] << 16);
          if (i2 == 0 && nv < need) wv[0] = (wv[0] & 0xffff0000u) | 0xffffu;
          gc[i2 / 8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // the leader's MMAs (which write both CTAs' TMEM and read both CTAs'
  // stages) are complete, and no CTA still arrives on the other's barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host

template <int KL, int kEpi, bool kFlat = false>
cudaError_t launch_kl(const CUtensorMap& mq, const CUtensorMap& mc, int B, int H, int n, int nch,
                      int kbc, float hint_z, float* list_v, unsigned short* list_c, int* status,
                      int stall, cudaStream_t stream, int64_t* out_idx = nullptr,
                      float* out_w = nullptr, int k = 0, int* clear_words = nullptr,
                      int clear_count = 0) {
  auto kernel = select_2sm_kernel<KL, kEpi, kFlat>;
  constexpr int SMEM_BYTES = Shape2<kEpi>::kSmem;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(Shape2<kEpi>::kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;
  if (!max_clusters) {
    cfg.gridDim = dim3(2 * (tc::sm_count() / 2));
    cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  }
  const int units = (B + 2 * BM - 1) / (2 * BM) * H * (kFlat ? 1 : 2);
  cfg.gridDim = dim3(2 * (units < max_clusters ? units : max_clusters));
  return cudaLaunchKernelEx(&cfg, kernel, mq, mc, B, H, n, nch, kbc, hint_z, list_v, list_c,
                            out_idx, out_w, k, status, stall, clear_words, clear_count);
}

}  // namespace

cudaError_t launch_select_2sm(const CUtensorMap& tmap_q, const CUtensorMap& tmap_c_half, int B,
                              int H, int d_q, int n_keys, int k, float hint_z, float* list_v,
                              unsigned short* list_c, int* status, bool stall,
                              cudaStream_t stream, int epi, int* clear_words, int clear_count) {
  if (B == 0) return cudaSuccess;
  const int nch = (n_keys + NP - 1) / NP;
  const int kbc = (d_q / 2 + BK - 1) / BK;
  const int st = stall ? 1 : 0;
#define PKM_SEL2(KLv, EPIv)                                                                   \
  launch_kl<KLv, EPIv>(tmap_q, tmap_c_half, B, H, n_keys, nch, kbc, hint_z, list_v, list_c, \
                       status, st, stream, nullptr, nullptr, 0, clear_words, clear_count)
  if (epi == kEpiOneSet) return k <= 16 ? PKM_SEL2(16, kEpiOneSet) : PKM_SEL2(32, kEpiOneSet);
  return k <= 16 ? PKM_SEL2(16, kEpiTwoSets) : PKM_SEL2(32, kEpiTwoSets);
#undef PKM_SEL2
}

cudaError_t launch_select_2sm_flat(const CUtensorMap& tmap_q, const CUtensorMap& tmap_keys, int B,
                                   int H, int d_q, int N, int k, int64_t* idx, float* w,
                                   int* status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int nch = (N + NP - 1) / NP;
  const int kbc = (d_q + BK - 1) / BK;
  // one epilogue set with 5 tile stages: once a row's threshold has risen,
  // the flat search mostly compares and drops, so the tile pipeline bounds it
  // (mid_flat on GB300: 1.91 ms with two sets, 1.21 ms with one)
  return k <= 16 ? launch_kl<16, kEpiOneSet, true>(tmap_q, tmap_keys, B, H, N, nch, kbc,
                                                    -INFINITY, nullptr, nullptr, status, 0,
                                                    stream, idx, w, k)
                 : launch_kl<32, kEpiOneSet, true>(tmap_q, tmap_keys, B, H, N, nch, kbc,
                                                    -INFINITY, nullptr, nullptr, status, 0,
                                                    stream, idx, w, k);
}

}  // namespace pkm
