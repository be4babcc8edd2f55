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
// This kernel does steps a1-a3: one work unit is 128 queries x one head x
// one half; CTAs are persistent over units:
//   warp 0      TMA producer: 128x64 query slabs and NCx64 subkey slabs
//               (bf16, 128-byte swizzle) into a 3-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=NC<=128, K=16, fp32 accumulate) into four TMEM
//               buffers, shared out among the epilogue sets, so scoring
//               overlaps selection;
//   warps 2..   the epilogue sets of four warps, each set on every other
//               unit (or one set on every unit); one thread per query row
//               (= TMEM lane) reads its row's scores with tcgen05.ld and
//               selects the half's exact top-KL (selection helpers below),
//               then writes the half's list by (score desc, subkey asc) to
//               global memory.
// Forms (template arguments, chosen per call by the host): two sets per CTA
// in clusters of two CTAs that share each subkey slab by multicast
// (kPair); two sets per CTA alone (the retry pass); one set per CTA whose
// stages each hold a query slab and two key chunks' subkey slabs (wide
// half-queries, where the tile bytes an SM receives bound the kernel).
// The k^2 merge and the softmax (a4, a5) run in lookup_merge.cu, one thread
// per (query, head).  A retry launch of this kernel re-selects, without the
// threshold hint, the units listed in a device array.  Scores never leave
// the SM.  Every mbarrier wait is
// bounded; on time-out the kernel records PKM_ERR_TIMEOUT, stops issuing
// work, waits (bounded) for its own copies and MMAs in flight, frees TMEM and
// returns.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "pkm_internal.cuh"
#include "select_net.cuh"
#include "tc_common.cuh"

namespace pkm {
namespace {

using namespace tc;

constexpr int BM = 128;             // query rows per tile (MMA M)
constexpr int BK = 64;              // bf16 elements per k-slab: one 128-byte swizzle row
constexpr int NCMAX = 128;          // subkeys per chunk (MMA N)
constexpr int A_BYTES = BM * BK * 2;     // 16 KiB
constexpr int B_BYTES = NCMAX * BK * 2;  // 16 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TBUFS = 4;                 // 128-column TMEM score buffers
constexpr uint32_t TMEM_COLS = TBUFS * NCMAX;

// ---------------------------------------------------- selection helpers
//
// Per-half selection in the epilogue, one thread per query row.  Issue slots
// and the half-rate ALU pipe (compares, min/max, selects) are the scarce
// resources here, so the exact top-KL is found without a per-candidate
// sorted insertion:
//   1. a per-row threshold hint from the mean and spread of the first 256
//      scores (FMA-pipe arithmetic), aimed at a few times KL of the row's n
//      scores;
//   2. every score above the threshold is appended, with its column, to a
//      per-row log in shared memory: one compare and one predicated 8-byte
//      store per score;
//   3. when a log could overflow it is compacted: value-only sorting
//      networks fold the new entries into V, the sorted values of the log's
//      KL best; entries below the KL-th score x (and ties at x beyond the
//      ones the top-KL keeps, later columns first out) are dropped, and x
//      becomes the new strict threshold.  x is a valid lower bound on the
//      row's final KL-th score (KL logged scores are >= x), so everything
//      that can still be selected is in the log: the result stays exact
//      whatever the hint was;
//   4. at the end of the half the log is compacted to exactly KL entries;
//      each entry's place in the (score desc, column asc) order comes from a
//      binary search of its score in V.
// A row whose hint was above its final KL-th score ends with fewer than KL
// entries; its list is marked, and the retry pass selects its unit again
// without the hint.

constexpr int LOG_CAP = 64;                 // log entries per row and epilogue set
constexpr int SUB = 8;                      // scores appended between two overflow checks
constexpr int LOG_STEP = BM * 8;            // bytes from one slot of a row to the next
constexpr int LOG_BYTES = LOG_CAP * LOG_STEP;

// Per-row log in shared memory: 8-byte entries (score bits, column),
// [slot][row] so a warp's 32 rows touch distinct banks whatever their lengths.
struct RowLog {
  uint2* e;  // [LOG_CAP][BM]
  int row;
  __device__ __forceinline__ uint2& at(int s) const { return e[s * BM + row]; }
  __device__ __forceinline__ uint32_t addr(int s) const { return smem_u32(e + s * BM + row); }
};

// Fold the values of log entries [b0, b0 + NB) (those below len) into V;
// when V holds nothing yet (first fold of a half), the sorted block is V.
template <int KL, int NB>
__device__ __forceinline__ void fold_block(const RowLog& L, int b0, int len, float (&V)[KL],
                                           bool v_empty) {
  float Bv[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const int e = b0 + j < LOG_CAP ? b0 + j : LOG_CAP - 1;  // in bounds, read unconditionally
    const float x = __uint_as_float(L.at(e).x);
    Bv[j] = (b0 + j < len) ? x : -INFINITY;
  }
  sort_desc<NB>(Bv);
  if (v_empty) {
#pragma unroll
    for (int i = 0; i < KL; ++i) V[i] = i < NB ? Bv[i] : -INFINITY;
  } else {
    merge_top<KL, NB>(V, Bv);
  }
}

// Fold the log entries [nsorted, len) into V; then, if the log holds more
// than KL entries, keep only those KL (ties at the KL-th score: earliest
// columns) in column order and raise the threshold to the KL-th score.
// Warp-uniform: every lane runs the networks, lanes without new entries fold
// -inf.
template <int KL>
__device__ __forceinline__ void compact_log(const RowLog& L, int& len, int& nsorted,
                                            float (&V)[KL], float& thr, bool& v_empty) {
#pragma unroll 1
  for (int b0 = nsorted; __any_sync(0xffffffffu, len > b0); b0 += 32) {
    if (__any_sync(0xffffffffu, len > b0 + 16))
      fold_block<KL, 32>(L, b0, len, V, v_empty);
    else
      fold_block<KL, 16>(L, b0, len, V, v_empty);
    v_empty = false;
  }
  nsorted = len;
  if (len <= KL) return;  // at most KL entries: all of them stay
  const float x = V[KL - 1];
  int gt = 0;
#pragma unroll
  for (int i = 0; i < KL; ++i) gt += V[i] > x;
  int budget = KL - gt;  // ties at x that stay (earliest columns)
  const uint2* rp = &L.at(0);
  uint2* wp = &L.at(0);
#pragma unroll 4
  for (int r = 0; r < len; ++r, rp += BM) {
    // slot w <= r was already read, so it can be written whether or not the
    // entry stays; w only advances past kept entries
    const uint2 t = *rp;
    const float v = __uint_as_float(t.x);
    const bool eq = v == x;
    const bool keep = v > x || (eq && budget > 0);
    budget -= (eq && keep);
    *wp = t;
    wp += keep ? BM : 0;
  }
  len = KL;
  nsorted = KL;
  thr = fmaxf(thr, x);
}

// Write the log's entries [0, len) (column order, values sorted in V) to
// slots [KL, 2KL) ordered by (score desc, column asc): an entry's slot is
// the number of larger values, plus the number of earlier entries with the
// same value.  Unused slots get -inf.
template <int KL>
__device__ __forceinline__ void sorted_list(const RowLog& L, int len, const float (&V)[KL],
                                            bool check_ties) {
  bool tie = false;
#pragma unroll
  for (int i = 0; i + 1 < KL; ++i) tie |= (V[i] == V[i + 1]) && (V[i] > -INFINITY);
  tie &= check_ties;
#pragma unroll 2
  for (int e = 0; e < len; ++e) {
    const uint2 t = L.at(e);
    const float x = __uint_as_float(t.x);
    int r = count_greater<KL>(V, x);
    if (tie)
      for (int e2 = 0; e2 < e; ++e2) r += __uint_as_float(L.at(e2).x) == x;
    L.at(KL + r) = t;
  }
#pragma unroll 1
  for (int r = len; r < KL; ++r) L.at(KL + r) = make_uint2(__float_as_uint(-INFINITY), 0u);
}

// ---------------------------------------------------------------- kernel

// Shape of a launch by its number of epilogue warp sets: two sets (each
// with 2 TMEM buffers, 3 tile stages) where the selection work dominates, or
// one set (4 TMEM buffers, 5 tile stages: 160 KB of tiles in flight instead of
// 96 KB) where the tile pipeline does (wide half-queries).
// The one-set form also loads each query slab once for two key chunks (a
// stage holds the query slab and both chunks' subkey slabs, and two MMAs read
// it), so a chunk pair streams 384 KB into the SM instead of 512 KB.
template <int kSets>
struct SelShape {
  static constexpr int kCps = kSets == 1 ? 2 : 1;  // key chunks per stage
  static constexpr int kStageBytes = A_BYTES + kCps * B_BYTES;
  static constexpr int kStages = 3;
  static constexpr int kBufs = TBUFS / kSets;  // TMEM buffers per set
  static constexpr int kThreads = 64 + kSets * 128;
  static constexpr int kTiles = kStages * kStageBytes;
  static constexpr int kSmem = kTiles + kSets * LOG_BYTES + 1024;  // + alignment slack
  static_assert(kSmem <= 227 * 1024, "selection kernel shared memory");
};

// A CTA's units are u_i = blockIdx.x + i * gridDim.x; epilogue set i % kSets
// takes unit u_i.  The producer and the MMA walk the units kSets at a time,
// chunk by chunk, alternating sets, so every set is fed; set s's chunks go to
// its kBufs TMEM buffers in turn.
// kPair: clusters of two CTAs on neighbouring row tiles (2j, 2j+1) of the same
// (head, half), in lockstep, so each subkey slab crosses from L2 once for the
// pair: CTA rank r loads rows [r NC/2, (r+1) NC/2) of it (tmap_c_half) and
// multicasts them to both.  A stage is then free only when both CTAs' MMAs
// have read it: each MMA's release commit arrives on both CTAs' empty
// barriers.  The pair's units are p_i = cluster + i * clusters.
template <int KL, bool kPair, int kSets>
__global__ void __launch_bounds__(SelShape<kSets>::kThreads, 1)
select_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_c,
                 const __grid_constant__ CUtensorMap tmap_c_half,
                 int B, int H, int n, int NC, int nch, int kb_count, float hint_z,
                 float* __restrict__ list_v, unsigned short* __restrict__ list_c,
                 int* __restrict__ status, const int* __restrict__ unit_list,
                 const int* __restrict__ unit_count, int stall, int* __restrict__ clear_words,
                 int clear_count) {
  using Shape = SelShape<kSets>;
  constexpr int STAGES = Shape::kStages, SETS = kSets, BUFS = Shape::kBufs, CPS = Shape::kCps;
  constexpr int SMEM_TILES = Shape::kTiles, STAGE_BYTES = Shape::kStageBytes;
  static_assert(!kPair || CPS == 1, "pairs multicast one subkey slab per stage");
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * STAGES + 2 * TBUFS + 1];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  // the main pass clears the call's retry bookkeeping first: the merge after
  // this kernel counts into it (every CTA helps, also one without units)
  if (clear_words)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < clear_count;
         i += gridDim.x * blockDim.x)
      clear_words[i] = 0;
  // work unit u: tile u / 2 (row tile, head), half u % 2.  The CTA's i-th
  // unit is entry blockIdx.x + i * gridDim.x of all units, or of unit_list
  // when one is given (a retry launch).  A CTA without units returns at once.
  const int row_tiles = (B + BM - 1) / BM;
  // pair mode: the cluster's work item (pair unit) index and count, and this
  // CTA's rank in it; otherwise the CTA's own
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int slot = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int slots = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int units = kPair ? (row_tiles + 1) / 2 * H * 2
                          : (unit_list ? *unit_count : row_tiles * H * 2);
  const int mine = slot < units ? (units - 1 - slot) / slots + 1 : 0;
  if (mine == 0) return;  // (pair mode: both CTAs of the cluster alike)
  auto unit_at = [&](int i) {
    const int e = slot + i * slots;
    if (kPair) {  // pair unit (pair tile, head, half) -> this CTA's row tile of it
      const int pt = (e >> 1) / H, h = (e >> 1) - ((e >> 1) / H) * H;
      return ((((2 * pt + (int)rank) * H) + h) << 1) | (e & 1);
    }
    return unit_list ? unit_list[e] : e;
  };

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
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), kPair ? 2 : 1);  // pair: both CTAs' MMAs release it
    }
    for (int b = 0; b < TBUFS; ++b) {
      mbar_init(bar_tfull(b), 1);
      mbar_init(bar_tempty(b), 4);  // one arrival per warp of the buffer's set
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
  if (kPair) cluster_sync();  // the peer's barriers exist before any multicast reaches them
  const uint32_t tmem = s_tmem_base;
  const Ctl ctl{&s_abort, status};


  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    // (stall: a test of the bounded waits; nothing is loaded, so the MMA
    // warp's first wait runs out, the kernel records PKM_ERR_TIMEOUT and every
    // warp returns; no copy is ever in flight)
    if (lane == 0 && !stall) {
      uint32_t it = 0;
      bool ok = true;
      for (int i0 = 0; ok && i0 < mine; i0 += SETS)
        for (int ch = 0; ok && ch < nch; ch += CPS)
          for (int st = 0; ok && st < SETS && i0 + st < mine; ++st) {
            const int u = unit_at(i0 + st);
            const int tile = u >> 1, half = u & 1;
            const int rt = tile / H, h = tile - rt * H;
            const int nc = CPS == 2 && ch + 1 < nch ? 2 : 1;  // key chunks in these stages
            const uint32_t tx = (uint32_t)(A_BYTES + nc * NC * BK * 2);
            for (int kb = 0; kb < kb_count; ++kb) {
              const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
              if (!wait_phase(bar_empty(s), ph ^ 1u, ctl)) {
                ok = false;
                break;
              }
              mbar_expect_tx(bar_full(s), tx);
              const uint32_t a_dst = tiles_u32 + s * STAGE_BYTES;
              tma_load_4d(a_dst, &tmap_q, kb * BK, half, h, rt * BM, bar_full(s));
              if (kPair)  // this CTA's half of the subkey slab, to both CTAs
                tma_load_3d_mc(a_dst + A_BYTES + rank * (NC / 2) * 128, &tmap_c_half, kb * BK,
                               ch * NC + (int)rank * (NC / 2), h * 2 + half, bar_full(s), 3);
              else
                for (int c = 0; c < nc; ++c)
                  tma_load_3d(a_dst + A_BYTES + c * B_BYTES, &tmap_c, kb * BK, (ch + c) * NC,
                              h * 2 + half, bar_full(s));
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
      uint32_t it = 0, cnt[SETS] = {};
      bool ok = true;
      for (int i0 = 0; ok && i0 < mine; i0 += SETS)
        for (int ch = 0; ok && ch < nch; ch += CPS)
          for (int st = 0; ok && st < SETS && i0 + st < mine; ++st) {
            const int nc = CPS == 2 && ch + 1 < nch ? 2 : 1;  // key chunks in these stages
            uint32_t buf[CPS];
            for (int c = 0; ok && c < nc; ++c) {
              buf[c] = st * BUFS + cnt[st] % BUFS;
              const uint32_t use = cnt[st] / BUFS;
              ++cnt[st];
              if (!wait_phase(bar_tempty(buf[c]), (use & 1u) ^ 1u, ctl)) ok = false;
            }
            if (!ok) break;
            tc_fence_after();
            for (int kb = 0; kb < kb_count; ++kb, ++it) {
              const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
              if (!wait_phase(bar_full(s), ph, ctl)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t a_desc = sw128_desc(tiles_u32 + s * STAGE_BYTES);
              for (int c = 0; c < nc; ++c) {
                const uint32_t d_tmem = tmem + buf[c] * NCMAX;
                const uint64_t b_desc =
                    sw128_desc(tiles_u32 + s * STAGE_BYTES + A_BYTES + c * B_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                  tc_mma(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc, (kb | kk) != 0);
              }
              // frees the stage once these MMAs have read it (pair: in both CTAs,
              // whose halves of the subkey slab it holds)
              if (kPair)
                tc_commit_mc(bar_empty(s), 3);
              else
                tc_commit(bar_empty(s));
            }
            if (!ok) break;
            for (int c = 0; c < nc; ++c) tc_commit(bar_tfull(buf[c]));  // chunks complete in TMEM
          }
      // all issued MMAs complete before TMEM is released
      tc_commit(bar_done);
      wait_phase_drain(bar_done, 0);
    }
  } else {
    // ---------------------------------------------------- epilogue sets
    const int set = (warp - 2) >> 2;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const RowLog L{reinterpret_cast<uint2*>(smem + SMEM_TILES + set * LOG_BYTES), row};
    const uint32_t log0 = L.addr(0);
    // a log at or below this address has room for SUB more entries
    const uint32_t log_room = log0 + (uint32_t)(LOG_CAP - SUB) * LOG_STEP;
    const int need = KL < n ? KL : n;  // valid entries a full list holds
    uint32_t cnt = 0;                  // chunks of this set consumed so far
    bool ok = true;
    for (int i = set; ok && i < mine; i += SETS) {
      const int u = unit_at(i);
      const int tile = u >> 1, half = u & 1;
      const int rt = tile / H, h = tile - rt * H;
      int nsorted = 0;
      bool v_empty = true;    // warp-uniform: nothing folded into V yet
      float thr = -INFINITY;  // a score is logged when it is > thr
      float V[KL];            // sorted values of the log's KL best (entries < nsorted)
#pragma unroll
      for (int i2 = 0; i2 < KL; ++i2) V[i2] = -INFINITY;
      uint32_t va = log0;  // next free slot of this row's log
#pragma unroll 1
      for (int ch = 0; ch < nch; ++ch) {
        // wait for this chunk; at the start of a unit also for the next one
        // (the threshold hint uses the first two chunks' scores), which is
        // then not waited for again
        const int upto = (ch == 0 && nch > 1) ? 2 : 1;
        if (ch != 1) {
          for (int c = 0; c < upto && ok; ++c) {
            const uint32_t cc = cnt + (uint32_t)c;
            ok = __all_sync(0xffffffffu,
                            wait_phase(bar_tfull(set * BUFS + cc % BUFS), (cc / BUFS) & 1u, ctl));
          }
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t base = lane_addr + (set * BUFS + cnt % BUFS) * NCMAX;
        if (ch == 0 && n > LOG_CAP && hint_z > -INFINITY) {
          // threshold hint: mean + z * spread of the first chunks' scores
          float a1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
          for (int c = 0; c < upto; ++c) {
            const uint32_t cb = lane_addr + (set * BUFS + (cnt + c) % BUFS) * NCMAX;
#pragma unroll 1
            for (int gg = 0; gg < NC; gg += 32) {
              float v[32];
              tmem_ld32(cb + gg, v);
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                a1[j & 3] += v[j];
                a2[j & 3] = fmaf(v[j], v[j], a2[j & 3]);
              }
            }
          }
          const float s1 = (a1[0] + a1[1]) + (a1[2] + a1[3]);
          const float s2 = (a2[0] + a2[1]) + (a2[2] + a2[3]);
          // columns >= n score exactly 0 here (zero-filled subkeys)
          const float m = (float)(n < upto * NC ? n : upto * NC);
          const float mu = s1 / m;
          const float sd = sqrtf(fmaxf(s2 / m - mu * mu, 0.0f));
          thr = nextafterf(fmaf(hint_z, sd, mu), -INFINITY);  // v > thr <=> v >= hint
        }
        const int col_end = n - ch * NC;  // columns of this chunk below n (may exceed NC)
#pragma unroll 1
        for (int g = 0; g < NC; g += 16) {
          float v[16];
          tmem_ld16(base + g, v);
          if (g + 16 > col_end) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (g + j >= col_end) v[j] = -INFINITY;
          }
          const uint32_t c0 = (uint32_t)(ch * NC + g);
#pragma unroll
          for (int j = 0; j < 8; ++j) log_push<LOG_STEP>(va, v[j], thr, c0 + j);
          if (__any_sync(0xffffffffu, va > log_room)) {
            int len = (int)((va - log0) / LOG_STEP);
            compact_log<KL>(L, len, nsorted, V, thr, v_empty);
            va = log0 + (uint32_t)len * LOG_STEP;
          }
#pragma unroll
          for (int j = 8; j < 16; ++j) log_push<LOG_STEP>(va, v[j], thr, c0 + j);
          if (__any_sync(0xffffffffu, va > log_room)) {
            int len = (int)((va - log0) / LOG_STEP);
            compact_log<KL>(L, len, nsorted, V, thr, v_empty);
            va = log0 + (uint32_t)len * LOG_STEP;
          }
        }
        // chunk consumed: hand the TMEM buffer back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty(set * BUFS + cnt % BUFS));
        ++cnt;
      }
      if (!ok) break;
      // everything folded and the log cut to KL entries
      int len = (int)((va - log0) / LOG_STEP);
      compact_log<KL>(L, len, nsorted, V, thr, v_empty);
      const int b = rt * BM + row;
      // the half's list by (score desc, subkey asc) into log slots [KL, 2KL),
      // then to global memory; a list with fewer than `need` entries (the
      // threshold hint was above the row's KL-th score) is marked by the
      // subkey 0xffff in its first slot and selected again by the retry pass
      sorted_list<KL>(L, len, V, b < B);
      if (b < B) {
        const size_t off = (((size_t)b * H + h) * 2 + half) * KL;
        float4* gv = reinterpret_cast<float4*>(list_v + off);
        uint4* gc = reinterpret_cast<uint4*>(list_c + off);
#pragma unroll
        for (int i2 = 0; i2 < KL; i2 += 8) {
          uint2 t[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) t[q] = L.at(KL + i2 + q);
          gv[i2 / 4] = make_float4(__uint_as_float(t[0].x), __uint_as_float(t[1].x),
                                   __uint_as_float(t[2].x), __uint_as_float(t[3].x));
          gv[i2 / 4 + 1] = make_float4(__uint_as_float(t[4].x), __uint_as_float(t[5].x),
                                       __uint_as_float(t[6].x), __uint_as_float(t[7].x));
          uint32_t wv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) wv[q] = (t[2 * q].y & 0xffffu) | (t[2 * q + 1].y << 16);
          if (i2 == 0 && len < need) wv[0] = (wv[0] & 0xffff0000u) | 0xffffu;
          gc[i2 / 8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
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
  // pair: neither CTA leaves while the other may still load into its shared
  // memory or arrive on its barriers
  if (kPair) cluster_sync();
}

// ------------------------------------------------------------------ host

// One selection launch.  pair: the main pass over all units, as clusters of
// two CTAs sharing each subkey slab (see select_tc_kernel); as many clusters
// as can be resident at once, so the grid stays persistent.
template <int KL, bool kPair, int kSets>
cudaError_t launch_kl(const CUtensorMap& mq, const CUtensorMap& mc, const CUtensorMap& mch,
                      int B, int H, int n, int NC, int nch, int kbc, float hint_z,
                      float* list_v, unsigned short* list_c, int* status, const int* unit_list,
                      const int* unit_count, int stall, cudaStream_t stream,
                      int* clear_words = nullptr, int clear_count = 0) {
  using Shape = SelShape<kSets>;
  auto kernel = select_tc_kernel<KL, kPair, kSets>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Shape::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(Shape::kThreads);
  cfg.dynamicSmemBytes = Shape::kSmem;
  cfg.stream = stream;
  if (kPair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_clusters = 0;
    if (!max_clusters) {
      cfg.gridDim = dim3(2 * sm_count() / 2);
      cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    }
    const int pair_units = ((B + BM - 1) / BM + 1) / 2 * H * 2;
    cfg.gridDim = dim3(2 * (pair_units < max_clusters ? pair_units : max_clusters));
  } else {
    const int units = (B + BM - 1) / BM * H * 2;  // also the most a retry can list
    cfg.gridDim = dim3(units < sm_count() ? units : sm_count());  // one CTA per SM
  }
  return cudaLaunchKernelEx(&cfg, kernel, mq, mc, mch, B, H, n, NC, nch, kbc, hint_z, list_v,
                            list_c, status, unit_list, unit_count, stall, clear_words,
                            clear_count);
}

// z with P(N(0,1) > z) = p, by bisection on the normal tail (host, once per call).
float normal_upper_quantile(double p) {
  double lo = -10.0, hi = 10.0;
  for (int i = 0; i < 100; ++i) {
    const double mid = 0.5 * (lo + hi);
    if (0.5 * erfc(mid / sqrt(2.0)) > p) lo = mid; else hi = mid;
  }
  return (float)(0.5 * (lo + hi));
}

}  // namespace

float default_hint_z(int n_keys, int k) {
  // Aim the per-row threshold at about 3 KL of the n scores of a half.  The
  // hint comes from one chunk's mean and spread, so it is noisy; for normally
  // distributed scores (n = 256..2048) fewer than KL above it then happened
  // in none of 10^5 simulated rows, and the log compactions raise the
  // threshold to exact bounds as the log fills.
  const int KL = k <= 16 ? 16 : 32;
  const double target = 3.0 * KL;
  double p = target / (double)n_keys;
  if (p > 0.5) p = 0.5;
  return normal_upper_quantile(p);
}

int list_slots(int k) { return k <= 16 ? 16 : 32; }

cudaError_t launch_lookup_tc(const uint16_t* q, const uint16_t* subkeys, int B, int H, int d_q,
                             int n_keys, int k, float hint_z, int64_t* idx, float* w, int* status,
                             const RetryScratch& retry, float* list_v, unsigned short* list_c,
                             cudaStream_t stream, bool stall, int form) {
  if (B == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int hd = d_q / 2;
  const int NC = n_keys >= NCMAX ? NCMAX : (n_keys + 31) / 32 * 32;
  const int nch = (n_keys + NC - 1) / NC;
  const int kbc = (hd + BK - 1) / BK;

  CUtensorMap mq, mc, mch, m2;
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
    // the same view in half-chunk boxes (NC/2 subkeys): each CTA of a pair
    // loads one half and multicasts it
    const cuuint32_t hbox[3] = {BK, (cuuint32_t)NC / 2, 1};
    if (enc(&mch, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(subkeys), dims,
            strides, hbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    // the two-SM form: each CTA loads 128 subkeys (half of a 256-key chunk)
    const cuuint32_t box2[3] = {BK, 128, 1};
    if (enc(&m2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(subkeys), dims,
            strides, box2, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the main pass as CTA pairs sharing each subkey slab when there are at
  // least two row tiles and the half-query is at most 512 wide (8 k-slabs);
  // the retry pass (listed units) one CTA per unit.  Measured on GB300
  // (lookup call): page 0.318 -> 0.308 ms and the skewed workload 2.03 ->
  // 1.77 ms with pairs, where the selection work dominates; the large
  // workload (16 k-slabs, pipeline-latency-bound with three stages) 1.25 ->
  // 1.35 ms, since each stage of a pair waits for the slower of its two CTAs
  const bool pair_shape = (B + BM - 1) / BM >= 2 && kbc <= 8;
  // wide half-queries (more than 8 k-slabs per chunk) are bound by the tile
  // pipeline, not by the selection: their main pass runs one epilogue set per
  // CTA with 5 tile stages in flight
  const bool deep = kbc > 8;
  // the two-SM form (MMAs of 256 query rows over a CTA pair, each CTA
  // receiving half of every subkey slab) for the main pass of any batch of
  // more than one row tile (a lone 128-row tile runs on one SM)
  const bool two_sm = form >= 2 || (form == 0 && B > BM);
  // the one-SM pair form multicasts subkey slabs: only with this device's
  // own memory
  const void* const operands[2] = {q, subkeys};
  const bool pair = !two_sm && pair_shape && tc::buffers_on_this_device(operands, 2);
  // the two-SM kernel's epilogue form: one set with deeper tile stages for
  // the pipeline-bound wide half-queries (measured on GB300, large workload's
  // lookup call: 1.003 -> 0.885 ms), two sets otherwise (page 0.287 against
  // 0.306 ms with one set, skewed 1.678 against 1.938)
  const int epi = form == 3 || (form == 0 && deep) ? 1 : 2;
  // the main pass also clears the retry bookkeeping (counts and the per-unit
  // flags, one buffer) before anything else, in place of a memset
  const int clear_count = 2 + (int)retry_units(B, H);
  auto select = [&](float z, const int* list, const int* count, int st) {
    int* clear = list ? nullptr : retry.counts;
    if (two_sm && !list)
      return launch_select_2sm(mq, m2, B, H, d_q, n_keys, k, z, list_v, list_c, status, st != 0,
                               stream, epi, clear, clear_count);
#define PKM_SELECT(KLv, PAIRv, SETSv)                                                          \
  launch_kl<KLv, PAIRv, SETSv>(mq, mc, mch, B, H, n_keys, NC, nch, kbc, z, list_v, list_c, \
                               status, list, count, st, stream, clear, clear_count)
    if (pair && !list) return k <= 16 ? PKM_SELECT(16, true, 2) : PKM_SELECT(32, true, 2);
    if (deep && !list) return k <= 16 ? PKM_SELECT(16, false, 1) : PKM_SELECT(32, false, 1);
    return k <= 16 ? PKM_SELECT(16, false, 2) : PKM_SELECT(32, false, 2);
#undef PKM_SELECT
  };
  cudaError_t e = select(hint_z, nullptr, nullptr, stall ? 1 : 0);
  // a4, a5: the k^2 merge and softmax, one thread per (query, head); lists
  // the units whose threshold hint was above a row's KL-th score
  if (e == cudaSuccess)
    e = launch_merge(list_v, list_c, B, H, n_keys, k, idx, w, retry, false, stream);
  // retry: those units again without the hint (exact), then their pairs;
  // both launches return at once when nothing is listed
  if (e == cudaSuccess) e = select(-INFINITY, retry.unit_list, retry.counts + 1, 0);
  if (e == cudaSuccess)
    e = launch_merge(list_v, list_c, B, H, n_keys, k, idx, w, retry, true, stream);
  return e;
}

}  // namespace pkm
