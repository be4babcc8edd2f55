// Steps a4-a5: the k^2 merge of the two per-half lists and the softmax.
//
// Product-Key Memory, "Factorising the key space": the global top-k lies
// inside top_k(half 1) x top_k(half 2); code listing: k^2 sums
// s1[i] + s2[j] with flat index i1 * n_keys + i2, their top-k, and a softmax
// over the winners.  One thread owns one (query, head) pair, so many warps
// per SM hide the latency of the per-pair work.
//
// The lists come from the selection kernel, each ordered by (score desc,
// subkey asc).  Only pairs (i, j) with (i + 1)(j + 1) <= KL can reach the top
// KL (every (i', j') with i' <= i, j' <= j scores at least as much).  Their
// sums reach the sorted KL best sums V through value-only bitonic merges of
// the grid's sorted runs (its first rows and columns) and one small fold;
// each surviving pair's output slot is the number of larger sums (equal sums
// in flat index order) and its softmax weight follows from V.  When more
// than KL pairs reach the KL-th sum x (a tie at the cut), the pairs above x
// are placed that way and those at x fill the places left in flat index
// order.  A list marked failed (subkey 0xffff in its first slot: the
// selection threshold hint was above the row's KL-th score) lists its work
// unit for the retry pass, which selects that unit again without the hint
// and then merges the unit's pairs in this kernel's retry mode.
#include <math.h>
#include <stdint.h>

#include "pkm_internal.cuh"
#include "select_net.cuh"

namespace pkm {
namespace {

constexpr int kThreads = 64;    // pairs (threads) per CTA
constexpr int kTileRows = 128;  // queries per selection row tile (a retry unit's rows)
constexpr int kSplit = kTileRows / kThreads;  // CTAs per retry unit

int tc_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int KL>
struct MergeLayout {
  static constexpr MergePairs<KL> P{};
  // the pairs outside the sorted runs (i, j >= 3), staged and folded in one
  // block of kRestBlock (a power of two)
  static constexpr int rest() {
    int c = 0;
    for (int q = 0; q < P.kCount; ++q) c += P.i[q] >= 3 && P.j[q] >= 3;
    return c;
  }
  static constexpr int kRest = rest();
  static constexpr int kRestBlock = kRest <= 2 ? 2 : kRest <= 4 ? 4 : kRest <= 8 ? 8 : 16;
  static_assert(kRest >= 1 && kRest <= 16, "merge: pairs outside the sorted runs");
  // region A, 4-byte slots in [slot][thread] order: the scores of the pairs
  // outside the runs staged for folding (slots [0, kRest)), later the
  // survivors' scores (slots [0, kSurvCap)) and pair codes (slots
  // [kSurvCap, 2 kSurvCap)).  Every use keeps a thread inside its own
  // column, so warps in different phases never touch each other's slots.
  // First, in the first pass, it holds the CTA's lists as loaded, [pair][2KL
  // + 4] floats (rows 16-byte aligned; the +4 spreads rows over banks).
  static constexpr int kSlotsA = kRest > 2 * KL + 4 ? kRest : 2 * KL + 4;
  // survivors held (scores and codes): KL and two more, so a tie at the KL-th
  // sum that brings one or two more pairs is resolved from the store
  static constexpr int kSurvCap = KL + 2;
  static_assert(2 * kSurvCap <= kSlotsA, "merge: survivor store");
  static constexpr int kRegionA = kSlotsA * 4 * kThreads;
  // the lists' subkeys, [pair][2KL + 2] 16-bit (odd word stride: a thread's
  // own row and the cooperative fill are both free of bank conflicts)
  static constexpr int kCodeRow = 2 * KL + 2;
  static constexpr int kRegionC = kRegionA + (kCodeRow * 2 * kThreads + 15) / 16 * 16;
  // region C, [place][thread]: the survivors' pair codes (16-bit) by output
  // place
  static constexpr int kBytes = kRegionC + (KL * 2 * kThreads + 15) / 16 * 16;
};

// One CTA's pairs: first pass, pair = cta * 64 + thread; retry pass, listed
// unit cta / 2 and thread t its row tile's query 64 (cta % 2) + t.
template <int KL>
__device__ __forceinline__ void merge_cta(const float* __restrict__ list_v,
                                          const unsigned short* __restrict__ list_c, int B, int H,
                                          int n, int k, int64_t* __restrict__ idx,
                                          float* __restrict__ w, const RetryScratch& retry,
                                          bool retry_pass, int cta) {
  using Lay = MergeLayout<KL>;
  constexpr MergePairs<KL> P{};
  extern __shared__ __align__(16) unsigned char smem[];
  float* stg = reinterpret_cast<float*>(smem);                                  // [kRest][T]
  constexpr int kCap = Lay::kSurvCap;
  float* sv = reinterpret_cast<float*>(smem);                                   // [kCap][T]
  uint32_t* sp = reinterpret_cast<uint32_t*>(sv + kCap * kThreads);             // [kCap][T]
  unsigned short* sc = reinterpret_cast<unsigned short*>(smem + Lay::kRegionA); // [T][2KL+2]
  unsigned short* so = reinterpret_cast<unsigned short*>(smem + Lay::kRegionC); // [KL][T]
  const int t = threadIdx.x;
  int pair;
  // every lane stays until the last warp vote (below); lanes without a pair
  // of their own work on zeros until then and store nothing
  bool valid;
  if (retry_pass) {
    const int tile = retry.unit_list[cta / kSplit] >> 1;
    const int rt = tile / H, h = tile - (tile / H) * H;
    const int b = rt * kTileRows + (cta % kSplit) * kThreads + t;
    valid = b < B;
    pair = valid ? b * H + h : 0;
  } else {
    pair = cta * kThreads + t;
    valid = pair < B * H;
  }

  const float* v1 = list_v + (size_t)(valid ? pair : 0) * 2 * KL;
  unsigned short* my_sc = sc + t * Lay::kCodeRow;
  float s1v[KL], s2v[KL];
  if (!retry_pass) {
    // the CTA's pairs are consecutive, so are their lists: coalesced copies
    // by the whole CTA into shared memory, then each thread takes its own row
    // (a thread's own lists are 256 + 128 scattered bytes apart from its
    // neighbours')
    constexpr int kRowV = 2 * KL + 4;
    const int pair0 = cta * kThreads;
    const int np = min(kThreads, B * H - pair0);
    // asynchronous copies (no registers held), all in flight before the wait
    const uint32_t st0 = static_cast<uint32_t>(__cvta_generic_to_shared(stg));
    const uint32_t sc0 = static_cast<uint32_t>(__cvta_generic_to_shared(sc));
    const float4* gv = reinterpret_cast<const float4*>(list_v + (size_t)pair0 * 2 * KL);
#pragma unroll 4
    for (int q = t; q < np * (KL / 2); q += kThreads) {
      const int p = q / (KL / 2), s4 = q - p * (KL / 2);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       st0 + (uint32_t)(p * kRowV + 4 * s4) * 4u),
                   "l"(gv + q)
                   : "memory");
    }
    const uint32_t* gc = reinterpret_cast<const uint32_t*>(list_c + (size_t)pair0 * 2 * KL);
#pragma unroll 4
    for (int q = t; q < np * KL; q += kThreads) {  // KL words (2 KL codes) per pair
      const int p = q / KL, m = q - p * KL;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                       sc0 + (uint32_t)(p * (Lay::kCodeRow / 2) + m) * 4u),
                   "l"(gc + q)
                   : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    const float4* r4 = reinterpret_cast<const float4*>(stg + t * kRowV);
#pragma unroll
    for (int i = 0; i < KL / 4; ++i) {
      const float4 a = r4[i], b = r4[KL / 4 + i];
      s1v[4 * i] = a.x; s1v[4 * i + 1] = a.y; s1v[4 * i + 2] = a.z; s1v[4 * i + 3] = a.w;
      s2v[4 * i] = b.x; s2v[4 * i + 1] = b.y; s2v[4 * i + 2] = b.z; s2v[4 * i + 3] = b.w;
    }
    __syncthreads();  // region A is reused below
  } else {
    const float4* g = reinterpret_cast<const float4*>(v1);
#pragma unroll
    for (int i = 0; i < KL / 4; ++i) {
      const float4 a = g[i], b = g[KL / 4 + i];
      s1v[4 * i] = a.x; s1v[4 * i + 1] = a.y; s1v[4 * i + 2] = a.z; s1v[4 * i + 3] = a.w;
      s2v[4 * i] = b.x; s2v[4 * i + 1] = b.y; s2v[4 * i + 2] = b.z; s2v[4 * i + 3] = b.w;
    }
    const uint4* gc = reinterpret_cast<const uint4*>(list_c + (size_t)(valid ? pair : 0) * 2 * KL);
    uint32_t* my32 = reinterpret_cast<uint32_t*>(my_sc);
#pragma unroll
    for (int i = 0; i < KL / 4; ++i) {
      const uint4 u = gc[i];
      my32[4 * i] = u.x;
      my32[4 * i + 1] = u.y;
      my32[4 * i + 2] = u.z;
      my32[4 * i + 3] = u.w;
    }
  }
  const bool bad1 = my_sc[0] == 0xffffu, bad2 = my_sc[KL] == 0xffffu;
  if (valid && (bad1 || bad2) && !retry_pass) {  // without the hint every list is complete
    atomicAdd(&retry.counts[0], 1);
    const int b = pair / H, h = pair - (pair / H) * H;
    const int unit0 = ((b / kTileRows) * H + h) << 1;
    for (int hf = 0; hf < 2; ++hf)
      if ((hf ? bad2 : bad1) && atomicExch(&retry.unit_flag[unit0 | hf], 1) == 0)
        retry.unit_list[atomicAdd(&retry.counts[1], 1)] = unit0 | hf;
    valid = false;
  }
  if (!valid) {
#pragma unroll
    for (int i = 0; i < KL; ++i) s1v[i] = s2v[i] = 0.0f;
  }
  auto col1 = [&](int i) { return (int)my_sc[i]; };
  auto col2 = [&](int j) { return (int)my_sc[KL + j]; };

  // V: the sorted KL best sums.  Rows and columns of the candidate grid are
  // sorted runs: row 0 starts V, and row 1, column 0, column 1 and the rest
  // of row 2 and of column 2 are merged in, one bitonic merge each.  The
  // pairs left (i, j >= 3: twelve at KL = 32) are staged when above V's
  // KL-th sum and folded in one block.
  float V[KL];
#pragma unroll
  for (int j = 0; j < KL; ++j) V[j] = s1v[0] + s2v[j];
  {
    float R[KL / 2];  // row 1
#pragma unroll
    for (int j = 0; j < KL / 2; ++j) R[j] = s1v[1] + s2v[j];
    merge_top<KL, KL / 2>(V, R);
  }
  {
    float R[KL - 2];  // column 0, rows 2 ..
#pragma unroll
    for (int u = 0; u < KL - 2; ++u) R[u] = s1v[2 + u] + s2v[0];
    merge_top<KL, KL - 2>(V, R);
  }
  {
    float R[KL / 2 - 2];  // column 1, rows 2 ..
#pragma unroll
    for (int u = 0; u < KL / 2 - 2; ++u) R[u] = s1v[2 + u] + s2v[1];
    merge_top<KL, KL / 2 - 2>(V, R);
  }
  {
    float R[KL / 3 - 2];  // row 2, columns 2 ..
#pragma unroll
    for (int u = 0; u < KL / 3 - 2; ++u) R[u] = s1v[2] + s2v[2 + u];
    merge_top<KL, KL / 3 - 2>(V, R);
  }
  {
    float R[KL / 3 - 3];  // column 2, rows 3 ..
#pragma unroll
    for (int u = 0; u < KL / 3 - 3; ++u) R[u] = s1v[3 + u] + s2v[2];
    merge_top<KL, KL / 3 - 3>(V, R);
  }
  {
    const float x1 = V[KL - 1];
    const uint32_t a0 = static_cast<uint32_t>(__cvta_generic_to_shared(stg + t));
    uint32_t a = a0;
#pragma unroll
    for (int c = 0; c < P.kCount; ++c)
      if (P.i[c] >= 3 && P.j[c] >= 3) stage_push<kThreads * 4>(a, s1v[P.i[c]] + s2v[P.j[c]], x1);
    const int m = (int)((a - a0) / (kThreads * 4));
    if (__any_sync(0xffffffffu, m > 0)) {
      constexpr int NR = Lay::kRestBlock;
      float Bv[NR];
#pragma unroll
      for (int u = 0; u < NR; ++u) {
        const float v = stg[(u < Lay::kRest ? u : 0) * kThreads + t];
        Bv[u] = u < m ? v : -INFINITY;
      }
      sort_desc<NR>(Bv);
      merge_top<KL, NR>(V, Bv);
    }
  }
  const float x = V[KL - 1];
  // bit i: V[i] == V[i + 1] (a sum that occurs more than once in the best KL)
  uint32_t dup = 0;
#pragma unroll
  for (int i = 0; i + 1 < KL; ++i) dup |= (V[i] == V[i + 1] ? 1u : 0u) << i;
  // survivors: pairs scoring >= x, the first kCap of them held; more than KL
  // of them means a tie at x (region A is free again: the staged scores were
  // all folded)
  const uint32_t va0 = static_cast<uint32_t>(__cvta_generic_to_shared(sv + t));
  const uint32_t va_end = va0 + kCap * (kThreads * 4);
  uint32_t va = va0, nsurv = 0;
  const float below_x = nextafterf(x, -INFINITY);  // >= x  <=>  > below_x
#pragma unroll
  for (int c = 0; c < P.kCount; ++c) {
    const float s = s1v[P.i[c]] + s2v[P.j[c]];
    surv_push<kThreads * 4, kCap * kThreads * 4>(va, nsurv, va_end, s, below_x,
                                                 (uint32_t)(P.i[c] * 32 + P.j[c]));
  }
  // the warp's vote for the equal-sum pass below, taken while every lane is
  // still here (lanes without a pair leave at the next line and wait at the
  // caller's barrier)
  const bool any_equal = __any_sync(0xffffffffu, valid && (dup != 0u || nsurv > (uint32_t)KL));
  if (!valid) return;
  int64_t* ip = idx + (size_t)pair * k;
  float* wp = w + (size_t)pair * k;
  auto flat_of = [&](uint32_t pc) { return (int64_t)col1((int)(pc >> 5)) * n + col2((int)(pc & 31)); };
  uint32_t held = nsurv < (uint32_t)kCap ? nsurv : (uint32_t)kCap;
  // a tie at x (more than KL pairs reach it): the pairs at x are ranked by
  // flat index after the larger sums, and those ranked KL or later dropped
  bool cut = nsurv > (uint32_t)KL;
  if (nsurv > (uint32_t)kCap) {
    // more pairs at x than the store holds: hold the pairs above x only
    // (fewer than KL) and fill the places left after them below.  Rare:
    // plain loops over the lists in global memory keep this code small.
    uint32_t va2 = va0;
    held = 0;
    cut = false;
#pragma unroll 1
    for (int i = 0; i < KL; ++i) {
      const float xi = v1[i];
#pragma unroll 1
      for (int j = 0; (i + 1) * (j + 1) <= KL; ++j)
        surv_push<kThreads * 4, kCap * kThreads * 4>(va2, held, va_end, xi + v1[KL + j], x,
                                                     (uint32_t)(i * 32 + j));
    }
  }
  // Each held survivor's output place is the number of larger sums (its
  // pair code goes to that place's slot of this thread's column); branch
  // free, several survivors in flight.
#pragma unroll 4
  for (int e = 0; e < kCap; ++e) {
    const float s = sv[e * kThreads + t];
    const uint32_t pc = sp[e * kThreads + t];
    const int place = count_greater<KL>(V, s);
    if (e < (int)held && place < KL) so[place * kThreads + t] = (unsigned short)pc;
    // kept beside the code (bits 16 and up) for the equal-sum pass
    if (any_equal && e < (int)held) sp[e * kThreads + t] = pc | ((uint32_t)place << 16);
  }
  // A sum that occurs more than once (dup bit set at its place, or a sum at
  // x cut by the tie) moves up by the number of equal held survivors with a
  // lower flat index (the lowest keeps its place).  Rare: warps enter only
  // when one of their rows has equal sums.
  if (any_equal) {
#pragma unroll 1
    for (int e = 0; e < (int)held; ++e) {
      const float s = sv[e * kThreads + t];
      const uint32_t pc = sp[e * kThreads + t] & 0xffffu;
      int place = (int)(sp[e * kThreads + t] >> 16);
      if (((dup >> place) & 1u) || (cut && s == x)) {
        const int64_t f = flat_of(pc);
#pragma unroll 1
        for (int e2 = 0; e2 < (int)held; ++e2)
          place += sv[e2 * kThreads + t] == s && flat_of(sp[e2 * kThreads + t] & 0xffffu) < f;
        if (place < KL) so[place * kThreads + t] = (unsigned short)pc;
      }
    }
  }
  if (nsurv > (uint32_t)kCap && (int)held < k) {
    // the places left (sum x each) in flat index order: per place, a scan for
    // the lowest flat index above the previous place's among the pairs at x
    int64_t last = -1;
#pragma unroll 1
    for (int r = (int)held; r < k; ++r) {
      int64_t best = INT64_MAX;
      uint32_t bc = 0;
#pragma unroll 1
      for (int i = 0; i < KL; ++i) {
        const float xi = v1[i];
#pragma unroll 1
        for (int j = 0; (i + 1) * (j + 1) <= KL; ++j) {
          if (xi + v1[KL + j] == x) {
            const uint32_t pc = (uint32_t)(i * 32 + j);
            const int64_t f = flat_of(pc);
            if (f > last && f < best) {
              best = f;
              bc = pc;
            }
          }
        }
      }
      so[r * kThreads + t] = (unsigned short)bc;
      last = best;
    }
  }
  // then the places in order: flat index and softmax weight (the place's sum
  // is V[r]; the softmax over the first k, V[0] the largest), written as
  // whole vectors when the row holds KL
  float ex[KL];
  float z4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int r = 0; r < KL; ++r) {
    ex[r] = r < k ? expf(V[r] - V[0]) : 0.0f;
    z4[r & 3] += ex[r];
  }
  const float inv_z = 1.0f / ((z4[0] + z4[1]) + (z4[2] + z4[3]));
  auto flat = [&](int r) { return flat_of(so[r * kThreads + t]); };
  if (k == KL) {
#pragma unroll
    for (int r = 0; r < KL; r += 4) {
      reinterpret_cast<longlong2*>(ip + r)[0] = make_longlong2(flat(r), flat(r + 1));
      reinterpret_cast<longlong2*>(ip + r)[1] = make_longlong2(flat(r + 2), flat(r + 3));
      reinterpret_cast<float4*>(wp + r)[0] = make_float4(ex[r] * inv_z, ex[r + 1] * inv_z,
                                                         ex[r + 2] * inv_z, ex[r + 3] * inv_z);
    }
  } else {
#pragma unroll
    for (int r = 0; r < KL; ++r) {
      if (r < k) {
        ip[r] = flat(r);
        wp[r] = ex[r] * inv_z;
      }
    }
  }
}

// First pass: CTA c merges pairs [64c, 64c + 64).  Retry pass: a persistent
// grid walks the listed units, two CTA-sized halves each (none listed: every
// CTA returns at once).
template <int KL>
// 128 registers: seven 64-thread CTAs per SM (14 warps; the register file is
// split over the SM's four schedulers, 16,384 registers each, and a scheduler
// holding four warps leaves 128 to each), so the page-size batch's 1024 CTAs
// run in one wave; shared memory allows seven as well.  The cap spills a few
// hundred bytes per thread; 144 registers would fit only three warps per
// scheduler (two waves, slower).
__global__ void __maxnreg__(128)
merge_kernel(const float* __restrict__ list_v, const unsigned short* __restrict__ list_c, int B,
             int H, int n, int k, int64_t* __restrict__ idx, float* __restrict__ w,
             RetryScratch retry, bool retry_pass) {
  // one call site: a single inlined copy of the per-pair code serves both
  // passes (the code is long and runs once per warp, so its size is fetch
  // time).  Lanes without a pair return from merge_cta early and wait at the
  // barrier below, so merge_cta takes no warp vote after they leave.
  const int end = retry_pass ? retry.counts[1] * kSplit : (int)blockIdx.x + 1;
  for (int u = (int)blockIdx.x; u < end; u += (int)gridDim.x) {
    merge_cta<KL>(list_v, list_c, B, H, n, k, idx, w, retry, retry_pass, u);
    __syncthreads();  // the CTA's shared-memory columns are reused by its next unit
  }
}

template <int KL>
cudaError_t launch_merge_kl(const float* list_v, const unsigned short* list_c, int B, int H, int n,
                            int k, int64_t* idx, float* w, const RetryScratch& retry,
                            bool retry_pass, cudaStream_t stream) {
  const size_t smem = MergeLayout<KL>::kBytes;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(merge_kernel<KL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // seven CTAs per SM need the whole shared-memory carveout
    e = cudaFuncSetAttribute(merge_kernel<KL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t units = retry_units(B, H);
  const int64_t grid = retry_pass ? (units * kSplit < 7 * tc_sms() ? units * kSplit : 7 * tc_sms())
                                  : ((int64_t)B * H + kThreads - 1) / kThreads;
  merge_kernel<KL><<<(unsigned)grid, kThreads, smem, stream>>>(list_v, list_c, B, H, n, k, idx, w,
                                                                retry, retry_pass);
  return cudaGetLastError();
}

}  // namespace

int64_t retry_units(int64_t B, int64_t H) { return (B + kTileRows - 1) / kTileRows * H * 2; }

cudaError_t launch_merge(const float* list_v, const unsigned short* list_c, int B, int H,
                         int n_keys, int k, int64_t* idx, float* w, const RetryScratch& retry,
                         bool retry_pass, cudaStream_t stream) {
  if ((int64_t)B * H == 0) return cudaSuccess;
  if (k <= 16)
    return launch_merge_kl<16>(list_v, list_c, B, H, n_keys, k, idx, w, retry, retry_pass,
                               stream);
  return launch_merge_kl<32>(list_v, list_c, B, H, n_keys, k, idx, w, retry, retry_pass, stream);
}

}  // namespace pkm
