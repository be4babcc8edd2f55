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
// sums go through value-only sorting networks to the sorted KL best sums V;
// when those are all distinct and no left-out pair ties the KL-th, each
// surviving pair's output slot is the number of larger sums and its softmax
// weight follows from V.  Exact ties take a frontier walk that orders equal
// sums by flat index.  A list marked failed (subkey 0xffff in its first
// slot: the selection threshold hint was above the row's KL-th score) lists
// its work unit for the retry pass, which selects that unit again without
// the hint and then merges the unit's pairs in this kernel's retry mode.
#include <math.h>
#include <stdint.h>

#include "pkm_internal.cuh"
#include "select_net.cuh"

namespace pkm {
namespace {

constexpr int kThreads = 128;

int tc_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int KL>
struct MergeLayout {
  static constexpr MergePairs<KL> P{};
  static constexpr int kRow01 = KL + KL / 2;         // candidates of rows 0 and 1 (table is row-major)
  static constexpr int kRest = P.kCount - kRow01;    // candidates of rows >= 2
  // region A, 4-byte slots in [slot][thread] order: the rows >= 2 scores
  // staged for folding (slots [0, kRest)), later the survivors' scores
  // (slots [0, KL)) and pair codes (slots [KL, 2KL)).  Every use keeps a
  // thread inside its own column, so warps in different phases never touch
  // each other's slots.
  // First, in the first pass, it holds the CTA's lists as loaded, [pair][2KL
  // + 4] floats (rows 16-byte aligned; the +4 spreads rows over banks).
  static constexpr int kSlotsA = kRest > 2 * KL + 4 ? kRest : 2 * KL + 4;
  static constexpr int kRegionA = kSlotsA * 4 * kThreads;
  // the lists' subkeys, [pair][2KL + 2] 16-bit (odd word stride: a thread's
  // own row and the cooperative fill are both free of bank conflicts)
  static constexpr int kCodeRow = 2 * KL + 2;
  static constexpr int kRegionC = kRegionA + (kCodeRow * 2 * kThreads + 15) / 16 * 16;
  // region C, [place][thread]: the survivors' pair codes by output place
  static constexpr int kBytes = kRegionC + KL * 4 * kThreads;
};

// One CTA's pairs: first pass, pair = cta * 128 + thread; retry pass, listed
// unit `cta` and thread t its row tile's query t.
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
  float* sv = reinterpret_cast<float*>(smem);                                   // [KL][T]
  uint32_t* sp = reinterpret_cast<uint32_t*>(sv + KL * kThreads);               // [KL][T]
  unsigned short* sc = reinterpret_cast<unsigned short*>(smem + Lay::kRegionA); // [T][2KL+2]
  uint32_t* so = reinterpret_cast<uint32_t*>(smem + Lay::kRegionC);             // [KL][T]
  const int t = threadIdx.x;
  int pair;
  // every lane stays to the end (warp votes below); lanes without a pair of
  // their own work on zeros and store nothing
  bool valid;
  if (retry_pass) {
    const int tile = retry.unit_list[cta] >> 1;
    const int rt = tile / H, h = tile - (tile / H) * H;
    const int b = rt * kThreads + t;  // row tiles hold 128 queries, one per thread
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
    // the CTA's pairs are consecutive, so are their lists: coalesced 16-byte
    // loads by the whole CTA into shared memory, then each thread takes its
    // own row (a thread's own lists are 256 + 128 scattered bytes apart from
    // its neighbours')
    constexpr int kRowV = 2 * KL + 4;
    const int pair0 = cta * kThreads;
    const int np = min(kThreads, B * H - pair0);
    const float4* gv = reinterpret_cast<const float4*>(list_v + (size_t)pair0 * 2 * KL);
    for (int q = t; q < np * (KL / 2); q += kThreads) {
      const int p = q / (KL / 2), s4 = q - p * (KL / 2);
      *reinterpret_cast<float4*>(stg + p * kRowV + 4 * s4) = gv[q];
    }
    const uint4* gc = reinterpret_cast<const uint4*>(list_c + (size_t)pair0 * 2 * KL);
    uint32_t* sc32 = reinterpret_cast<uint32_t*>(sc);
    for (int q = t; q < np * (KL / 4); q += kThreads) {
      const int p = q / (KL / 4), m = q - p * (KL / 4);
      const uint4 u = gc[q];
      uint32_t* d = sc32 + p * (Lay::kCodeRow / 2) + 4 * m;
      d[0] = u.x;
      d[1] = u.y;
      d[2] = u.z;
      d[3] = u.w;
    }
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
    const int unit0 = ((b / kThreads) * H + h) << 1;
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

  // V: the sorted KL best sums.  Row 0 of the candidate grid is already in
  // descending order; row 1 is too, and one bitonic merge takes it in.
  float V[KL];
#pragma unroll
  for (int j = 0; j < KL; ++j) V[j] = s1v[0] + s2v[j];
  {
    float R[KL / 2];
#pragma unroll
    for (int j = 0; j < KL / 2; ++j) R[j] = s1v[1] + s2v[j];
    merge_top<KL, KL / 2>(V, R);
  }
  // rows >= 2: only sums above V's KL-th can change V; they are staged in
  // shared memory and folded in blocks
  {
    const float x1 = V[KL - 1];
    const uint32_t a0 = static_cast<uint32_t>(__cvta_generic_to_shared(stg + t));
    uint32_t a = a0;
#pragma unroll
    for (int c = Lay::kRow01; c < P.kCount; ++c)
      stage_push<kThreads * 4>(a, s1v[P.i[c]] + s2v[P.j[c]], x1);
    const int m = (int)((a - a0) / (kThreads * 4));
#pragma unroll 1
    for (int b0 = 0; __any_sync(0xffffffffu, m > b0); b0 += 32) {
      if (__any_sync(0xffffffffu, m > b0 + 16)) {
        float Bv[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int e = b0 + u < Lay::kRest ? b0 + u : Lay::kRest - 1;
          const float x = stg[e * kThreads + t];
          Bv[u] = b0 + u < m ? x : -INFINITY;
        }
        sort_desc<32>(Bv);
        merge_top<KL, 32>(V, Bv);
      } else {
        float Bv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int e = b0 + u < Lay::kRest ? b0 + u : Lay::kRest - 1;
          const float x = stg[e * kThreads + t];
          Bv[u] = b0 + u < m ? x : -INFINITY;
        }
        sort_desc<16>(Bv);
        merge_top<KL, 16>(V, Bv);
      }
    }
  }
  const float x = V[KL - 1];
  bool tie = false;
#pragma unroll
  for (int i = 0; i + 1 < KL; ++i) tie |= V[i] == V[i + 1];
  // survivors: pairs scoring >= x; more than KL of them means a tie at x
  // (region A is free again: the staged scores were all folded)
  const uint32_t va0 = static_cast<uint32_t>(__cvta_generic_to_shared(sv + t));
  const uint32_t va_end = va0 + KL * (kThreads * 4);
  uint32_t va = va0, nsurv = 0;
  const float below_x = nextafterf(x, -INFINITY);  // >= x  <=>  > below_x
#pragma unroll
  for (int c = 0; c < P.kCount; ++c) {
    const float s = s1v[P.i[c]] + s2v[P.j[c]];
    surv_push<kThreads * 4, KL * kThreads * 4>(va, nsurv, va_end, s, below_x,
                                               (uint32_t)(P.i[c] * 32 + P.j[c]));
  }
  if (!valid) return;
  float z = 0.0f;
#pragma unroll
  for (int r = 0; r < KL; ++r)
    if (r < k) z += expf(V[r] - V[0]);
  int64_t* ip = idx + (size_t)pair * k;
  float* wp = w + (size_t)pair * k;
  if (!tie && nsurv == (uint32_t)KL) {
    // each survivor's output place is the number of larger sums; its pair
    // code goes to that place's slot of this thread's column
#pragma unroll 2
    for (int e = 0; e < KL; ++e) {
      const float s = sv[e * kThreads + t];
      so[count_greater<KL>(V, s) * kThreads + t] = sp[e * kThreads + t];
    }
    // then the places in order: flat index and softmax weight (the place's
    // sum is V[r]), written as whole vectors when the row holds KL
    const float inv_z = 1.0f / z;
    auto flat = [&](int r) {
      const int pc = (int)so[r * kThreads + t];
      return (int64_t)(col1(pc >> 5) * n + col2(pc & 31));
    };
    if (k == KL) {
#pragma unroll
      for (int r = 0; r < KL; r += 4) {
        reinterpret_cast<longlong2*>(ip + r)[0] = make_longlong2(flat(r), flat(r + 1));
        reinterpret_cast<longlong2*>(ip + r)[1] = make_longlong2(flat(r + 2), flat(r + 3));
        reinterpret_cast<float4*>(wp + r)[0] =
            make_float4(expf(V[r] - V[0]) * inv_z, expf(V[r + 1] - V[0]) * inv_z,
                        expf(V[r + 2] - V[0]) * inv_z, expf(V[r + 3] - V[0]) * inv_z);
      }
    } else {
#pragma unroll
      for (int r = 0; r < KL; ++r) {
        if (r < k) {
          ip[r] = flat(r);
          wp[r] = expf(V[r] - V[0]) * inv_z;
        }
      }
    }
    return;
  }
  // frontier walk (exact ties): row i of the candidate grid is sorted, the
  // next winner is the best of the rows' heads, (score desc, flat asc)
  float fv[KL];
  int ff[KL], fp[KL];
#pragma unroll
  for (int i = 0; i < KL; ++i) {
    fv[i] = s1v[i] + s2v[0];
    ff[i] = col1(i) * n + col2(0);
    fp[i] = 0;
  }
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    float bv = fv[0];
    int bf = ff[0], bi = 0, bp = fp[0];
#pragma unroll
    for (int i = 1; i < KL; ++i) {
      const bool better = fv[i] > bv || (fv[i] == bv && ff[i] < bf);
      bv = better ? fv[i] : bv;
      bf = better ? ff[i] : bf;
      bi = better ? i : bi;
      bp = better ? fp[i] : bp;
    }
    ip[r] = (int64_t)bf;
    wp[r] = expf(bv - V[0]) / z;
    const int np = bp + 1;
    float nv = -INFINITY;
    int nf = 0;
    if (np < KL) {
      nv = v1[bi] + v1[KL + np];
      nf = col1(bi) * n + col2(np);
    }
#pragma unroll
    for (int i = 0; i < KL; ++i) {
      if (i == bi) {
        fv[i] = nv;
        ff[i] = nf;
        fp[i] = np;
      }
    }
  }
}

// First pass: CTA c merges pairs [128c, 128c + 128).  Retry pass: a
// persistent grid walks the listed units (none listed: every CTA returns at
// once).
template <int KL>
__global__ void __launch_bounds__(kThreads)
merge_kernel(const float* __restrict__ list_v, const unsigned short* __restrict__ list_c, int B,
             int H, int n, int k, int64_t* __restrict__ idx, float* __restrict__ w,
             RetryScratch retry, bool retry_pass) {
  if (!retry_pass) {
    merge_cta<KL>(list_v, list_c, B, H, n, k, idx, w, retry, false, (int)blockIdx.x);
    return;
  }
  const int listed = retry.counts[1];
  for (int u = (int)blockIdx.x; u < listed; u += (int)gridDim.x) {
    merge_cta<KL>(list_v, list_c, B, H, n, k, idx, w, retry, true, u);
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
    attr_set = true;
  }
  const int64_t units = retry_units(B, H);
  const int64_t grid = retry_pass ? (units < 2 * tc_sms() ? units : 2 * tc_sms())
                                  : ((int64_t)B * H + kThreads - 1) / kThreads;
  merge_kernel<KL><<<(unsigned)grid, kThreads, smem, stream>>>(list_v, list_c, B, H, n, k, idx, w,
                                                                retry, retry_pass);
  return cudaGetLastError();
}

}  // namespace

int64_t retry_units(int64_t B, int64_t H) { return (B + kThreads - 1) / kThreads * H * 2; }

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
