// Selection building blocks shared by the lookup kernels: sorting networks
// on values (alone, or carrying a 32-bit payload that orders equal values),
// a register binary search, the candidate-pair table of the k^2 merge and
// branch-free appends to per-thread logs in shared memory.
#pragma once

#include <stdint.h>

namespace pkm {

// Batcher's odd-even merge sort network on N (a power of two) inputs, as a
// compile-time list of compare-exchanges (hi, lo): 19, 63 and 191 of them
// for N = 8, 16 and 32, against 24, 80 and 240 for the bitonic sorter.
template <int N>
struct OddEvenMergeNet {
  template <typename F>
  static constexpr void visit(F f) {
    for (int p = 1; p < N; p <<= 1)
      for (int k = p; k >= 1; k >>= 1)
        for (int j = k % p; j + k < N; j += 2 * k)
          for (int i = 0; i < k && i < N - j - k; ++i)
            if ((i + j) / (2 * p) == (i + j + k) / (2 * p)) f(i + j, i + j + k);
  }
  static constexpr int count() {
    int c = 0;
    visit([&c](int, int) { ++c; });
    return c;
  }
  static constexpr int kCount = count();
  int hi[kCount], lo[kCount];
  constexpr OddEvenMergeNet() : hi(), lo() {
    int c = 0;
    visit([this, &c](int a, int b) {
      hi[c] = a;
      lo[c] = b;
      ++c;
    });
  }
};

// Sort of N values, descending, through the odd-even merge network.
template <int N>
__device__ __forceinline__ void sort_desc(float (&a)[N]) {
  constexpr OddEvenMergeNet<N> net{};
#pragma unroll
  for (int c = 0; c < net.kCount; ++c) {
    const float x = a[net.hi[c]], y = a[net.lo[c]];
    a[net.hi[c]] = fmaxf(x, y);
    a[net.lo[c]] = fminf(x, y);
  }
}

// V (descending, KL) <- the KL largest of V and B (descending, NB).  The
// elementwise max of V and B reversed (B padded with -inf) holds the KL
// largest of both and is bitonic; a bitonic merge sorts it.
template <int KL, int NB>
__device__ __forceinline__ void merge_top(float (&V)[KL], const float (&B)[NB]) {
  if constexpr (NB >= KL) {
#pragma unroll
    for (int i = 0; i < KL; ++i) V[i] = fmaxf(V[i], B[KL - 1 - i]);
  } else {
#pragma unroll
    for (int i = 0; i < NB; ++i) V[KL - NB + i] = fmaxf(V[KL - NB + i], B[NB - 1 - i]);
  }
#pragma unroll
  for (int stride = KL >> 1; stride > 0; stride >>= 1)
#pragma unroll
    for (int i = 0; i < KL; ++i) {
      const int j = i ^ stride;
      if (j > i) {
        const float hi = fmaxf(V[i], V[j]), lo = fminf(V[i], V[j]);
        V[i] = hi;
        V[j] = lo;
      }
    }
}

// Number of entries of V (descending) greater than x: a binary search whose
// probes are taken from registers by selects (no dynamic indexing).  P holds
// the current window of V, halved at every step.
template <int KL>
__device__ __forceinline__ int count_greater(const float (&V)[KL], float x) {
  float P[KL];
#pragma unroll
  for (int i = 0; i < KL; ++i) P[i] = V[i];
  int r = 0;
#pragma unroll
  for (int s = KL / 2; s >= 1; s >>= 1) {
    const bool gt = P[s - 1] > x;  // the whole lower half of the window is > x
    r += gt ? s : 0;
    if (s > 1) {
#pragma unroll
      for (int i = 0; i < s; ++i) P[i] = gt ? P[s + i] : P[i];
    }
  }
  return r;
}

// The candidate pairs (i, j) of the k^2 merge that can reach the top KL:
// (i + 1)(j + 1) <= KL, since every (i', j') with i' <= i and j' <= j scores
// at least as much.  Row-major, padded to a multiple of 32 with (-1, -1).
template <int KL>
struct MergePairs {
  static constexpr int count() {
    int c = 0;
    for (int i = 0; i < KL; ++i)
      for (int j = 0; (i + 1) * (j + 1) <= KL; ++j) ++c;
    return c;
  }
  static constexpr int kCount = count();
  static constexpr int kPadded = (kCount + 31) / 32 * 32;
  int i[kPadded], j[kPadded];
  constexpr MergePairs() : i(), j() {
    int c = 0;
    for (int a = 0; a < KL; ++a)
      for (int b = 0; (a + 1) * (b + 1) <= KL; ++b) {
        i[c] = a;
        j[c] = b;
        ++c;
      }
    for (; c < kPadded; ++c) {
      i[c] = -1;
      j[c] = -1;
    }
  }
};

// Append the 8-byte entry (v, col) at a log's end when v > thr, without a
// branch: one predicated store, and the shared-memory address of the next
// free slot advances by STEP bytes when the entry is taken.
template <int STEP>
__device__ __forceinline__ void log_push(uint32_t& a, float v, float thr, uint32_t col) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.gt.f32 p, %1, %2;\n\t"
      "@p st.shared.v2.b32 [%0], {%1, %3};\n\t"
      "@p add.u32 %0, %0, %4;\n\t}"
      : "+r"(a)
      : "f"(v), "f"(thr), "r"(col), "n"(STEP)
      : "memory");
}

// As log_push for a log filled from its top slot downwards: the address of
// the next free slot falls by STEP bytes when the entry is taken.  Two such
// logs, one growing up and one down in the same slots, give two
// independent address chains.
template <int STEP>
__device__ __forceinline__ void log_push_down(uint32_t& a, float v, float thr, uint32_t col) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.gt.f32 p, %1, %2;\n\t"
      "@p st.shared.v2.b32 [%0], {%1, %3};\n\t"
      "@p sub.u32 %0, %0, %4;\n\t}"
      : "+r"(a)
      : "f"(v), "f"(thr), "r"(col), "n"(STEP)
      : "memory");
}

// Append the score v at a stage's end when v > thr (predicated store; the
// address advances by STEP bytes when the score is taken).
template <int STEP>
__device__ __forceinline__ void stage_push(uint32_t& a, float v, float thr) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.gt.f32 p, %1, %2;\n\t"
      "@p st.shared.f32 [%0], %1;\n\t"
      "@p add.u32 %0, %0, %3;\n\t}"
      : "+r"(a)
      : "f"(v), "f"(thr), "n"(STEP)
      : "memory");
}

// Count v > thr in `count`; while the score address is below va_end, also
// store v at the score address and the 32-bit code OFF bytes after it
// (predicated stores, no branch), and advance the address by STEP.  Both
// outputs are written after every input has been read, so the compiler may
// place an input in an output's register.
template <int STEP, int OFF>
__device__ __forceinline__ void surv_push(uint32_t& va, uint32_t& count, uint32_t va_end, float v,
                                          float thr, uint32_t code) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.gt.f32 p, %2, %3;\n\t"
      "setp.lt.and.u32 q, %0, %5, p;\n\t"
      "@q st.shared.f32 [%0], %2;\n\t"
      "@q st.shared.b32 [%0+%7], %4;\n\t"
      "@q add.u32 %0, %0, %6;\n\t"
      "@p add.u32 %1, %1, 1;\n\t}"
      : "+r"(va), "+r"(count)
      : "f"(v), "f"(thr), "r"(code), "r"(va_end), "n"(STEP), "n"(OFF)
      : "memory");
}

// ----------------------------------------------- networks with a payload
//
// Lists in (value desc, payload asc) order: value-only compare-exchanges,
// then equal neighbours put in payload order (rows that hold none skip it).

// Compare-exchange (value desc) carrying a 32-bit payload.
__device__ __forceinline__ void cx_payload(float& a, float& b, uint32_t& ca, uint32_t& cb) {
  const bool sw = b > a;
  const float x = a, y = b;
  const uint32_t cx = ca, cy = cb;
  a = sw ? y : x;
  b = sw ? x : y;
  ca = sw ? cy : cx;
  cb = sw ? cx : cy;
}

template <int N>
__device__ __forceinline__ void sort_desc_payload(float (&a)[N], uint32_t (&c)[N]) {
  constexpr OddEvenMergeNet<N> net{};
#pragma unroll
  for (int q = 0; q < net.kCount; ++q) cx_payload(a[net.hi[q]], a[net.lo[q]], c[net.hi[q]], c[net.lo[q]]);
}

// Put equal neighbours of a (value desc) sorted list in payload order:
// odd-even transposition passes over the equal pairs, until a pass changes
// nothing.  Rows without equal finite neighbours skip it (the order of -inf
// padding does not matter).
template <int N>
__device__ __forceinline__ void order_ties(float (&a)[N], uint32_t (&c)[N]) {
  bool eq = false;
#pragma unroll
  for (int i = 0; i + 1 < N; ++i) eq |= a[i] == a[i + 1] && a[i] > -INFINITY;
  if (!eq) return;
#pragma unroll 1
  for (int pass = 0; pass < N; ++pass) {
    bool moved = false;
#pragma unroll
    for (int i = 0; i + 1 < N; ++i) {
      if ((i & 1) != (pass & 1)) continue;
      const bool sw = a[i] == a[i + 1] && c[i] > c[i + 1];
      const uint32_t x = c[i], y = c[i + 1];
      c[i] = sw ? y : x;
      c[i + 1] = sw ? x : y;
      moved |= sw;
    }
    if (!moved && pass > 0) break;
  }
}

// V / C (KL) <- the KL best of V and B (NB <= KL), both in (value desc,
// payload asc) order, payloads alongside: the first step pairs V's last NB
// with B reversed and keeps the better of each pair (a bitonic split, exact
// under that order), the rest is a bitonic merge by value.
template <int KL, int NB>
__device__ __forceinline__ void merge_top_payload(float (&V)[KL], uint32_t (&C)[KL],
                                                  const float (&Bv)[NB], const uint32_t (&Bc)[NB]) {
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const float a = V[KL - NB + i], b = Bv[NB - 1 - i];
    const uint32_t ca = C[KL - NB + i], cb = Bc[NB - 1 - i];
    const bool take = b > a || (b == a && cb < ca);
    V[KL - NB + i] = take ? b : a;
    C[KL - NB + i] = take ? cb : ca;
  }
#pragma unroll
  for (int stride = KL >> 1; stride > 0; stride >>= 1)
#pragma unroll
    for (int i = 0; i < KL; ++i) {
      const int j = i ^ stride;
      if (j > i) cx_payload(V[i], V[j], C[i], C[j]);
    }
  order_ties<KL>(V, C);
}

}  // namespace pkm
