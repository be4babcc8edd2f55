// Internal interface between the C-ABI layer (pkm_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkm.h"

namespace pkm {

// Device status word values are the PKM_ERR_* codes of pkm.h.

// The fp8 value table: codes [N, d_v] then fp32 scales [N] in `out`.
cudaError_t launch_quantize_fp8(const void* values, int value_dtype, int64_t N, int d_v, void* out,
                                cudaStream_t stream);

// Step a6 (value read).  values: [N, d_v] of value_dtype; idx/w: [B, H*k];
// out: [B, d_v] fp32.  Returns a cudaError_t of the launch.
cudaError_t launch_gather(const void* values, int value_dtype, int64_t N, int d_v, int B,
                          int rows_per_bag, const int64_t* idx, const float* w, float* out,
                          int* status, cudaStream_t stream);

// Steps a1-a5 for fp32 queries/subkeys on the CUDA cores.
cudaError_t launch_lookup_simt(const float* q, const float* subkeys, int B, int H, int d_q,
                               int n_keys, int k, int64_t* idx, float* w, cudaStream_t stream);

// Steps a1-a5 for bf16 queries/subkeys: tcgen05 scoring with the per-half
// selection fused into its epilogue, then the k^2 merge and softmax kernel.
// hint_z sets the per-row selection threshold (mean + hint_z * spread of a
// row's scores; any value gives exact results).  Device scratch: fb_count /
// fb_list (1 and B*H ints) list the (query, head) pairs recomputed by the
// CUDA-core fallback; list_v / list_c (B*H*2*list_slots(k) floats and
// 16-bit subkeys) hold the per-half lists between the two kernels.
cudaError_t launch_lookup_tc(const uint16_t* q, const uint16_t* subkeys, int B, int H, int d_q,
                             int n_keys, int k, float hint_z, int64_t* idx, float* w, int* status,
                             int* fb_count, int* fb_list, float* list_v, unsigned short* list_c,
                             cudaStream_t stream);

// Entries of one per-half list for a given k.
int list_slots(int k);

// Steps a4-a5 from the per-half lists (lookup_merge.cu).
cudaError_t launch_merge(const float* list_v, const unsigned short* list_c, int B, int H,
                         int n_keys, int k, int64_t* idx, float* w, int* fb_count, int* fb_list,
                         cudaStream_t stream);

// The hint_z launch_lookup_tc uses unless a handle overrides it.
float default_hint_z(int n_keys, int k);

// Exact recomputation of the listed (query, head) pairs, bf16 inputs, fp32
// FMA on the CUDA cores; grid CTAs walk pair_list[0 .. *pair_count).
cudaError_t launch_lookup_fallback(const uint16_t* q, const uint16_t* subkeys, int B, int H,
                                   int d_q, int n_keys, int k, const int* pair_count,
                                   const int* pair_list, int64_t* idx, float* w, int grid,
                                   cudaStream_t stream);

// Limits of each path (checked on the host before a launch).
constexpr int kSimtMaxK = 64;
constexpr int kSimtMaxNKeys = 4096;
constexpr int kSimtMaxDq = 8192;
constexpr int kTcMaxK = 32;
constexpr int kListMaxSlots = 32;  // list_slots(k) for every supported k
constexpr int kGatherMaxVecPerRow = 1024;  // 16-byte vectors per value row

}  // namespace pkm
