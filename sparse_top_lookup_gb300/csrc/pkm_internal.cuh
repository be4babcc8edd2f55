// Internal interface between the C-ABI layer (pkm_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkm.h"

namespace pkm {

// Device status word values are the PKM_ERR_* codes of pkm.h.

// The fp8 value table: codes [N, d_v] then fp32 scales [N] in `out`.
cudaError_t launch_quantize_fp8(const void* values, int value_dtype, int64_t N, int d_v, void* out,
                                cudaStream_t stream);

// The query network (qnet.cu): per-feature scale / shift of an eval-mode
// BatchNorm1d, and q = (x W^T) * scale + shift in bf16 on the tensor cores.
cudaError_t launch_bn_fold(const float* gamma, const float* beta, const float* mean,
                           const float* var, float eps, int F, float* scale, float* shift,
                           cudaStream_t stream);
cudaError_t launch_qnet(const uint16_t* x, const uint16_t* w, int B, int dim, int F,
                        const float* scale, const float* shift, uint16_t* q, int* status,
                        cudaStream_t stream);
// The training form: q normalised by the batch's own per-feature mean and
// biased variance (two GEMM passes, see qnet.cu); workspace of
// qnet_batch_workspace_bytes(B, F); batch_mean / batch_var may be NULL.
size_t qnet_batch_workspace_bytes(int B, int F);
cudaError_t launch_qnet_batch(const uint16_t* x, const uint16_t* w, int B, int dim, int F,
                              const float* gamma, const float* beta, float eps, void* workspace,
                              uint16_t* q, float* batch_mean, float* batch_var, int* status,
                              cudaStream_t stream);

// Backward pass for a fixed selection (backward.cu), in two parts.
// Read part: dw = dout . V[idx] (overwritten) and the value-table gradient,
// either added to the dense dvalues (rows_out == NULL) or written sparse:
// the distinct selected rows ascending in rows_out[0 .. *n_rows) and their
// gradients in grad_rows [*n_rows, d_v]; bf16 or fp32 values; B*H*k < 2^31;
// workspace: backward_read_workspace_bytes.  Score part: dq overwritten and
// dsubkeys added to, from w, dw and the selection, through the winning
// subkeys only (fp32); bf16 queries/subkeys, k <= 32, d_q <= 2048;
// workspace: backward_scores_workspace_bytes.  A handle's backward scratch
// is backward_workspace_bytes: dw (backward_dw_bytes), then one region the
// two parts take in turn.
size_t backward_workspace_bytes(int B, int H, int n_keys, int k);
size_t backward_dw_bytes(int B, int H, int k);
size_t backward_read_workspace_bytes(int B, int H, int n_keys, int k);
size_t backward_scores_workspace_bytes(int B, int H, int n_keys, int k);
cudaError_t launch_backward_read(const void* values, int value_dtype, int B, int H, int n_keys,
                                 int d_v, int k, const int64_t* idx, const float* w,
                                 const float* dout, float* dw, float* dvalues, int64_t* rows_out,
                                 float* grad_rows, int* n_rows, void* workspace, int* status,
                                 cudaStream_t stream);
cudaError_t launch_backward_scores(const uint16_t* q, const uint16_t* subkeys, int B, int H,
                                   int d_q, int n_keys, int k, const int64_t* idx, const float* w,
                                   const float* dw, float* dq, float* dsubkeys, void* workspace,
                                   cudaStream_t stream);

// Step a6 (value read).  values: [N, d_v] of value_dtype; idx/w: [B, H*k];
// out: [B, d_v] fp32.  ctas > 0 and a row shape that gather_bulk_ok accepts:
// a persistent grid of at most ctas CTAs (one per SM) streaming whole rows
// with bulk copies; otherwise one CTA per bag on every SM.  Returns a
// cudaError_t of the launch.  stall (tests of the bounded waits only): the
// bulk-copy form issues no copy, so its consumers' waits run out (about 2 s)
// and it records PKM_ERR_TIMEOUT; the output is not meaningful.
cudaError_t launch_gather(const void* values, int value_dtype, int64_t N, int d_v, int B,
                          int rows_per_bag, const int64_t* idx, const float* w, float* out,
                          int* status, cudaStream_t stream, int ctas = 0, bool stall = false);
bool gather_bulk_ok(int value_dtype, int d_v, int rows_per_bag);

// Steps a1-a5 on the CUDA cores: fp32 queries/subkeys, and bf16 ones with a
// k above the tensor-core path's kTcMaxK (inputs widened exactly).
cudaError_t launch_lookup_simt(const float* q, const float* subkeys, int B, int H, int d_q,
                               int n_keys, int k, int64_t* idx, float* w, cudaStream_t stream);
cudaError_t launch_lookup_simt_bf16(const uint16_t* q, const uint16_t* subkeys, int B, int H,
                                    int d_q, int n_keys, int k, int64_t* idx, float* w,
                                    cudaStream_t stream);

// Device scratch of the bf16 lookup's retry pass.  A per-half list whose
// selection threshold hint was above the row's KL-th score is marked by the
// selection kernel; the merge then lists that list's work unit (128 queries x
// one head x one half; unit index ((row tile * H + head) << 1) | half), and
// the listed units are scored and selected again without the hint, which is
// exact by construction, and their pairs merged again.
// counts and unit_flag are one buffer (unit_flag == counts + 2), cleared at
// the start of each call by the main pass's selection kernel.
struct RetryScratch {
  int* counts;     // [0] pairs that had a marked list, [1] units listed for the retry
  int* unit_flag;  // [retry_units(B, H)]: nonzero once a unit is listed
  int* unit_list;  // [retry_units(B, H)]
};
int64_t retry_units(int64_t B, int64_t H);

// Steps a1-a5 for bf16 queries/subkeys: tcgen05 scoring with the per-half
// selection fused into its epilogue, then the k^2 merge and softmax kernel,
// then the retry pass (it returns at once when no unit is listed).  hint_z
// sets the per-row selection threshold (mean + hint_z * spread of a row's
// first scores; any value gives exact results).  list_v / list_c
// (B*H*2*list_slots(k) floats and 16-bit subkeys) hold the per-half lists
// between the kernels.
// stall (tests of the bounded waits only): the first selection launch loads
// nothing, so its pipeline wait runs out (about 2 s) and it records
// PKM_ERR_TIMEOUT; the lists it leaves are not meaningful.
// form: the selection kernel's main pass (PKM_OPT_SELECT_FORM: 0 automatic,
// 1 one-SM forms, 2 the two-SM form).
cudaError_t launch_lookup_tc(const uint16_t* q, const uint16_t* subkeys, int B, int H, int d_q,
                             int n_keys, int k, float hint_z, int64_t* idx, float* w, int* status,
                             const RetryScratch& retry, float* list_v, unsigned short* list_c,
                             cudaStream_t stream, bool stall = false, int form = 0);

// The two-SM selection kernel (lookup_2sm.cu), the main pass of a bf16
// lookup: per-half lists of every (query, head) in list_v / list_c.
// tmap_q: q viewed as [B][H][2][d_q/2] in 128x64 boxes; tmap_c_half: the
// subkeys viewed as [2H][n_keys][d_q/2] in 128x64 boxes; both 128-byte
// swizzled.  epi: the epilogue form (1: one set of epilogue warps, 2: two
// sets on alternate work units).  clear_words (may be NULL): clear_count
// ints the kernel zeroes before anything else (the call's retry
// bookkeeping, which the merge after it counts into).
cudaError_t launch_select_2sm(const CUtensorMap& tmap_q, const CUtensorMap& tmap_c_half, int B,
                              int H, int d_q, int n_keys, int k, float hint_z, float* list_v,
                              unsigned short* list_c, int* status, bool stall,
                              cudaStream_t stream, int epi = 2, int* clear_words = nullptr,
                              int clear_count = 0);

// The flat exact top-k (flat.cu), the baseline the factorisation replaces:
// the full key table [H][n_keys^2][d_q] (bf16) from the subkeys, and per
// (query, head) the top-k of all N full keys, each scored as one d_q-long
// dot product, with its softmax: idx / w [B][H][k] (flat index a * n_keys +
// b; ties to the lower index).  k <= kTcMaxK, d_q % 16 == 0.  The selection
// is the flat form of the two-SM kernel (tmap_q: q as [B][H][1][d_q] in
// 128x64 boxes; tmap_keys: the full keys in 128x64 boxes).
cudaError_t launch_full_keys(const uint16_t* subkeys, int H, int n_keys, int d_q, uint16_t* keys,
                             cudaStream_t stream);
cudaError_t launch_flat_lookup(const uint16_t* q, const uint16_t* keys, int B, int H, int d_q,
                               int N, int k, int64_t* idx, float* w, int* status,
                               cudaStream_t stream);
cudaError_t launch_select_2sm_flat(const CUtensorMap& tmap_q, const CUtensorMap& tmap_keys, int B,
                                   int H, int d_q, int N, int k, int64_t* idx, float* w,
                                   int* status, cudaStream_t stream);

// Entries of one per-half list for a given k.
int list_slots(int k);

// Steps a4-a5 from the per-half lists (lookup_merge.cu).  First pass: every
// pair; pairs with a marked list are counted in retry.counts[0] and their
// units listed.  Retry pass: the pairs of the units in
// retry.unit_list[0 .. retry.counts[1]), two CTAs per listed unit (64
// queries each).
cudaError_t launch_merge(const float* list_v, const unsigned short* list_c, int B, int H,
                         int n_keys, int k, int64_t* idx, float* w, const RetryScratch& retry,
                         bool retry_pass, cudaStream_t stream);

// The hint_z launch_lookup_tc uses unless a handle overrides it.
float default_hint_z(int n_keys, int k);

// Limits of each path (checked on the host before a launch).
constexpr int kSimtMaxK = 64;
constexpr int kSimtMaxNKeys = 4096;
constexpr int kSimtMaxDq = 8192;
constexpr int kTcMaxK = 32;
constexpr int kListMaxSlots = 32;  // list_slots(k) for every supported k
constexpr int kGatherMaxVecPerRow = 1024;  // 16-byte vectors per value row

}  // namespace pkm
