// The C ABI of include/pkm.h: argument checks, scratch ownership and launch
// order.  No arithmetic of the lookup lives here.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "pkm_internal.cuh"
#include "tc_common.cuh"

// pkm_forward_host staging slots: a call's copies in can start while the two
// calls before it still compute or copy out
constexpr int kHostSlots = 3;

struct pkm_handle {
  pkm_config cfg;
  int device;
  int64_t* ws_idx;   // [max_B, max_H, max_k] when the caller passes idx == NULL
  float* ws_w;       // [max_B, max_H, max_k] when the caller passes w == NULL
  int* status;       // device status word
  int* retry_counts;  // [2 + units]: pairs of the last bf16 lookup that needed the retry,
                      // units retried, then the per-unit flags (units = retry_units(max_B, max_H))
  int* unit_list;     // [units]
  void* bwd_ws;         // with_backward: dw and the two parts' scratch
  float* list_v;     // [max_B * max_H * 2 * 32] per-half lists between the two bf16 kernels
  unsigned short* list_c;
  float hint_z;      // selection threshold hint override (NaN: automatic)
  // pkm_forward_host staging (optional), kHostSlots slots used by turns, so
  // call's copies in can run while the previous call computes
  void* stage_q[kHostSlots];
  float* stage_out[kHostSlots];
  int64_t* stage_idx[kHostSlots];
  float* stage_w[kHostSlots];
  int next_slot;
  // pkm_forward_host pipeline: copies in / out on their own streams, so the
  // copy engines move batch i+1 in and batch i-1 out while batch i computes;
  // ev_done[s]: the last copy out of the call that used slot s
  cudaStream_t s_in, s_out;
  cudaEvent_t ev_done[kHostSlots], ev_in[PKM_HOST_MAX_CHUNKS], ev_comp[PKM_HOST_MAX_CHUNKS];
  int host_chunks;
  bool host_chunks_set;  // PKM_OPT_HOST_CHUNKS given by the caller
  int test_stall;        // PKM_OPT_TEST_STALL: 1 stalls the selection kernel, 2 the bulk read
  int sms;               // SMs of the device
  int read_sms;          // PKM_OPT_READ_SMS: SMs of the value read (0: all)
  int select_form;       // PKM_OPT_SELECT_FORM
};

namespace {

int elem_size(int dtype) { return dtype == PKM_FP8_E4M3 ? 1 : dtype == PKM_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_config(const pkm_config* c) {
  if (!c) return PKM_ERR_INVALID;
  if (c->d_q < 2 || (c->d_q & 1) || c->d_v < 1) return PKM_ERR_INVALID;
  if (c->max_B < 0 || c->max_H < 1 || c->max_n_keys < 1 || c->max_k < 1) return PKM_ERR_INVALID;
  for (int dt : {c->q_dtype, c->key_dtype})
    if (dt != PKM_F32 && dt != PKM_BF16) return PKM_ERR_UNSUPPORTED;
  if (c->value_dtype != PKM_F32 && c->value_dtype != PKM_BF16 && c->value_dtype != PKM_FP8_E4M3)
    return PKM_ERR_UNSUPPORTED;
  if (c->q_dtype != c->key_dtype) return PKM_ERR_UNSUPPORTED;
  if (c->with_backward && (c->q_dtype != PKM_BF16 || c->value_dtype == PKM_FP8_E4M3 ||
                           c->d_q > 2048 ||
                          (int64_t)c->max_B * c->max_H * c->max_k > INT32_MAX ||
                          (int64_t)c->max_B * c->d_v / 4 > INT32_MAX))
    return PKM_ERR_UNSUPPORTED;
  if ((int64_t)c->d_v * elem_size(c->value_dtype) % 16) return PKM_ERR_UNSUPPORTED;
  if ((int64_t)c->d_v * elem_size(c->value_dtype) / 16 > pkm::kGatherMaxVecPerRow)
    return PKM_ERR_UNSUPPORTED;
  if (c->q_dtype == PKM_BF16) {
    if (c->d_q % 16) return PKM_ERR_UNSUPPORTED;  // TMA strides are multiples of 16 bytes
    // k above the tensor-core path's lists: the CUDA-core path (forward only)
    if (c->max_k > pkm::kTcMaxK &&
        (c->max_k > pkm::kSimtMaxK || c->d_q > pkm::kSimtMaxDq ||
         c->max_n_keys > pkm::kSimtMaxNKeys || c->with_backward))
      return PKM_ERR_UNSUPPORTED;
  } else {
    if (c->d_q > pkm::kSimtMaxDq || c->max_k > pkm::kSimtMaxK) return PKM_ERR_UNSUPPORTED;
    if (c->max_n_keys > pkm::kSimtMaxNKeys) return PKM_ERR_UNSUPPORTED;
  }
  if ((int64_t)c->max_n_keys * c->max_n_keys > INT32_MAX) return PKM_ERR_UNSUPPORTED;
  return PKM_OK;
}

int check_call(const pkm_config* c, int B, int H, int n, int k) {
  int rc = check_config(c);
  if (rc) return rc;
  if (B < 0 || H < 1 || n < 1 || k < 1) return PKM_ERR_INVALID;
  if (B > c->max_B || H > c->max_H || n > c->max_n_keys || k > c->max_k || k > n)
    return PKM_ERR_RANGE;
  if (B > 0 && (int64_t)B * H > INT32_MAX) return PKM_ERR_RANGE;
  return PKM_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? PKM_OK : PKM_ERR_CUDA; }

int run_lookup(pkm_t h, const void* q, const void* subkeys, int B, int H, int n, int k,
               int64_t* idx, float* w, cudaStream_t s) {
  if (h->cfg.q_dtype == PKM_BF16 && k > pkm::kTcMaxK) {
    // exact without a threshold hint: nothing to retry (the count reads 0)
    if (cudaMemsetAsync(h->retry_counts, 0, sizeof(int), s) != cudaSuccess) return PKM_ERR_CUDA;
    return cuda_rc(pkm::launch_lookup_simt_bf16(static_cast<const uint16_t*>(q),
                                                static_cast<const uint16_t*>(subkeys), B, H,
                                                h->cfg.d_q, n, k, idx, w, s));
  }
  if (h->cfg.q_dtype == PKM_BF16) {
    const float z = isnan(h->hint_z) ? pkm::default_hint_z(n, k) : h->hint_z;
    return cuda_rc(pkm::launch_lookup_tc(static_cast<const uint16_t*>(q),
                                         static_cast<const uint16_t*>(subkeys), B, H, h->cfg.d_q,
                                         n, k, z, idx, w, h->status,
                                         {h->retry_counts, h->retry_counts + 2, h->unit_list},
                                         h->list_v, h->list_c, s, (h->test_stall & 1) != 0,
                                         h->select_form));
  }
  return cuda_rc(pkm::launch_lookup_simt(static_cast<const float*>(q),
                                         static_cast<const float*>(subkeys), B, H, h->cfg.d_q, n,
                                         k, idx, w, s));
}

// ctas: SMs of the read (bulk-copy form where the row shape suits it); 0:
// the handle's PKM_OPT_READ_SMS, whose 0 means every SM
int run_gather(pkm_t h, const void* values, int B, int H, int n, int k, const int64_t* idx,
               const float* w, float* out, cudaStream_t s, int ctas = 0) {
  if (ctas <= 0) ctas = h->read_sms > 0 ? h->read_sms : h->sms;
  return cuda_rc(pkm::launch_gather(values, h->cfg.value_dtype, (int64_t)n * n, h->cfg.d_v, B,
                                    H * k, idx, w, out, h->status, s, ctas,
                                    (h->test_stall & 2) != 0));
}

}  // namespace

extern "C" {

int pkm_abi_version(void) { return PKM_ABI_VERSION; }

const char* pkm_strerror(int code) {
  switch (code) {
    case PKM_OK: return "ok";
    case PKM_ERR_INVALID: return "invalid argument (NULL pointer, non-positive or odd dimension)";
    case PKM_ERR_RANGE: return "size outside the handle's configuration or k > n_keys";
    case PKM_ERR_UNSUPPORTED: return "unsupported dtype combination, k or layout";
    case PKM_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case PKM_ERR_CUDA: return "CUDA runtime error";
    case PKM_ERR_NOMEM: return "device allocation failed";
    case PKM_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case PKM_ERR_BAD_INDEX: return "row index outside the value table";
    case PKM_ERR_NO_STAGING: return "handle was created without host staging";
    case PKM_ERR_OPTION: return "unknown option or value";
    case PKM_ERR_NO_BACKWARD: return "handle was created without with_backward";
    default: return "unknown error code";
  }
}

int pkm_check_args(const pkm_config* cfg, int B, int H, int n_keys, int k) {
  return check_call(cfg, B, H, n_keys, k);
}

void pkm_destroy(pkm_t h) {
  if (!h) return;
  cudaFree(h->ws_idx);
  cudaFree(h->ws_w);
  cudaFree(h->status);
  cudaFree(h->retry_counts);
  cudaFree(h->unit_list);
  cudaFree(h->list_v);
  cudaFree(h->list_c);
  cudaFree(h->bwd_ws);
  for (int s = 0; s < kHostSlots; ++s) {
    cudaFree(h->stage_q[s]);
    cudaFree(h->stage_out[s]);
    cudaFree(h->stage_idx[s]);
    cudaFree(h->stage_w[s]);
    if (h->ev_done[s]) cudaEventDestroy(h->ev_done[s]);
  }
  if (h->s_in) cudaStreamDestroy(h->s_in);
  if (h->s_out) cudaStreamDestroy(h->s_out);
  for (int i = 0; i < PKM_HOST_MAX_CHUNKS; ++i) {
    if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
    if (h->ev_comp[i]) cudaEventDestroy(h->ev_comp[i]);
  }
  free(h);
}

int pkm_create(pkm_t* out, const pkm_config* cfg) {
  if (!out) return PKM_ERR_INVALID;
  int rc = check_config(cfg);
  if (rc) return rc;
  pkm_t h = static_cast<pkm_t>(calloc(1, sizeof(pkm_handle)));
  if (!h) return PKM_ERR_NOMEM;
  h->cfg = *cfg;
  h->hint_z = NAN;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    free(h);
    return PKM_ERR_CUDA;
  }
  const size_t sel = (size_t)cfg->max_B * cfg->max_H * cfg->max_k;
  bool ok = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device) ==
                cudaSuccess &&
            cudaMalloc(&h->status, sizeof(int)) == cudaSuccess &&
            cudaMemset(h->status, 0, sizeof(int)) == cudaSuccess;
  if (ok && sel) {
    ok = cudaMalloc(&h->ws_idx, sel * sizeof(int64_t)) == cudaSuccess &&
         cudaMalloc(&h->ws_w, sel * sizeof(float)) == cudaSuccess;
  }
  if (ok) {
    const size_t pairs = (size_t)cfg->max_B * cfg->max_H;
    const size_t units =
        cfg->q_dtype == PKM_BF16 ? (size_t)pkm::retry_units(cfg->max_B, cfg->max_H) : 0;
    ok = cudaMalloc(&h->retry_counts, (2 + units) * sizeof(int)) == cudaSuccess &&
         cudaMemset(h->retry_counts, 0, (2 + units) * sizeof(int)) == cudaSuccess &&
         cudaMalloc(&h->unit_list, (units ? units : 1) * sizeof(int)) == cudaSuccess;
    if (ok && cfg->q_dtype == PKM_BF16 && pairs) {
      const size_t slots = pairs * 2 * pkm::kListMaxSlots;
      ok = cudaMalloc(&h->list_v, slots * sizeof(float)) == cudaSuccess &&
           cudaMalloc(&h->list_c, slots * sizeof(unsigned short)) == cudaSuccess;
    }
  }
  if (ok && cfg->host_staging && cfg->max_B) {
    const size_t qb = (size_t)cfg->max_B * cfg->max_H * cfg->d_q * elem_size(cfg->q_dtype);
    for (int st = 0; ok && st < kHostSlots; ++st)
      ok = cudaMalloc(&h->stage_q[st], qb) == cudaSuccess &&
           cudaMalloc(&h->stage_out[st], (size_t)cfg->max_B * cfg->d_v * sizeof(float)) ==
               cudaSuccess &&
           cudaMalloc(&h->stage_idx[st], sel * sizeof(int64_t)) == cudaSuccess &&
           cudaMalloc(&h->stage_w[st], sel * sizeof(float)) == cudaSuccess &&
           cudaEventCreateWithFlags(&h->ev_done[st], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < PKM_HOST_MAX_CHUNKS; ++i)
      ok = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&h->ev_comp[i], cudaEventDisableTiming) == cudaSuccess;
    h->host_chunks = 3;
  }
  if (ok && cfg->with_backward) {
    const size_t ws = pkm::backward_workspace_bytes(cfg->max_B, cfg->max_H, cfg->max_n_keys,
                                                    cfg->max_k);
    ok = cudaMalloc(&h->bwd_ws, ws ? ws : 256) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    pkm_destroy(h);
    return PKM_ERR_NOMEM;
  }
  *out = h;
  return PKM_OK;
}

int pkm_lookup(pkm_t h, const void* q, const void* subkeys, int B, int H, int n_keys, int k,
               int64_t* idx, float* w, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (B == 0) return PKM_OK;
  if (!q || !subkeys || !idx || !w) return PKM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(subkeys) || !aligned16(idx) || !aligned16(w))
    return PKM_ERR_ALIGN;
  return run_lookup(h, q, subkeys, B, H, n_keys, k, idx, w, static_cast<cudaStream_t>(stream));
}

int pkm_full_keys(pkm_t h, const void* subkeys, int H, int n_keys, void* keys, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, 0, H, n_keys, 1);
  if (rc) return rc;
  if (h->cfg.key_dtype != PKM_BF16) return PKM_ERR_UNSUPPORTED;
  if (!subkeys || !keys) return PKM_ERR_INVALID;
  if (!aligned16(subkeys) || !aligned16(keys)) return PKM_ERR_ALIGN;
  return cuda_rc(pkm::launch_full_keys(static_cast<const uint16_t*>(subkeys), H, n_keys,
                                       h->cfg.d_q, static_cast<uint16_t*>(keys),
                                       static_cast<cudaStream_t>(stream)));
}

int pkm_flat_lookup(pkm_t h, const void* q, const void* keys, int B, int H, int n_keys, int k,
                    int64_t* idx, float* w, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (h->cfg.q_dtype != PKM_BF16 || k > pkm::kTcMaxK) return PKM_ERR_UNSUPPORTED;
  if (B == 0) return PKM_OK;
  if (!q || !keys || !idx || !w) return PKM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(keys) || !aligned16(idx) || !aligned16(w))
    return PKM_ERR_ALIGN;
  return cuda_rc(pkm::launch_flat_lookup(static_cast<const uint16_t*>(q),
                                         static_cast<const uint16_t*>(keys), B, H, h->cfg.d_q,
                                         n_keys * n_keys, k, idx, w, h->status,
                                         static_cast<cudaStream_t>(stream)));
}

int pkm_gather(pkm_t h, const void* values, int B, int H, int n_keys, int k, const int64_t* idx,
               const float* w, float* out, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (B == 0) return PKM_OK;
  if (!values || !idx || !w || !out) return PKM_ERR_INVALID;
  if (!aligned16(values) || !aligned16(idx) || !aligned16(w) || !aligned16(out))
    return PKM_ERR_ALIGN;
  return run_gather(h, values, B, H, n_keys, k, idx, w, out, static_cast<cudaStream_t>(stream));
}

int pkm_forward(pkm_t h, const void* q, const void* subkeys, const void* values, int B, int H,
                int n_keys, int k, float* out, int64_t* idx, float* w, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (B == 0) return PKM_OK;
  if (!q || !subkeys || !values || !out) return PKM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(subkeys) || !aligned16(values) || !aligned16(out) ||
      (idx && !aligned16(idx)) || (w && !aligned16(w)))
    return PKM_ERR_ALIGN;
  if (!idx) idx = h->ws_idx;
  if (!w) w = h->ws_w;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = run_lookup(h, q, subkeys, B, H, n_keys, k, idx, w, s);
  if (rc) return rc;
  return run_gather(h, values, B, H, n_keys, k, idx, w, out, s);
}

// The part of a handle's backward scratch the read and score parts take in turn.
static void* backward_region(pkm_t h) {
  return static_cast<unsigned char*>(h->bwd_ws) +
         pkm::backward_dw_bytes(h->cfg.max_B, h->cfg.max_H, h->cfg.max_k);
}

// The read part, dense (rows == NULL: dvalues added to) or sparse.
static int backward_read(pkm_t h, const void* values, int B, int H, int n_keys, int k,
                         const int64_t* idx, const float* w, const float* dout, float* dw,
                         float* dvalues, int64_t* rows, float* grad_rows, int* n_rows,
                         void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (!h->cfg.with_backward) return PKM_ERR_NO_BACKWARD;
  const bool sparse = rows != nullptr || grad_rows != nullptr || n_rows != nullptr;
  if (sparse && (!rows || !grad_rows || !n_rows)) return PKM_ERR_INVALID;
  if (!sparse && B == 0) return PKM_OK;
  if (B > 0 && (!values || !idx || !w || !dout || !dw || (!sparse && !dvalues)))
    return PKM_ERR_INVALID;
  for (const void* p : {values, (const void*)idx, (const void*)w, (const void*)dout,
                        (const void*)dw, (const void*)dvalues, (const void*)rows,
                        (const void*)grad_rows})
    if (p && !aligned16(p)) return PKM_ERR_ALIGN;
  return cuda_rc(pkm::launch_backward_read(values, h->cfg.value_dtype, B, H, n_keys,
                                           h->cfg.d_v, k, idx, w, dout, dw, dvalues, rows,
                                           grad_rows, n_rows, backward_region(h), h->status,
                                           static_cast<cudaStream_t>(stream)));
}

int pkm_backward_read(pkm_t h, const void* values, int B, int H, int n_keys, int k,
                      const int64_t* idx, const float* w, const float* dout, float* dw,
                      float* dvalues, void* stream) {
  if (!dvalues && B > 0) return PKM_ERR_INVALID;
  return backward_read(h, values, B, H, n_keys, k, idx, w, dout, dw, dvalues, nullptr, nullptr,
                       nullptr, stream);
}

int pkm_backward_read_sparse(pkm_t h, const void* values, int B, int H, int n_keys, int k,
                             const int64_t* idx, const float* w, const float* dout, float* dw,
                             int64_t* rows, float* grad_rows, int* n_rows, void* stream) {
  if (!rows || !grad_rows || !n_rows) return PKM_ERR_INVALID;
  return backward_read(h, values, B, H, n_keys, k, idx, w, dout, dw, nullptr, rows, grad_rows,
                       n_rows, stream);
}

int pkm_backward_scores(pkm_t h, const void* q, const void* subkeys, int B, int H, int n_keys,
                        int k, const int64_t* idx, const float* w, const float* dw, float* dq,
                        float* dsubkeys, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (!h->cfg.with_backward) return PKM_ERR_NO_BACKWARD;
  if (B == 0) return PKM_OK;
  if (!q || !subkeys || !idx || !w || !dw || !dq || !dsubkeys) return PKM_ERR_INVALID;
  for (const void* p : {q, subkeys, (const void*)idx, (const void*)w, (const void*)dw,
                        (const void*)dq, (const void*)dsubkeys})
    if (!aligned16(p)) return PKM_ERR_ALIGN;
  return cuda_rc(pkm::launch_backward_scores(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(subkeys), B, H, h->cfg.d_q,
      n_keys, k, idx, w, dw, dq, dsubkeys, backward_region(h),
      static_cast<cudaStream_t>(stream)));
}

static int backward_all(pkm_t h, const void* q, const void* subkeys, const void* values, int B,
                        int H, int n_keys, int k, const int64_t* idx, const float* w,
                        const float* dout, float* dq, float* dsubkeys, float* dvalues,
                        int64_t* rows, float* grad_rows, int* n_rows, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (!h->cfg.with_backward) return PKM_ERR_NO_BACKWARD;
  if (B > 0 && (!q || !subkeys || !dq || !dsubkeys)) return PKM_ERR_INVALID;
  float* dw = static_cast<float*>(h->bwd_ws);
  rc = backward_read(h, values, B, H, n_keys, k, idx, w, dout, dw, dvalues, rows, grad_rows,
                     n_rows, stream);
  if (rc || B == 0) return rc;
  return pkm_backward_scores(h, q, subkeys, B, H, n_keys, k, idx, w, dw, dq, dsubkeys, stream);
}

int pkm_backward(pkm_t h, const void* q, const void* subkeys, const void* values, int B, int H,
                 int n_keys, int k, const int64_t* idx, const float* w, const float* dout,
                 float* dq, float* dsubkeys, float* dvalues, void* stream) {
  if (!dvalues && B > 0) return PKM_ERR_INVALID;
  return backward_all(h, q, subkeys, values, B, H, n_keys, k, idx, w, dout, dq, dsubkeys, dvalues,
                      nullptr, nullptr, nullptr, stream);
}

int pkm_backward_sparse(pkm_t h, const void* q, const void* subkeys, const void* values, int B,
                        int H, int n_keys, int k, const int64_t* idx, const float* w,
                        const float* dout, float* dq, float* dsubkeys, int64_t* rows,
                        float* grad_rows, int* n_rows, void* stream) {
  if (!rows || !grad_rows || !n_rows) return PKM_ERR_INVALID;
  return backward_all(h, q, subkeys, values, B, H, n_keys, k, idx, w, dout, dq, dsubkeys, nullptr,
                      rows, grad_rows, n_rows, stream);
}

// The host-buffer forward: the batch in slices, each slice's copy in on s_in,
// its lookup and read on `stream`, its copies out on s_out.  The call takes
// the next of the kHostSlots staging slots; its copies in first wait (on the
// device) for the last copy out of the call that used the slot before, so
// kHostSlots calls can be in flight.  sync: wait for the copies out; else record
// `done` on s_out after them.
static int forward_host(pkm_t h, const void* q_host, const void* subkeys, const void* values,
                        int B, int H, int n_keys, int k, float* out_host, int64_t* idx_host,
                        float* w_host, cudaStream_t s, bool sync, cudaEvent_t done) {
  if (!h) return PKM_ERR_INVALID;
  int rc = check_call(&h->cfg, B, H, n_keys, k);
  if (rc) return rc;
  if (B == 0) return sync ? PKM_OK : cuda_rc(cudaEventRecord(done, h->s_out));
  if (!h->stage_q[0]) return PKM_ERR_NO_STAGING;
  if (!q_host || !subkeys || !values || !out_host) return PKM_ERR_INVALID;
  if (!aligned16(subkeys) || !aligned16(values)) return PKM_ERR_ALIGN;
  const int slot = h->next_slot;
  h->next_slot = (slot + 1) % kHostSlots;
  const size_t qrow = (size_t)H * h->cfg.d_q * elem_size(h->cfg.q_dtype);  // bytes per query
  const size_t orow = (size_t)h->cfg.d_v * sizeof(float);
  const size_t srow = (size_t)H * k;  // selections per query
  // batch split into at most host_chunks slices, each a multiple of 8
  // queries (keeps every device offset 16-byte aligned); the first and the
  // last slice are half the size of the others, which shortens the pipeline's
  // fill (the first slice's copy in) and drain (the last slice's copy out):
  // slice i covers [cut(i), cut(i+1)) with cut(i) = B * (i - 1/2) / (chunks - 1)
  // (pkm_forward_host_async: one slice unless the caller chose the count;
  // the call in flight beside it already hides its copies)
  const int want = !sync && !h->host_chunks_set ? 1 : h->host_chunks < 1 ? 1 : h->host_chunks;
  int cut[PKM_HOST_MAX_CHUNKS + 1];
  int chunks = 0;
  cut[0] = 0;
  for (int i = 1; i <= want; ++i) {
    int64_t c = i == want ? B : ((int64_t)B * (2 * i - 1) / (2 * (want - 1)) + 7) / 8 * 8;
    if (c > B) c = B;
    if (c > cut[chunks]) cut[++chunks] = (int)c;
  }
  const char* qh = static_cast<const char*>(q_host);
  char* qd = static_cast<char*>(h->stage_q[slot]);
  // copies in wait for the slot's previous user to have copied its results
  // out (copies out follow each slice's computation, itself after the
  // caller's earlier work on `stream`)
  if (cudaStreamWaitEvent(h->s_in, h->ev_done[slot], 0) != cudaSuccess) return PKM_ERR_CUDA;
  for (int c = 0; c < chunks; ++c) {
    const int b0 = cut[c], nb = cut[c + 1] - cut[c];
    if (cudaMemcpyAsync(qd + b0 * qrow, qh + b0 * qrow, nb * qrow, cudaMemcpyHostToDevice,
                        h->s_in) != cudaSuccess ||
        cudaEventRecord(h->ev_in[c], h->s_in) != cudaSuccess ||
        cudaStreamWaitEvent(s, h->ev_in[c], 0) != cudaSuccess)
      return PKM_ERR_CUDA;
    int64_t* idx_d = h->stage_idx[slot] + b0 * srow;
    float* w_d = h->stage_w[slot] + b0 * srow;
    float* out_d = h->stage_out[slot] + (size_t)b0 * h->cfg.d_v;
    rc = run_lookup(h, qd + b0 * qrow, subkeys, nb, H, n_keys, k, idx_d, w_d, s);
    if (rc) return rc;
    rc = run_gather(h, values, nb, H, n_keys, k, idx_d, w_d, out_d, s);
    if (rc) return rc;
    if (cudaEventRecord(h->ev_comp[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(h->s_out, h->ev_comp[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(out_host + (size_t)b0 * h->cfg.d_v, out_d, nb * orow,
                        cudaMemcpyDeviceToHost, h->s_out) != cudaSuccess)
      return PKM_ERR_CUDA;
    if (idx_host && cudaMemcpyAsync(idx_host + b0 * srow, idx_d, nb * srow * sizeof(int64_t),
                                    cudaMemcpyDeviceToHost, h->s_out) != cudaSuccess)
      return PKM_ERR_CUDA;
    if (w_host && cudaMemcpyAsync(w_host + b0 * srow, w_d, nb * srow * sizeof(float),
                                  cudaMemcpyDeviceToHost, h->s_out) != cudaSuccess)
      return PKM_ERR_CUDA;
  }
  if (cudaEventRecord(h->ev_done[slot], h->s_out) != cudaSuccess) return PKM_ERR_CUDA;
  if (!sync) return cuda_rc(cudaEventRecord(done, h->s_out));
  if (cudaStreamWaitEvent(s, h->ev_done[slot], 0) != cudaSuccess) return PKM_ERR_CUDA;
  return cuda_rc(cudaStreamSynchronize(s));
}

int pkm_forward_host(pkm_t h, const void* q_host, const void* subkeys, const void* values, int B,
                     int H, int n_keys, int k, float* out_host, int64_t* idx_host, float* w_host,
                     void* stream) {
  return forward_host(h, q_host, subkeys, values, B, H, n_keys, k, out_host, idx_host, w_host,
                      static_cast<cudaStream_t>(stream), true, nullptr);
}

int pkm_forward_host_async(pkm_t h, const void* q_host, const void* subkeys, const void* values,
                           int B, int H, int n_keys, int k, float* out_host, int64_t* idx_host,
                           float* w_host, void* stream, void* done_event) {
  if (!done_event) return PKM_ERR_INVALID;
  return forward_host(h, q_host, subkeys, values, B, H, n_keys, k, out_host, idx_host, w_host,
                      static_cast<cudaStream_t>(stream), false,
                      static_cast<cudaEvent_t>(done_event));
}

int pkm_set_option(pkm_t h, int option, double value) {
  if (!h) return PKM_ERR_INVALID;
  switch (option) {
    case PKM_OPT_HINT_Z:
      if (!isnan(value) && !isfinite(value)) return PKM_ERR_OPTION;
      h->hint_z = (float)value;
      return PKM_OK;
    case PKM_OPT_HOST_CHUNKS:
      if (!(value >= 1 && value <= PKM_HOST_MAX_CHUNKS) || value != (int)value)
        return PKM_ERR_OPTION;
      h->host_chunks = (int)value;
      h->host_chunks_set = true;
      return PKM_OK;
    case PKM_OPT_TEST_STALL:
      if (!(value >= 0 && value <= 3) || value != (int)value) return PKM_ERR_OPTION;
      h->test_stall = (int)value;
      return PKM_OK;
    case PKM_OPT_SELECT_FORM:
      if (!(value >= 0 && value <= 3) || value != (int)value) return PKM_ERR_OPTION;
      h->select_form = (int)value;
      return PKM_OK;
    case PKM_OPT_READ_SMS:
      if (!(value >= 0 && value <= h->sms) || value != (int)value) return PKM_ERR_OPTION;
      h->read_sms = (int)value;
      return PKM_OK;
    default:
      return PKM_ERR_OPTION;
  }
}

int pkm_multicast_ok(const void* const* ptrs, int count) {
  if (!ptrs || count < 0) return 0;
  return pkm::tc::buffers_on_this_device(ptrs, count) ? 1 : 0;
}

int pkm_get_fallback_count(pkm_t h, void* stream, int* count) {
  if (!h || !count) return PKM_ERR_INVALID;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKM_ERR_CUDA;
  if (cudaMemcpy(count, h->retry_counts, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PKM_ERR_CUDA;
  return PKM_OK;
}

int pkm_get_status(pkm_t h, void* stream) {
  if (!h) return PKM_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKM_ERR_CUDA;
  if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PKM_ERR_CUDA;
  if (v != PKM_OK && cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) return PKM_ERR_CUDA;
  return v;
}

}  // extern "C"
