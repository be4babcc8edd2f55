/*
 * pkm.h - C ABI of the product-key memory (PKM) lookup on one NVIDIA GB300
 * GPU (sm_103a): the forward pass (pkm_forward; its two stages pkm_lookup and
 * pkm_gather; pkm_forward_host / pkm_forward_host_async with host buffers;
 * the allocation-free pkm_lookup_static), its backward pass for the selection
 * it made (pkm_backward, pkm_backward_sparse and their two parts), the query
 * network ahead of it (pkm_bn_fold, pkm_query_net) and the fp8 value-table
 * quantiser (pkm_quantize_values_fp8).
 *
 * The operation (Product-Key Memory, "Factorising the key space", and the
 * forward method of the page's code listing; Memory Retrieval Mechanisms,
 * the top-k retrieval equations):
 *
 *   for every query b and head h, with q = q[b,h,:] split into halves
 *   q1 = q[0 : d_q/2] and q2 = q[d_q/2 : d_q]:
 *     s1[a] = q1 . C[h,0,a,:]          s2[a] = q2 . C[h,1,a,:]      (a < n_keys)
 *     A1 = top-k of s1, A2 = top-k of s2                  (per-half winners)
 *     candidates (i, j) in A1 x A2: score s1[i] + s2[j], flat i*n_keys + j
 *     idx[b,h,:] = the k best candidates, (score desc, flat asc)
 *     w[b,h,:]   = softmax of their scores (no temperature)
 *   out[b,:] = sum over h and j of w[b,h,j] * V[idx[b,h,j], :]
 *
 * The factorised search is exact: its result equals a top-k over all
 * n_keys^2 full keys (q . concat(C[h,0,a], C[h,1,j])).  Ties are broken
 * toward the lower subkey index within a half and the lower flat index
 * overall.  Heads score their own subkeys with their own slice of q, share
 * one value table, and their reads are summed.
 *
 * Layouts (all row-major, contiguous, device memory unless stated):
 *   q        [B, H, d_q]            q_dtype
 *   subkeys  [H, 2, n_keys, d_q/2]  key_dtype   (must equal q_dtype)
 *   values   [n_keys^2, d_v]        value_dtype (PKM_FP8_E4M3: see below)
 *   out      [B, d_v]               fp32, overwritten
 *   idx      [B, H, k]              int64 flat row indices
 *   w        [B, H, k]              fp32 softmax weights aligned with idx
 * bf16 arguments are raw IEEE bfloat16 bit patterns (uint16).
 *
 * Low-precision value table (Product-Key Memory, note after the code listing:
 * the value table is "a good candidate for keeping in a lower precision"):
 * with value_dtype = PKM_FP8_E4M3, `values` is one buffer holding the
 * N = n_keys^2 rows of d_v fp8 e4m3 codes (N * d_v bytes, row-major) followed
 * directly by N fp32 row scales; row r reads as V[r, c] = e4m3(code[r, c]) *
 * scale[r].  e4m3 is the OCP 8-bit floating-point format (bias 7, 3 mantissa
 * bits, subnormals, no infinities, largest finite 448).
 * pkm_quantize_values_fp8 writes such a buffer from an fp32 or bf16 table.
 *
 * Arithmetic: bf16 queries and subkeys are scored on the tensor cores with
 * fp32 accumulation; fp32 queries and subkeys are scored with fp32 FMA on the
 * CUDA cores.  Candidate sums, the softmax and the weighted row sum are fp32.
 *
 * Ownership: the caller owns every tensor pointer; nothing is retained after a
 * call returns.  A handle owns only its scratch (device workspace for idx/w
 * when the caller passes NULL, a device status word, optional staging for
 * pkm_forward_host, and for pkm_backward the gradient
 * scratch).  pkm_create is the only call that allocates.
 *
 * Asynchrony: every call enqueues work on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and returns without synchronising, except
 * pkm_get_status and pkm_forward_host, which synchronise `stream`
 * (pkm_forward_host_async signals an event instead).  Results are
 * valid once the stream has been synchronised.  Calls on one handle must not
 * overlap on the GPU when they use the handle's scratch (idx/w == NULL, every
 * backward call, every host-buffer call).
 *
 * Errors: every call returns PKM_OK (0) or a negative code, checked on the
 * host before anything is launched.  Device-side failures (an out-of-range
 * index reaching the value read, a bounded wait that gave up) are recorded in
 * the handle's status word and returned by pkm_get_status.
 */
#ifndef PKM_H
#define PKM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKM_ABI_VERSION 3

/* element types (PKM_FP8_E4M3: value tables only) */
enum { PKM_F32 = 0, PKM_BF16 = 1, PKM_FP8_E4M3 = 2 };

/* return codes */
enum {
  PKM_OK = 0,
  PKM_ERR_INVALID = -1,     /* NULL handle / tensor pointer, non-positive dims, odd d_q */
  PKM_ERR_RANGE = -2,       /* B, H, n_keys or k outside the handle's config, k > n_keys */
  PKM_ERR_UNSUPPORTED = -3, /* dtype combination, k above 64 (bf16 lookups with k <= 32
                               score on the tensor cores, those with 32 < k <= 64 and
                               fp32 ones on the CUDA cores, which also bound d_q <= 8192
                               and n_keys <= 4096; a with_backward handle takes k <= 32),
                               n_keys^2 >= 2^31, d_q or d_v layout */
  PKM_ERR_ALIGN = -4,       /* a tensor pointer not 16-byte aligned */
  PKM_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
  PKM_ERR_NOMEM = -6,       /* pkm_create could not allocate its scratch */
  PKM_ERR_TIMEOUT = -7,     /* device: a bounded wait inside a kernel gave up */
  PKM_ERR_BAD_INDEX = -8,   /* device: a row index outside [0, n_keys^2) reached the value read */
  PKM_ERR_NO_STAGING = -9,  /* pkm_forward_host on a handle created without host staging */
  PKM_ERR_OPTION = -10,     /* pkm_set_option: unknown option or value */
  PKM_ERR_NO_BACKWARD = -11 /* pkm_backward on a handle created without with_backward */
};

/* options of pkm_set_option */
enum {
  /* bf16 path: the per-row selection threshold is mean + z * spread of the
     row's first 256 scores.  Any finite z gives exact results (a low z costs
     more log compactions; a high z makes more rows miss their k-th score, and
     their row tiles are selected again without the hint); NaN restores the
     automatic choice. */
  PKM_OPT_HINT_Z = 1,
  /* pkm_forward_host: number of batch slices (1 .. PKM_HOST_MAX_CHUNKS,
     default 3) pipelined so the copy of slice i+1 in and of slice i-1 out
     overlap the computation of slice i; the first and last slices are half
     the size of the others (shorter pipeline fill and drain). */
  PKM_OPT_HOST_CHUNKS = 2,
  /* Tests of failure reporting only (a bit mask, 0 off): with bit 0 the bf16
     lookups of this handle run their selection kernel with its loads held
     back, with bit 1 the bulk-copy value read issues no copy; the kernel's
     bounded waits run out (about 2 s), it records PKM_ERR_TIMEOUT in the
     status word and returns; results of such calls are not meaningful.  The
     GPU context stays usable. */
  PKM_OPT_TEST_STALL = 3,
  /* SMs of the value read (pkm_gather, pkm_forward, pkm_forward_host); 0
     (default): all of them.  Value rows of 512-byte multiples (up to 8 KB)
     stream through shared memory as whole-row bulk copies, one persistent CTA
     per SM; other row widths are read with one CTA per query on every SM
     whatever this option says. */
  PKM_OPT_READ_SMS = 4,
  /* bf16 lookups with k <= 32: the form of the selection kernel's main pass.
     0 (default): automatic (the two-SM form above 128 queries, with one
     epilogue set for half-queries wider than 512, two otherwise); 1: one-SM
     forms (tcgen05 MMAs of 128 query rows per SM); 2: the two-SM form (MMAs of 256 query rows spanning the two
     CTAs of a cluster, each loading half of every subkey slab) with two
     epilogue warp sets on alternate work units; 3: the two-SM form with one
     epilogue warp set.  Results are the same in every form. */
  PKM_OPT_SELECT_FORM = 5
};
#define PKM_HOST_MAX_CHUNKS 16

typedef struct pkm_handle *pkm_t;

/*
 * Fixed shape of a handle.  d_q: query width per head (even; a multiple of 16
 * for bf16).  d_v: value row width (d_v * element size a multiple of 16
 * bytes; a multiple of 16 for PKM_FP8_E4M3).  max_*: the largest B, H,
 * n_keys and k any call will pass (sizes the scratch).  host_staging:
 * nonzero to also allocate device staging for pkm_forward_host (three slots of
 * max_B queries and outputs).  with_backward: nonzero to also allocate what
 * pkm_backward needs (bf16 queries and subkeys with d_q <= 2048, bf16 or
 * fp32 values): scratch for the gradients (about 44 * max_B * max_H * max_k
 * bytes, or 28 * max_B * max_H * max_k + max_n_keys^2 / 32 if larger);
 * max_B * max_H * max_k and max_B * d_v / 4 must stay below 2^31.
 */
typedef struct {
  int d_q, d_v;
  int max_B, max_H, max_n_keys, max_k;
  int q_dtype, key_dtype, value_dtype;
  int host_staging;
  int with_backward;
} pkm_config;

/* Allocate a handle on the current CUDA device.  *out is set only on success. */
int pkm_create(pkm_t *out, const pkm_config *cfg);

/* Free a handle and its scratch.  NULL is a no-op.  Synchronises the device work
   that may still use the scratch (cudaFree semantics). */
void pkm_destroy(pkm_t h);

/*
 * The whole forward pass: scoring, per-half top-k, k^2 merge, softmax and the
 * weighted value read summed over heads.  idx and w may each be NULL, in which
 * case the handle's scratch holds them.  B == 0 is a no-op returning PKM_OK.
 */
int pkm_forward(pkm_t h, const void *q, const void *subkeys, const void *values, int B, int H,
                int n_keys, int k, float *out, int64_t *idx, float *w, void *stream);

/* The lookup alone (scoring through softmax): writes idx and w, both required. */
int pkm_lookup(pkm_t h, const void *q, const void *subkeys, int B, int H, int n_keys, int k,
               int64_t *idx, float *w, void *stream);

/*
 * The flat exact top-k: the search that product keys replace, for measuring
 * what the factorisation saves on the same GPU ("Memory Retrieval
 * Mechanisms: From Soft to Efficient", top-k retrieval and its cost walk-
 * through: score all N keys, O(N d), keep the k best, softmax over them;
 * "Product-Key Memory", "Factorising the key space": a full key is the
 * concatenation of one subkey per half, 2 sqrt(N) subkey comparisons
 * instead of N).
 *
 * pkm_full_keys: keys [H][n_keys^2][d_q] bf16 (caller-owned, device,
 *   H * n_keys^2 * d_q * 2 bytes) from subkeys [H][2][n_keys][d_q/2] bf16:
 *   keys[h][a * n_keys + b] = concat(subkeys[h][0][a], subkeys[h][1][b]).
 * pkm_flat_lookup: per (query, head) every full key scored as one d_q-long
 *   dot product (bf16 inputs, fp32 accumulation, tensor cores), the k best by
 *   (score desc, flat index asc) in idx [B][H][k] int64 and their softmax in
 *   w [B][H][k] fp32, as pkm_lookup returns them.  Needs bf16 queries and
 *   keys and k <= 32; sizes are checked against the handle's configuration
 *   like pkm_lookup's, k <= n_keys included (PKM_ERR_RANGE /
 *   PKM_ERR_UNSUPPORTED).  A bounded wait
 *   that runs out records PKM_ERR_TIMEOUT (pkm_get_status).
 * Both are asynchronous on `stream`; device pointers, 16-byte aligned
 * (PKM_ERR_ALIGN); NULL pointers give PKM_ERR_INVALID; B == 0 is a no-op.
 */
int pkm_full_keys(pkm_t h, const void *subkeys, int H, int n_keys, void *keys, void *stream);
int pkm_flat_lookup(pkm_t h, const void *q, const void *keys, int B, int H, int n_keys, int k,
                    int64_t *idx, float *w, void *stream);

/*
 * The value read alone: out[b,:] = sum_{h,j} w[b,h,j] * values[idx[b,h,j], :]
 * (EmbeddingBag(mode="sum") with per-sample weights, bags of H*k rows).
 * Rows with an index outside [0, n_keys^2) contribute nothing and set
 * PKM_ERR_BAD_INDEX in the status word.
 */
int pkm_gather(pkm_t h, const void *values, int B, int H, int n_keys, int k, const int64_t *idx,
               const float *w, float *out, void *stream);

/*
 * pkm_forward with the per-call tensors in HOST memory: q_host is copied to
 * the handle's staging, the forward runs, and out_host (and idx_host / w_host
 * when not NULL) are copied back; the call synchronises `stream` before it
 * returns.  The batch is cut into slices (PKM_OPT_HOST_CHUNKS) whose copies
 * run on two streams of the handle, overlapping the computation, which stays
 * on `stream`.  subkeys and values stay device pointers (they are parameters,
 * resident on the GPU).  Host buffers should be pinned for full copy speed.
 * Needs a handle created with host_staging != 0.
 */
int pkm_forward_host(pkm_t h, const void *q_host, const void *subkeys, const void *values, int B,
                     int H, int n_keys, int k, float *out_host, int64_t *idx_host, float *w_host,
                     void *stream);

/*
 * pkm_forward_host without the final synchronisation, for callers that keep
 * several batches in flight: the call enqueues the copies and the forward and
 * returns; done_event (a cudaEvent_t, required) is recorded after the last
 * copy back, and out_host / idx_host / w_host are valid once it has
 * completed.  q_host must stay unchanged and the host buffers valid until
 * then.  The handle keeps three staging slots used in turn, so the copies in
 * of one call run while the two calls before it compute and copy out; a
 * fourth call's copies wait (on the device) until the first call's results
 * are copied back.  The batch is one slice unless PKM_OPT_HOST_CHUNKS was set
 * on the handle (the calls in flight beside it already hide the copies).  Calls in flight on one handle
 * share its lookup scratch, so they must be enqueued on the same stream.
 */
int pkm_forward_host_async(pkm_t h, const void *q_host, const void *subkeys, const void *values,
                           int B, int H, int n_keys, int k, float *out_host, int64_t *idx_host,
                           float *w_host, void *stream, void *done_event);

/* Set a tuning option of a handle (PKM_OPT_*).  Affects later calls only. */
int pkm_set_option(pkm_t h, int option, double value);

/* Synchronise `stream` and report in *count how many (query, head) pairs of
   the last bf16 lookup on this handle had a per-half selection threshold hint
   above their k-th score; their row tiles were scored and selected again
   without the hint (exact), in the same call. */
int pkm_get_fallback_count(pkm_t h, void *stream, int *count);

/* Synchronise `stream`, return the device status word (PKM_OK or a device error
   code) and reset it to PKM_OK. */
int pkm_get_status(pkm_t h, void *stream);

/* Host-only argument check of a call against a config (no CUDA calls). */
int pkm_check_args(const pkm_config *cfg, int B, int H, int n_keys, int k);

/* Static description of a return code. */
const char *pkm_strerror(int code);

/* PKM_ABI_VERSION of the library. */
int pkm_abi_version(void);

/*
 * 1 if every one of the `count` pointers is device memory of the current
 * device, else 0 (also on any CUDA error, or with no device).  The lookup's
 * one-SM selection form loads tiles once for two CTAs of a cluster (TMA
 * multicast) only when its operands pass this test;
 * other operands (host, managed or another GPU's memory) take the one-CTA
 * forms.  Host-side only; nothing is launched.
 */
int pkm_multicast_ok(const void *const *ptrs, int count);

/*
 * No counterpart on the pages: a library-level addition for callers that
 * cannot allocate device memory when they run a lookup (a serving process
 * whose GPU memory is budgeted at start-up, a host framework that owns every
 * device allocation through its own pool, a hot loop where cudaMalloc or
 * cudaFree would synchronise the device).  pkm_create allocates, so this
 * entry point takes no handle.
 *
 * pkm_lookup_static: the lookup alone (scoring through softmax) for bf16
 * queries and subkeys and k <= 32 (the tensor-core path; a larger k returns
 * PKM_ERR_UNSUPPORTED), as pkm_lookup on a bf16 handle with d_q given here:
 * idx and w [B, H, k] are written on `stream`.  It allocates nothing: its
 * scratch (a status word, the retry pass's counts, unit flags and unit list,
 * and the per-half candidate lists, for at most PKM_STATIC_MAX_PAIRS pairs)
 * is one fixed array of about 25 MiB in the library's device memory, which
 * every GPU that loads the library holds until the process exits.
 *   - B * H above PKM_STATIC_MAX_PAIRS returns PKM_ERR_RANGE; other argument
 *     errors are as for pkm_lookup.
 *   - status: if not NULL, a device int that receives the call's device
 *     status (PKM_OK or PKM_ERR_TIMEOUT) on `stream`.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it with the device's current
 *     context; make that first call before any stream capture.  A call in a
 *     new context of the device (after cudaDeviceReset) looks it up again.
 *   - All calls share the one array, and each call clears what must start at
 *     zero.  Calls whose work overlaps on the GPU (other streams, other host
 *     threads) race on it: serialise them.
 */
#define PKM_STATIC_MAX_PAIRS (1 << 16)
int pkm_lookup_static(const void *q, const void *subkeys, int B, int H, int d_q, int n_keys, int k,
                      int64_t *idx, float *w, int *status, void *stream);

/*
 * Backward pass of pkm_forward for the selection it made (the top-k choices
 * are not differentiated: gradient flows through the selected scores, the
 * softmax and the weighted read, as autograd does through the page's code
 * listing).  Inputs: the forward's q, subkeys and values (bf16 queries and
 * subkeys; bf16 or fp32 values), its idx and w, and dout [B, d_v] fp32 (the
 * gradient of out).  Outputs, fp32 device arrays:
 *   dq        [B, H, d_q]              overwritten;
 *   dsubkeys  [H, 2, n_keys, d_q/2]    added to (zero it first, or accumulate);
 *   dvalues   [n_keys^2, d_v]          added to (only the selected rows change).
 * With dw = dout . V[idx] and ds = w * (dw - sum(w * dw)): dvalues[idx] +=
 * w * dout; dq and dsubkeys take ds through each winner's two subkeys (the
 * winners sharing a subkey summed first), gathering only the winning
 * subkeys' rows and the queries' rows; all of it fp32 (the order in which a
 * subkey's contributions are added to dsubkeys varies from call to call).
 * Requires a handle created with with_backward (else PKM_ERR_NO_BACKWARD).
 * Enqueued on `stream`; an index outside [0, n_keys^2) sets
 * PKM_ERR_BAD_INDEX in the status word and contributes nothing.
 * pkm_backward = pkm_backward_read then pkm_backward_scores, with dw kept in
 * the handle's scratch.
 */
int pkm_backward(pkm_t h, const void *q, const void *subkeys, const void *values, int B, int H,
                 int n_keys, int k, const int64_t *idx, const float *w, const float *dout,
                 float *dq, float *dsubkeys, float *dvalues, void *stream);

/*
 * The read's part of the backward pass: dw [B, H, k] fp32 = dout[b] . V[idx]
 * (overwritten; the gradient of the softmax weights) and dvalues[idx] +=
 * w * dout[b].  The selections are grouped by value row first, so each
 * selected row of values and dvalues is read (and written) once; a row's
 * additions are fp32 and their order may vary between runs.  Requires
 * with_backward (its scratch).
 */
int pkm_backward_read(pkm_t h, const void *values, int B, int H, int n_keys, int k,
                      const int64_t *idx, const float *w, const float *dout, float *dw,
                      float *dvalues, void *stream);

/*
 * pkm_backward with the value-table gradient in sparse form, the way a
 * sparse optimiser consumes it (EmbeddingBag with sparse gradients): the
 * distinct selected rows, ascending, in rows[0 .. *n_rows) and each row's
 * gradient sum(w * dout) over its selections in grad_rows[i, :] (overwritten;
 * fp32, d_v wide).  n_rows is a device int written by the call; rows and
 * grad_rows must hold B * H * k entries (the case of no repeated row).  The
 * dense dvalues table is neither read nor written.  Same requirements and
 * status reporting as pkm_backward; an index outside [0, n_keys^2) is not
 * listed.
 */
int pkm_backward_sparse(pkm_t h, const void *q, const void *subkeys, const void *values, int B,
                        int H, int n_keys, int k, const int64_t *idx, const float *w,
                        const float *dout, float *dq, float *dsubkeys, int64_t *rows,
                        float *grad_rows, int *n_rows, void *stream);

/* The read's part of pkm_backward_sparse: dw and the sparse value-table gradient. */
int pkm_backward_read_sparse(pkm_t h, const void *values, int B, int H, int n_keys, int k,
                             const int64_t *idx, const float *w, const float *dout, float *dw,
                             int64_t *rows, float *grad_rows, int *n_rows, void *stream);

/*
 * The scores' part of the backward pass, from w and dw: dq overwritten,
 * dsubkeys added to, as in pkm_backward.  Requires with_backward.
 */
int pkm_backward_scores(pkm_t h, const void *q, const void *subkeys, int B, int H, int n_keys,
                        int k, const int64_t *idx, const float *w, const float *dw, float *dq,
                        float *dsubkeys, void *stream);

/*
 * Quantise a value table to the PKM_FP8_E4M3 layout above.  values: [N, d_v]
 * of value_dtype (PKM_F32 or PKM_BF16), device memory.  out: device buffer of
 * N * d_v + 4 * N bytes, 16-byte aligned, overwritten (codes, then scales).
 * Per row r, with amax = max_c |V[r, c]| (a recipe of this library; the page
 * fixes none): scale[r] = max(amax / 448, FLT_MIN) in fp32, and code[r, c] =
 * the e4m3 value nearest to V[r, c] / scale[r] (fp32 division, ties to the
 * even mantissa, saturated to +-448).  Enqueued on `stream`.  Errors:
 * PKM_ERR_INVALID (NULL pointer, N < 1, d_v < 1), PKM_ERR_UNSUPPORTED
 * (value_dtype, d_v not a multiple of 16), PKM_ERR_ALIGN, PKM_ERR_CUDA.
 */
int pkm_quantize_values_fp8(const void *values, int value_dtype, int64_t N, int d_v, void *out,
                            void *stream);

/*
 * The query network ahead of the lookup (Product-Key Memory, code listing:
 * q = BatchNorm1d(Linear(dim, dim, bias=False)(x)); with H heads of width d_q
 * the Linear maps dim -> F = H * d_q features and q is the [B, H, d_q] query
 * of pkm_forward).  The listing does not fix the BatchNorm's mode; both are
 * provided: the inference form with running statistics (pkm_bn_fold +
 * pkm_query_net) and the training form with the batch's own statistics
 * (pkm_query_net_batch; Product-Key Memory, "Keeping the memory in use":
 * the BatchNorm over the queries spreads them over the key space).
 *
 * pkm_bn_fold: scale[f] = gamma[f] / sqrt(var[f] + eps), shift[f] = beta[f] -
 * mean[f] * scale[f], fp32, f < F (device arrays; enqueued on `stream`).
 *
 * pkm_query_net: q[b, f] = bf16_rn((sum_t x[b, t] * W[f, t]) * scale[f] +
 * shift[f]), x [B, dim] bf16, W [F, dim] bf16 (nn.Linear's weight layout),
 * scale / shift [F] fp32, q [B, F] bf16; tensor cores, fp32 accumulation.
 * dim a multiple of 16, F a multiple of 32, pointers 16-byte aligned.
 * status: NULL, or a device int that receives PKM_ERR_TIMEOUT if a bounded
 * wait inside the kernel gives up (it is not cleared).  Errors:
 * PKM_ERR_INVALID (NULL pointer, B < 0, dim < 1, F < 1), PKM_ERR_UNSUPPORTED
 * (dim or F layout), PKM_ERR_ALIGN, PKM_ERR_CUDA.  B == 0 is a no-op.
 */
int pkm_bn_fold(const float *gamma, const float *beta, const float *running_mean,
                const float *running_var, float eps, int F, float *scale, float *shift,
                void *stream);
int pkm_query_net(const void *x, const void *weight, int B, int dim, int F, const float *scale,
                  const float *shift, void *q, int *status, void *stream);

/*
 * pkm_query_net_batch: the training form.  z = x W^T (bf16 in, fp32
 * accumulation on the tensor cores); per feature f the batch mean mu[f] =
 * sum_b z[b, f] / B and the biased variance var[f] = sum_b (z[b, f] -
 * mu[f])^2 / B; q[b, f] = bf16_rn(z[b, f] * s[f] + t[f]) with s[f] =
 * gamma[f] / sqrt(var[f] + eps) and t[f] = beta[f] - mu[f] * s[f].  The
 * statistics come from 32-row blocks (each block's mean and sum of squared
 * deviations, fp32) joined in fp32 by the law of total variance; z is computed twice (statistics, then
 * q) and never stored.  batch_mean / batch_var: NULL, or device [F] fp32
 * receiving mu and var (a running-statistics update would take the unbiased
 * var * B / (B - 1)).  workspace: device scratch of
 * pkm_query_net_batch_workspace_bytes(B, F) bytes (about 8 * F * B / 32),
 * caller-owned, 16-byte aligned.  Shapes, alignment, status and errors as
 * pkm_query_net's, and PKM_ERR_INVALID for eps < 0 or NaN, PKM_ERR_RANGE
 * when (B + 31) / 32 * F exceeds 2^31 - 1.  B == 1 gives var = 0 (q = beta).
 */
size_t pkm_query_net_batch_workspace_bytes(int B, int F);
int pkm_query_net_batch(const void *x, const void *weight, int B, int dim, int F,
                        const float *gamma, const float *beta, float eps, void *workspace, void *q,
                        float *batch_mean, float *batch_var, int *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKM_H */
