// pkm_lookup_static: the bf16 lookup without a handle and without any
// device allocation.
//
// Some callers cannot allocate device memory at the point where they run a
// lookup: a serving process whose GPU memory budget is fixed when it starts,
// a host framework that owns every device allocation through its own pool,
// or a latency-critical loop where cudaMalloc / cudaFree would synchronise
// the device.  pkm_create allocates the handle's scratch, so those callers
// use this entry point instead.  Its scratch (a status word, the retry
// pass's counts, per-unit flags and unit list, and the per-half lists passed
// from the selection kernel to the merge kernel) is one fixed-size array in
// the library's device memory, present on every GPU that loads the library
// until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkm_internal.cuh"

namespace {

// [0] device status word, [1..2] retry counts and from [3] the per-unit
// flags, then the retry pass's unit list and the per-half lists of at most
// PKM_STATIC_MAX_PAIRS pairs.  Work units number
// ceil(B / 128) * H * 2 <= 2 * (B*H / 128 + H).
constexpr size_t kMaxUnits = 2 * ((size_t)PKM_STATIC_MAX_PAIRS / 128 + PKM_STATIC_MAX_PAIRS);
constexpr size_t kHeader = (3 + kMaxUnits) * 4 / 256 * 256 + 256;
constexpr size_t kFbBytes = kMaxUnits * 4;
constexpr size_t kListSlots = (size_t)PKM_STATIC_MAX_PAIRS * 2 * pkm::kListMaxSlots;
constexpr size_t kStaticBytes = kHeader + kFbBytes + kListSlots * 4 + kListSlots * 2;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_addr[kMaxDevices] = {};  // device address of g_static_scratch, per device
CUcontext g_scratch_ctx[kMaxDevices] = {};        // the context the address was found in

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The device's current context (cuCtxGetCurrent through the runtime's
// driver entry point), or NULL when it cannot be found.
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of the scratch array on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress); later calls in the same
// context reuse it, and a new context of the device (after a device reset,
// which reloads the library's module) looks it up again.
int scratch_on_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  // (a thread with no current context yet reads NULL here; the symbol
  // lookup makes the device's primary context current, and it is read again)
  const CUcontext ctx = current_context();
  if (!g_scratch_addr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return PKM_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_addr[dev];
  return PKM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int pkm_lookup_static(const void* q, const void* subkeys, int B, int H, int d_q,
                                 int n_keys, int k, int64_t* idx, float* w, int* status,
                                 void* stream) {
  if (B < 0 || H < 1 || d_q < 2 || (d_q & 1) || n_keys < 1 || k < 1) return PKM_ERR_INVALID;
  if (k > n_keys) return PKM_ERR_RANGE;
  if (d_q % 16 || k > pkm::kTcMaxK || (int64_t)n_keys * n_keys > INT32_MAX)
    return PKM_ERR_UNSUPPORTED;
  if ((int64_t)B * H > PKM_STATIC_MAX_PAIRS) return PKM_ERR_RANGE;
  if (B == 0) return PKM_OK;
  if (!q || !subkeys || !idx || !w) return PKM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(subkeys) || !aligned16(idx) || !aligned16(w))
    return PKM_ERR_ALIGN;
  unsigned char* base = nullptr;
  int rc = scratch_on_current_device(&base);
  if (rc) return rc;
  int* scratch = reinterpret_cast<int*>(base);  // status, retry counts, unit flags
  int* unit_list = reinterpret_cast<int*>(base + kHeader);
  float* list_v = reinterpret_cast<float*>(base + kHeader + kFbBytes);
  unsigned short* list_c =
      reinterpret_cast<unsigned short*>(base + kHeader + kFbBytes + kListSlots * 4);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word starts clear on every call (the retry bookkeeping is
  // cleared by the lookup launch itself)
  if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess) return PKM_ERR_CUDA;
  cudaError_t e = pkm::launch_lookup_tc(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(subkeys), B, H, d_q, n_keys,
      k, pkm::default_hint_z(n_keys, k), idx, w, scratch, {scratch + 1, scratch + 3, unit_list},
      list_v, list_c, s);
  if (e != cudaSuccess) return PKM_ERR_CUDA;
  if (status &&
      cudaMemcpyAsync(status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return PKM_ERR_CUDA;
  return PKM_OK;
}
