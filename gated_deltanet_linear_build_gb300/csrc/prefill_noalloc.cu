// Chunked prefill for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain scratch memory: code
// running inside a host framework that owns every device allocation (a custom
// allocator or a memory pool it alone may call), plugins loaded into another
// process's CUDA context, or code paths that are not allowed to call
// cudaMalloc at all (for instance while the host is in a latency-critical
// section where an allocation could synchronise the device). For them this
// file provides gdn_delta_rule_prefill_chunked_noalloc: the same computation as
// gdn_delta_rule_prefill_chunked, with the scratch taken from a fixed array in
// the library's own device memory instead of a caller-provided workspace, and
// gdn_delta_rule_prefill_chunked_noalloc_status, which copies that array's two
// device-side status words to the caller.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits. Host code
// cannot pass the array's name to a kernel: on the host that name is only a
// stand-in symbol, not a device address. The device address belongs to the
// module as loaded into one CUDA context, so it is looked up with
// cudaGetSymbolAddress on the first call made in each context (the current
// device's current context), and cached under that context's unique id; a
// context created later (another context on the same device, or the primary
// context again after cudaDeviceReset) gets its own lookup.
#include <mutex>
#include <unordered_map>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
std::unordered_map<unsigned long long, void*> g_scratch_by_ctx;

// The driver's cuCtxGetCurrent and cuCtxGetId, reached through the runtime
// (the library does not link the driver library itself). Declared with plain
// types: a context handle is an opaque pointer, CUresult an int.
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);

bool context_api(CtxGetCurrentFn* get_current, CtxGetIdFn* get_id) {
  static CtxGetCurrentFn f_current = nullptr;
  static CtxGetIdFn f_id = nullptr;
  static const bool ok = [] {
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
    cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                         &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2) {
      cudaGetLastError();
      return false;
    }
    f_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    f_id = reinterpret_cast<CtxGetIdFn>(f2);
    return true;
  }();
  *get_current = f_current;
  *get_id = f_id;
  return ok;
}

// Device address of the scratch array in the calling thread's current context
// (looked up once per context). With no context current yet, the runtime's
// first call (the lookup itself) binds the current device's primary context
// to the thread, as any runtime call would.
gdn_status_t scratch_address(void** out) {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
  if (!context_api(&get_current, &get_id)) {
    set_cuda_error(cudaErrorSymbolNotFound);
    return GDN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  void* ctx = nullptr;
  void* fresh = nullptr;
  if (get_current(&ctx) != 0 || ctx == nullptr) {
    cudaError_t e = cudaGetSymbolAddress(&fresh, g_prefill_scratch);
    if (e != cudaSuccess || fresh == nullptr) {
      set_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return GDN_ERR_CUDA;
    }
    if (get_current(&ctx) != 0 || ctx == nullptr) {
      set_cuda_error(cudaErrorContextIsDestroyed);
      return GDN_ERR_CUDA;
    }
  }
  unsigned long long ctx_id = 0;
  if (get_id(ctx, &ctx_id) != 0) {
    set_cuda_error(cudaErrorContextIsDestroyed);
    return GDN_ERR_CUDA;
  }
  auto it = g_scratch_by_ctx.find(ctx_id);
  if (it == g_scratch_by_ctx.end()) {
    if (fresh == nullptr) {
      cudaError_t e = cudaGetSymbolAddress(&fresh, g_prefill_scratch);
      if (e != cudaSuccess || fresh == nullptr) {
        set_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        return GDN_ERR_CUDA;
      }
    }
    it = g_scratch_by_ctx.emplace(ctx_id, fresh).first;
  }
  *out = it->second;
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status_t gdn_delta_rule_prefill_chunked_noalloc(
    const void* q, const void* k, int64_t qk_stride, const void* v, int64_t v_stride,
    const float* a, const float* b, const int32_t* cu_seqlens, int32_t N, int32_t T, float* S,
    const uint8_t* has_initial_state, void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
    int32_t chunk, int32_t flags, void* stream) {
  // Every argument check and the size limit come first, so a rejected call
  // touches no CUDA state at all (no context set-up, no symbol lookup).
  // A plan (GDN_FLAG_PLANNED) would have to sit in the library's array,
  // which the caller cannot address: this variant always builds its own.
  if (flags & GDN_FLAG_PLANNED) return GDN_ERR_INVALID_ARG;
  bool nothing = false;
  gdn_status_t rc = check_prefill_args(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                                       o, Hk, Hv, dk, dv, chunk, flags, &nothing);
  if (rc != GDN_OK || nothing) return rc;
  const size_t need = gdn_delta_rule_prefill_workspace_size(T, N, Hv, dk, dv, chunk);
  if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != GDN_OK) return rc;
  return gdn_delta_rule_prefill_chunked(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                                        has_initial_state, o, Hk, Hv, dk, dv, chunk, flags,
                                        scratch, kNoAllocScratchBytes, stream);
}

extern "C" gdn_status_t gdn_delta_rule_prefill_chunked_noalloc_status(int32_t* status,
                                                                     void* stream) {
  if (!status) return GDN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  gdn_status_t rc = scratch_address(&scratch);
  if (rc != GDN_OK) return rc;
  // Words 1 and 2 of the workspace header (byte offsets 4 and 8).
  cudaError_t e = cudaMemcpyAsync(status, static_cast<unsigned char*>(scratch) + 4,
                                  2 * sizeof(int32_t), cudaMemcpyDefault,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_cuda_error(e);
    return GDN_ERR_CUDA;
  }
  return GDN_OK;
}
