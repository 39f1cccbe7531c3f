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
// the library's own device memory instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits. Host code
// cannot pass the array's name to a kernel: on the host that name is only a
// stand-in symbol, not a device address. The device address is looked up once
// per device with cudaGetSymbolAddress, on the first call made while that
// device is current, and cached.
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
gdn_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return GDN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return GDN_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status_t gdn_delta_rule_prefill_chunked_noalloc(
    const void* q, const void* k, int64_t qk_stride, const void* v, int64_t v_stride,
    const float* a, const float* b, const int32_t* cu_seqlens, int32_t N, int32_t T, float* S,
    const uint8_t* has_initial_state, void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
    int32_t chunk, int32_t qk_l2norm, void* stream) {
  // Argument checks and the size limit come first, so a rejected call touches
  // no CUDA state at all.
  if (T < 0 || N < 0) return GDN_ERR_INVALID_ARG;
  if (chunk != 64) return GDN_ERR_UNSUPPORTED;
  if (T == 0 || N == 0) return GDN_OK;
  const size_t need = gdn_delta_rule_prefill_workspace_size(T, N, Hv, dk, dv, chunk);
  if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  gdn_status_t rc = scratch_address(&scratch);
  if (rc != GDN_OK) return rc;
  return gdn_delta_rule_prefill_chunked(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                                        has_initial_state, o, Hk, Hv, dk, dv, chunk, qk_l2norm,
                                        scratch, kNoAllocScratchBytes, stream);
}
