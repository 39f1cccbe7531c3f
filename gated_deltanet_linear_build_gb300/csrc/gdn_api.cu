// C ABI of the GDN hot path: host-side argument validation, then the kernel
// launchers. Nothing here allocates device memory or synchronises.
#include <cstring>
#include <string>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {
// Text of the calling thread's most recent CUDA failure (like errno: a pointer
// returned to one thread is never invalidated by another thread's failure).
thread_local std::string t_err_text;
constexpr int kConvTaps = 4;

bool head_dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
}  // namespace

void set_cuda_error(cudaError_t e) {
  t_err_text = cudaGetErrorName(e);
  t_err_text += ": ";
  t_err_text += cudaGetErrorString(e);
}
}  // namespace gdn

namespace gdn {
namespace {
// One CTA waits, with the library's bounded wait, for a phase of a freshly
// initialised mbarrier that nothing completes.
__global__ void bounded_wait_selftest_kernel(int32_t* status, long long max_cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
  __syncthreads();
  const bool completed = tc::mbar_wait(&bar, 0, max_cycles);
  if (threadIdx.x == 0) {
    *status = completed ? GDN_OK : GDN_ERR_TIMEOUT;
    if (!completed) record_device_status(GDN_ERR_TIMEOUT);
  }
}
}  // namespace

GDN_DEFINE_STATUS_GATHER(gather_status_api)
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status_t gdn_selftest_bounded_wait(int32_t* device_status, int64_t max_cycles,
                                       void* stream) {
  if (!device_status || max_cycles < 1 || max_cycles > 4000000000LL) return GDN_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      device_status, (long long)max_cycles);
  return check_launch();
}

gdn_status_t gdn_device_status(int32_t* status, int32_t clear, void* stream) {
  if (!status || (clear != 0 && clear != 1)) return GDN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(status) & 3u) != 0) return GDN_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gdn_status_t rc;
  if ((rc = gather_status_api(status, clear, 1, st)) != GDN_OK) return rc;
  if ((rc = gather_status_conv(status, clear, 0, st)) != GDN_OK) return rc;
  if ((rc = gather_status_decode(status, clear, 0, st)) != GDN_OK) return rc;
  return gather_status_prefill_tc(status, clear, 0, st);
}

const char* gdn_status_string(gdn_status_t s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: shape or option not implemented";
    case GDN_ERR_ALIGNMENT: return "GDN_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace or capacity too small";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA call failed";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: bounded device wait gave up";
  }
  return "GDN: unknown status";
}

const char* gdn_last_cuda_error_string(void) { return t_err_text.c_str(); }

gdn_status_t gdn_build_conv_chunks(const int32_t* cu_seqlens, int32_t num_seqs,
                                   int32_t chunk_tokens, gdn_conv_chunk_t* chunks,
                                   int32_t capacity, int32_t* num_chunks,
                                   int32_t* device_status, void* stream) {
  if (!cu_seqlens || !num_chunks || num_seqs < 0 || capacity < 0) return GDN_ERR_INVALID_ARG;
  if (chunk_tokens < kConvTaps - 1) return GDN_ERR_INVALID_ARG;
  if (capacity > 0 && !chunks) return GDN_ERR_INVALID_ARG;
  if (chunks && !aligned16(chunks)) return GDN_ERR_ALIGNMENT;
  return launch_build_chunks(cu_seqlens, num_seqs, chunk_tokens, chunks, capacity, num_chunks,
                             device_status, static_cast<cudaStream_t>(stream));
}

static gdn_status_t check_conv_common(const void* x, int64_t x_stride, const void* w,
                                      const void* bias, void* conv_state, int32_t C, int32_t K,
                                      int32_t silu, void* y) {
  if (!x || !w || !conv_state || !y) return GDN_ERR_INVALID_ARG;
  if (C <= 0 || x_stride < C || (silu != 0 && silu != 1)) return GDN_ERR_INVALID_ARG;
  if (K != kConvTaps) return GDN_ERR_UNSUPPORTED;
  if (C % 8 != 0) return GDN_ERR_UNSUPPORTED;
  if (x_stride % 8 != 0) return GDN_ERR_ALIGNMENT;
  if (!aligned16(x) || !aligned16(w) || !aligned16(conv_state) || !aligned16(y) ||
      (bias && !aligned16(bias)))
    return GDN_ERR_ALIGNMENT;
  return GDN_OK;
}

// The state-slot argument pair of the *_slots entry points: a device array of
// N slot numbers and the number of slots in the state cache.
static gdn_status_t make_slots(const int32_t* state_indices, int32_t num_slots,
                               StateSlots* out) {
  if (!state_indices || num_slots < 0) return GDN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(state_indices) & 3u) != 0) return GDN_ERR_ALIGNMENT;
  out->idx = state_indices;
  out->count = num_slots;
  return GDN_OK;
}

static gdn_status_t conv_fwd_impl(const void* x, int64_t x_stride, const void* w,
                                  const void* bias, void* conv_state,
                                  const uint8_t* has_initial_state, const int32_t* cu_seqlens,
                                  const gdn_conv_chunk_t* chunks, const int32_t* num_chunks,
                                  int32_t max_chunks, int32_t T, int32_t C, int32_t K, int32_t N,
                                  int32_t silu, void* y, void* stream, StateSlots slots) {
  if (T < 0 || N < 0) return GDN_ERR_INVALID_ARG;
  if ((chunks == nullptr) != (num_chunks == nullptr)) return GDN_ERR_INVALID_ARG;
  if (chunks && max_chunks < 0) return GDN_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return GDN_OK;
  if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
  gdn_status_t rc = check_conv_common(x, x_stride, w, bias, conv_state, C, K, silu, y);
  if (rc != GDN_OK) return rc;
  if (chunks && !aligned16(chunks)) return GDN_ERR_ALIGNMENT;
  const int32_t units = chunks ? max_chunks : N;
  return launch_conv_fwd(x, x_stride, w, bias, conv_state, has_initial_state, cu_seqlens, chunks,
                         num_chunks, units, T, C, N, silu, y, static_cast<cudaStream_t>(stream),
                         slots);
}

gdn_status_t gdn_causal_conv1d_fwd(const void* x, int64_t x_stride, const void* w,
                                   const void* bias, void* conv_state,
                                   const uint8_t* has_initial_state,
                                   const int32_t* cu_seqlens,
                                   const gdn_conv_chunk_t* chunks,
                                   const int32_t* num_chunks, int32_t max_chunks,
                                   int32_t T, int32_t C, int32_t K, int32_t N,
                                   int32_t silu, void* y, void* stream) {
  return conv_fwd_impl(x, x_stride, w, bias, conv_state, has_initial_state, cu_seqlens, chunks,
                       num_chunks, max_chunks, T, C, K, N, silu, y, stream, StateSlots{});
}

gdn_status_t gdn_causal_conv1d_fwd_slots(const void* x, int64_t x_stride, const void* w,
                                         const void* bias, void* conv_state,
                                         const uint8_t* has_initial_state,
                                         const int32_t* cu_seqlens,
                                         const gdn_conv_chunk_t* chunks,
                                         const int32_t* num_chunks, int32_t max_chunks,
                                         int32_t T, int32_t C, int32_t K, int32_t N,
                                         int32_t silu, void* y,
                                         const int32_t* state_indices, int32_t num_slots,
                                         void* stream) {
  StateSlots slots;
  gdn_status_t rc = make_slots(state_indices, num_slots, &slots);
  if (rc != GDN_OK) return rc;
  return conv_fwd_impl(x, x_stride, w, bias, conv_state, has_initial_state, cu_seqlens, chunks,
                       num_chunks, max_chunks, T, C, K, N, silu, y, stream, slots);
}

static gdn_status_t conv_update_impl(const void* x, int64_t x_stride, const void* w,
                                     const void* bias, void* conv_state, int32_t N, int32_t C,
                                     int32_t K, int32_t silu, void* y, void* stream,
                                     StateSlots slots) {
  if (N < 0) return GDN_ERR_INVALID_ARG;
  if (N == 0) return GDN_OK;
  gdn_status_t rc = check_conv_common(x, x_stride, w, bias, conv_state, C, K, silu, y);
  if (rc != GDN_OK) return rc;
  return launch_conv_update(x, x_stride, w, bias, conv_state, N, C, silu, y,
                            static_cast<cudaStream_t>(stream), slots);
}

gdn_status_t gdn_causal_conv1d_update(const void* x, int64_t x_stride, const void* w,
                                      const void* bias, void* conv_state, int32_t N,
                                      int32_t C, int32_t K, int32_t silu, void* y,
                                      void* stream) {
  return conv_update_impl(x, x_stride, w, bias, conv_state, N, C, K, silu, y, stream,
                          StateSlots{});
}

gdn_status_t gdn_causal_conv1d_update_slots(const void* x, int64_t x_stride, const void* w,
                                            const void* bias, void* conv_state, int32_t N,
                                            int32_t C, int32_t K, int32_t silu, void* y,
                                            const int32_t* state_indices, int32_t num_slots,
                                            void* stream) {
  StateSlots slots;
  gdn_status_t rc = make_slots(state_indices, num_slots, &slots);
  if (rc != GDN_OK) return rc;
  return conv_update_impl(x, x_stride, w, bias, conv_state, N, C, K, silu, y, stream, slots);
}

static gdn_status_t check_delta_common(const void* q, const void* k, int64_t qk_stride,
                                       const void* v, int64_t v_stride, const float* a,
                                       const float* b, const float* S, const void* o,
                                       int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                       int32_t flags,
                                       int32_t allowed = GDN_FLAG_QK_L2NORM | GDN_FLAG_GATE_LOGITS) {
  if (!q || !k || !v || !a || !b || !S || !o) return GDN_ERR_INVALID_ARG;
  if (Hk <= 0 || Hv <= 0 || (flags & ~allowed) != 0) return GDN_ERR_INVALID_ARG;
  if (Hv % Hk != 0) return GDN_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDN_ERR_UNSUPPORTED;
  if (qk_stride < (int64_t)Hk * dk || v_stride < (int64_t)Hv * dv) return GDN_ERR_INVALID_ARG;
  if (qk_stride % 8 != 0 || v_stride % 8 != 0) return GDN_ERR_ALIGNMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S) || !aligned16(o))
    return GDN_ERR_ALIGNMENT;
  return GDN_OK;
}

static gdn_status_t decode_impl(const void* q, const void* k, int64_t qk_stride, const void* v,
                                int64_t v_stride, const float* a, const float* b, float* S,
                                void* o, int32_t N, int32_t Hk, int32_t Hv, int32_t dk,
                                int32_t dv, int32_t flags, void* stream, StateSlots slots) {
  if (N < 0) return GDN_ERR_INVALID_ARG;
  if (N == 0) return GDN_OK;
  gdn_status_t rc = check_delta_common(q, k, qk_stride, v, v_stride, a, b, S, o, Hk, Hv, dk, dv,
                                       flags);
  if (rc != GDN_OK) return rc;
  if ((int64_t)N * Hv > 0x7fffffff) return GDN_ERR_UNSUPPORTED;
  return launch_delta_decode(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, dk, dv,
                             flags, static_cast<cudaStream_t>(stream), slots);
}

gdn_status_t gdn_delta_rule_decode(const void* q, const void* k, int64_t qk_stride,
                                   const void* v, int64_t v_stride, const float* a,
                                   const float* b, float* S, void* o, int32_t N,
                                   int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                   int32_t flags, void* stream) {
  return decode_impl(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, dk, dv, flags,
                     stream, StateSlots{});
}

gdn_status_t gdn_delta_rule_decode_slots(const void* q, const void* k, int64_t qk_stride,
                                         const void* v, int64_t v_stride, const float* a,
                                         const float* b, float* S, void* o, int32_t N,
                                         int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                         int32_t flags, const int32_t* state_indices,
                                         int32_t num_slots, void* stream) {
  StateSlots slots;
  gdn_status_t rc = make_slots(state_indices, num_slots, &slots);
  if (rc != GDN_OK) return rc;
  return decode_impl(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, dk, dv, flags,
                     stream, slots);
}

gdn_status_t gdn_decode_step_fused(const void* x, int64_t x_stride, const void* w,
                                   const void* bias, const void* conv_state_in,
                                   void* conv_state_out, const float* a, const float* b,
                                   float* S, void* o, int32_t N, int32_t Hk, int32_t Hv,
                                   int32_t dk, int32_t dv, int32_t K, int32_t silu,
                                   int32_t flags, void* stream) {
  if (N < 0) return GDN_ERR_INVALID_ARG;
  if (N == 0) return GDN_OK;
  if (!x || !w || !conv_state_in || !conv_state_out || !a || !b || !S || !o)
    return GDN_ERR_INVALID_ARG;
  if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0) return GDN_ERR_INVALID_ARG;
  if ((silu != 0 && silu != 1) || (flags & ~(GDN_FLAG_QK_L2NORM | GDN_FLAG_GATE_LOGITS)) != 0) return GDN_ERR_INVALID_ARG;
  if (K != kConvTaps) return GDN_ERR_UNSUPPORTED;
  if (dk != 128 || dv != 128) return GDN_ERR_UNSUPPORTED;
  const int64_t C = 2 * (int64_t)Hk * dk + (int64_t)Hv * dv;
  if (C > 0x7fffffff || (int64_t)N * Hv * 2 > 0x7fffffff) return GDN_ERR_UNSUPPORTED;
  if (x_stride < C) return GDN_ERR_INVALID_ARG;
  if (x_stride % 8 != 0) return GDN_ERR_ALIGNMENT;
  if (!aligned16(x) || !aligned16(w) || (bias && !aligned16(bias)) || !aligned16(conv_state_in) ||
      !aligned16(conv_state_out) || !aligned16(S) || !aligned16(o))
    return GDN_ERR_ALIGNMENT;
  const uintptr_t si = reinterpret_cast<uintptr_t>(conv_state_in);
  const uintptr_t so = reinterpret_cast<uintptr_t>(conv_state_out);
  const uintptr_t sb = (uintptr_t)N * (uintptr_t)C * 3u * 2u;
  if (si < so + sb && so < si + sb) return GDN_ERR_INVALID_ARG;   // the states overlap
  return launch_decode_fused(x, x_stride, w, bias, conv_state_in, conv_state_out, a, b, S, o, N,
                             Hk, Hv, silu, flags, static_cast<cudaStream_t>(stream));
}

size_t gdn_delta_rule_prefill_workspace_size(int32_t T, int32_t N, int32_t Hv, int32_t dk,
                                             int32_t dv, int32_t chunk) {
  return prefill_workspace_bytes(T, N, Hv, dk, dv, chunk);
}

}  // extern "C"

namespace gdn {
gdn_status_t check_prefill_args(const void* q, const void* k, int64_t qk_stride, const void* v,
                                int64_t v_stride, const float* a, const float* b,
                                const int32_t* cu_seqlens, int32_t N, int32_t T, const float* S,
                                const void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                int32_t chunk, int32_t flags, bool* nothing_to_do) {
  *nothing_to_do = false;
  if (T < 0 || N < 0) return GDN_ERR_INVALID_ARG;
  if (chunk != 64) return GDN_ERR_UNSUPPORTED;
  if (T == 0 || N == 0) {
    *nothing_to_do = true;
    return GDN_OK;
  }
  if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
  gdn_status_t rc = check_delta_common(q, k, qk_stride, v, v_stride, a, b, S, o, Hk, Hv, dk, dv,
                                       flags,
                                       GDN_FLAG_QK_L2NORM | GDN_FLAG_GATE_LOGITS | GDN_FLAG_PLANNED);
  if (rc != GDN_OK) return rc;
  if (dk != dv) return GDN_ERR_UNSUPPORTED;
  if ((int64_t)N * Hv > 0x7fffffff) return GDN_ERR_UNSUPPORTED;   // one CTA per (sequence, head)
  return GDN_OK;
}
}  // namespace gdn

extern "C" {

static gdn_status_t prefill_impl(const void* q, const void* k, int64_t qk_stride,
                                 const void* v, int64_t v_stride, const float* a, const float* b,
                                 const int32_t* cu_seqlens, int32_t N, int32_t T, float* S,
                                 const uint8_t* has_initial_state, void* o, int32_t Hk,
                                 int32_t Hv, int32_t dk, int32_t dv, int32_t chunk,
                                 int32_t flags, void* workspace, size_t workspace_bytes,
                                 void* stream, StateSlots slots) {
  bool nothing = false;
  gdn_status_t rc = check_prefill_args(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                                       o, Hk, Hv, dk, dv, chunk, flags, &nothing);
  if (rc != GDN_OK || nothing) return rc;
  const size_t need = prefill_workspace_bytes(T, N, Hv, dk, dv, chunk);
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGNMENT;
  return launch_delta_prefill(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                              has_initial_state, o, Hk, Hv, dk, dv, chunk, flags, workspace,
                              static_cast<cudaStream_t>(stream), slots);
}

gdn_status_t gdn_delta_rule_prefill_plan(const int32_t* cu_seqlens, int32_t N, int32_t T,
                                         int32_t Hv, int32_t dk, int32_t dv, int32_t chunk,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || N < 0 || Hv <= 0) return GDN_ERR_INVALID_ARG;
  if (chunk != 64) return GDN_ERR_UNSUPPORTED;
  if (T == 0 || N == 0) return GDN_OK;
  if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv) || dk != dv) return GDN_ERR_UNSUPPORTED;
  if ((int64_t)N * Hv > 0x7fffffff) return GDN_ERR_UNSUPPORTED;
  const size_t need = prefill_workspace_bytes(T, N, Hv, dk, dv, chunk);
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGNMENT;
  return launch_prefill_plan(cu_seqlens, N, T, Hv, dk, workspace,
                             static_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_delta_rule_prefill_chunked(const void* q, const void* k, int64_t qk_stride,
                                            const void* v, int64_t v_stride,
                                            const float* a, const float* b,
                                            const int32_t* cu_seqlens, int32_t N, int32_t T,
                                            float* S, const uint8_t* has_initial_state,
                                            void* o, int32_t Hk, int32_t Hv, int32_t dk,
                                            int32_t dv, int32_t chunk, int32_t flags,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream) {
  return prefill_impl(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                      has_initial_state, o, Hk, Hv, dk, dv, chunk, flags, workspace,
                      workspace_bytes, stream, StateSlots{});
}

gdn_status_t gdn_delta_rule_prefill_chunked_slots(
    const void* q, const void* k, int64_t qk_stride, const void* v, int64_t v_stride,
    const float* a, const float* b, const int32_t* cu_seqlens, int32_t N, int32_t T, float* S,
    const uint8_t* has_initial_state, void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
    int32_t chunk, int32_t flags, void* workspace, size_t workspace_bytes,
    const int32_t* state_indices, int32_t num_slots, void* stream) {
  StateSlots slots;
  gdn_status_t rc = make_slots(state_indices, num_slots, &slots);
  if (rc != GDN_OK) return rc;
  return prefill_impl(q, k, qk_stride, v, v_stride, a, b, cu_seqlens, N, T, S,
                      has_initial_state, o, Hk, Hv, dk, dv, chunk, flags, workspace,
                      workspace_bytes, stream, slots);
}

}  // extern "C"
