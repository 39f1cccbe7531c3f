// Internal helpers shared by the GDN CUDA translation units (not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gdn.h"
#include "tc_ptx.cuh"

namespace gdn {

// ---------------------------------------------------------------------------
// Sticky device-side status. Every translation unit that includes this header
// owns one word (anonymous namespace: no cross-unit device symbols are needed,
// so no device link step). A kernel whose bounded wait gives up records
// GDN_ERR_TIMEOUT there (the first failure since the last clear stays);
// gdn_device_status reads the words of all units through their gather kernels.
// ---------------------------------------------------------------------------
namespace {
__device__ int32_t g_dev_status = 0;
__global__ void gather_status_kernel(int32_t* out, int clear, int first) {
  const int32_t v = *reinterpret_cast<volatile int32_t*>(&g_dev_status);
  if (first || *out == GDN_OK) *out = v;
  if (clear) g_dev_status = GDN_OK;
}
}  // namespace
__device__ __forceinline__ void record_device_status(int32_t status) {
  atomicCAS(&g_dev_status, (int32_t)GDN_OK, status);
}

// Bounded mbarrier wait for the phase of parity `parity` that also gives up as
// soon as *abort is non-zero (another role of the CTA gave up). On its own
// time-out (about `max_cycles` SM cycles) it sets *abort and records
// GDN_ERR_TIMEOUT in the sticky status. `sleep_ns` > 0 backs off between
// polls, so that a waiting warp takes few issue slots. Returns true when the
// phase completed.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t* mbar, uint32_t parity,
                                                    volatile int* abort, unsigned sleep_ns = 0,
                                                    long long max_cycles = 4000000000LL) {
  const long long t0 = clock64();
  while (!tc::mbar_try_wait(mbar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > max_cycles) {
      *abort = 1;
      record_device_status(GDN_ERR_TIMEOUT);
      return false;
    }
    if (sleep_ns) __nanosleep(sleep_ns);
  }
  return true;
}

// ---------------------------------------------------------------------------
// BF16 <-> float32 on packed 32-bit words (two BF16 values, element 0 in the
// low half). Widening is exact; narrowing rounds to nearest even.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// 8 BF16 values (one 16-byte vector) -> 8 floats.
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
  f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z);
  f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  return u;
}

// ---------------------------------------------------------------------------
// Pairs of float32 on the packed f32x2 FMA-pipe instructions of sm_100+ (one
// instruction for both halves; each half rounds exactly as the scalar op).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_bits(float2 v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 f2_from_bits(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return f2_from_bits(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return f2_from_bits(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return f2_from_bits(d);
}
// Two BF16 values of a packed word as a float pair (exact).
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }
__device__ __forceinline__ uint32_t f2_bf16x2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Read-only 16-byte global load (non-coherent path; inputs are never written
// by the kernel that reads them).
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// SiLU(x) = x / (1 + e^-x) = x * 1 / (1 + 2^(-x log2 e)), on the hardware
// base-2 exponential and reciprocal (ex2.approx.ftz, rcp.approx.ftz: a few
// float32 ulps, far below the BF16 rounding of the result). Two special-
// function operations and three FMA-pipe ones, where a libm-accurate exp and an
// IEEE division cost several times more and made the conv prefill ALU-bound.
// Large negative x gives 2^(+big) = inf, 1/inf = 0 and a (signed) zero result.
__device__ __forceinline__ float silu_f(float x) {
  float t, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + t));
  return x * r;
}

// silu_f on a pair, the multiplies and the add as f32x2 instructions (the same
// roundings as silu_f on each half).
__device__ __forceinline__ float2 silu2(float2 x) {
  const float2 t = mul2(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  float2 e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(t.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(t.y));
  const float2 d = add2(e, make_float2(1.0f, 1.0f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(d.y));
  return mul2(x, r);
}

// ---------------------------------------------------------------------------
// Option bits of the delta-rule entry points' `flags` (GDN_FLAG_* in gdn.h).
// ---------------------------------------------------------------------------
constexpr int kFlagL2 = GDN_FLAG_QK_L2NORM;
constexpr int kFlagGateLogits = GDN_FLAG_GATE_LOGITS;
constexpr int kFlagPlanned = GDN_FLAG_PLANNED;

// Gate activation from raw logits: a = exp(-softplus(z)) (decay), b =
// sigmoid(z) (write strength), on the hardware base-2 exponential and
// logarithm (ex2.approx / lg2.approx: errors near 2^-22, far below what the
// float32 state keeps): with u = log2 e,
//   log2 a = -(max(z, 0) u + log2(1 + 2^(-|z| u))),   b = 1 / (1 + 2^(-z u)),
// so that no intermediate overflows. Decays below 1e-30 act as 1e-30 in both
// gate forms (the kernels work with log a).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// log2 of the decay, clamped at log2(1e-30).
__device__ __forceinline__ float gate_log2_decay(float x, bool logits) {
  constexpr float kLog2Min = -99.65784284662087f;   // log2(1e-30)
  constexpr float kLog2e = 1.4426950408889634f;
  if (!logits) return log2f(fmaxf(x, 1e-30f));
  const float sp2 = fmaxf(x, 0.f) * kLog2e + lg2_approx(1.0f + ex2_approx(-fabsf(x) * kLog2e));
  return fmaxf(-sp2, kLog2Min);
}
// Natural log of the decay, clamped at ln(1e-30).
__device__ __forceinline__ float gate_ln_decay(float x, bool logits) {
  constexpr float kLn2 = 0.6931471805599453f;
  return logits ? gate_log2_decay(x, true) * kLn2 : logf(fmaxf(x, 1e-30f));
}
// The decay itself (decode forms).
__device__ __forceinline__ float gate_decay(float x, bool logits) {
  return logits ? ex2_approx(gate_log2_decay(x, true)) : x;
}
// The write strength.
__device__ __forceinline__ float gate_write(float x, bool logits) {
  if (!logits) return x;
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + ex2_approx(-x * 1.4426950408889634f)));
  return r;
}

// ---------------------------------------------------------------------------
// Host-side helpers
// ---------------------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Records the CUDA error text for gdn_last_cuda_error_string().
void set_cuda_error(cudaError_t e);

inline gdn_status_t check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

// Status of a launch call that returns its error (cudaLaunchKernelEx).
inline gdn_status_t check_launch(cudaError_t e) {
  if (e != cudaSuccess) {
    cudaGetLastError();   // clear it
    set_cuda_error(e);
    return GDN_ERR_CUDA;
  }
  return check_launch();
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel is launched with programmatic
// stream serialisation: it may start while the previous kernel on the stream
// is still finishing, runs only its own set-up (shared-memory barriers, tensor
// memory) before pdl_wait(), which returns once that kernel has completed and
// its writes are visible, and then lets the next kernel start launching
// (pdl_trigger()). Because a kernel triggers only after its own wait, every
// kernel two or more launches back has completed when a kernel starts. Without
// the launch attribute both instructions are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// L2 prefetch hints, usable before pdl_wait(): L2 is the point of coherence,
// so a line that the previous kernel writes afterwards is still read current.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Optional indirection from a sequence to its state slot: serving engines keep
// conv_state and S in a cache of slots and pass, per call, the slot of each
// sequence. idx == nullptr: the slot is the sequence index. A slot outside
// [0, count) marks a sequence whose state is not touched and whose outputs are
// not written (a padding entry).
// ---------------------------------------------------------------------------
struct StateSlots {
  const int32_t* idx = nullptr;
  int32_t count = 0;
};
__device__ __forceinline__ int state_slot(const StateSlots& s, int n) {
  if (s.idx == nullptr) return n;
  const int v = __ldg(s.idx + n);
  return (v >= 0 && v < s.count) ? v : -1;
}

// Status gathers of the kernel translation units (each launches its unit's
// gather_status_kernel): the first one called writes its word, the others only
// replace a GDN_OK.
gdn_status_t gather_status_api(int32_t* out, int clear, int first, cudaStream_t st);
gdn_status_t gather_status_conv(int32_t* out, int clear, int first, cudaStream_t st);
gdn_status_t gather_status_decode(int32_t* out, int clear, int first, cudaStream_t st);
gdn_status_t gather_status_prefill_tc(int32_t* out, int clear, int first, cudaStream_t st);
#define GDN_DEFINE_STATUS_GATHER(name)                                                   \
  gdn_status_t name(int32_t* out, int clear, int first, cudaStream_t st) {               \
    gather_status_kernel<<<1, 1, 0, st>>>(out, clear, first);                            \
    return check_launch();                                                               \
  }

// Launchers implemented in the kernel translation units. They assume their
// arguments were validated by the C ABI layer.
// order (device int32 [n] or nullptr): also write the sequences by descending
// chunk count (longest first), for kernels that start long sequences first.
gdn_status_t launch_build_chunks(const int32_t* cu, int32_t n, int32_t chunk_tokens,
                                 gdn_conv_chunk_t* chunks, int32_t capacity,
                                 int32_t* num_chunks, int32_t* status, cudaStream_t st,
                                 int32_t* order = nullptr);

gdn_status_t launch_conv_fwd(const void* x, int64_t x_stride, const void* w, const void* bias,
                             void* conv_state, const uint8_t* has_init, const int32_t* cu,
                             const gdn_conv_chunk_t* chunks, const int32_t* num_chunks,
                             int32_t units, int32_t T, int32_t C, int32_t N, int32_t silu,
                             void* y, cudaStream_t st, StateSlots slots = {});

gdn_status_t launch_conv_update(const void* x, int64_t x_stride, const void* w,
                                const void* bias, void* conv_state, int32_t N, int32_t C,
                                int32_t silu, void* y, cudaStream_t st, StateSlots slots = {});

gdn_status_t launch_delta_decode(const void* q, const void* k, int64_t qk_stride,
                                 const void* v, int64_t v_stride, const float* a,
                                 const float* b, float* S, void* o, int32_t N, int32_t Hk,
                                 int32_t Hv, int32_t dk, int32_t dv, int32_t flags,
                                 cudaStream_t st, StateSlots slots = {});

// Conv update and delta-rule decode in one launch (dk = dv = 128).
gdn_status_t launch_decode_fused(const void* x, int64_t x_stride, const void* w,
                                 const void* bias, const void* st_in, void* st_out,
                                 const float* a, const float* b, float* S, void* o, int32_t N,
                                 int32_t Hk, int32_t Hv, int32_t silu, int32_t flags,
                                 cudaStream_t st);

size_t prefill_workspace_bytes(int32_t T, int32_t N, int32_t Hv, int32_t dk, int32_t dv,
                               int32_t chunk);

// Host-side checks of gdn_delta_rule_prefill_chunked's arguments (everything
// but the workspace). GDN_OK with *nothing_to_do set: zero tokens or zero
// sequences, a valid call that enqueues nothing.
gdn_status_t check_prefill_args(const void* q, const void* k, int64_t qk_stride, const void* v,
                                int64_t v_stride, const float* a, const float* b,
                                const int32_t* cu_seqlens, int32_t N, int32_t T, const float* S,
                                const void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                int32_t chunk, int32_t flags, bool* nothing_to_do);

gdn_status_t launch_delta_prefill(const void* q, const void* k, int64_t qk_stride,
                                  const void* v, int64_t v_stride, const float* a,
                                  const float* b, const int32_t* cu, int32_t N, int32_t T,
                                  float* S, const uint8_t* has_init, void* o, int32_t Hk,
                                  int32_t Hv, int32_t dk, int32_t dv, int32_t chunk,
                                  int32_t flags, void* workspace, cudaStream_t st,
                                  StateSlots slots = {});

// The chunk plan of a prefill (descriptors, and the longest-first order for
// the tensor-core path) into the workspace.
gdn_status_t launch_prefill_plan(const int32_t* cu, int32_t N, int32_t T, int32_t Hv,
                                 int32_t dk, void* workspace, cudaStream_t st);
gdn_status_t launch_prefill_tc_plan(const int32_t* cu, int32_t N, int32_t T, int32_t Hv,
                                    void* workspace, cudaStream_t st);

// Tensor-core (tcgen05) chunked prefill for dk = dv = 128.
size_t prefill_tc_workspace_bytes(int32_t T, int32_t N, int32_t Hv);
gdn_status_t launch_prefill_tc(const void* q, const void* k, int64_t qk_stride, const void* v,
                               int64_t v_stride, const float* a, const float* b,
                               const int32_t* cu, int32_t N, int32_t T, float* S,
                               const uint8_t* has_init, void* o, int32_t Hk, int32_t Hv,
                               int32_t flags, void* workspace, cudaStream_t st,
                               StateSlots slots = {});

}  // namespace gdn
