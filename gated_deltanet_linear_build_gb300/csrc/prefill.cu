// Chunked (WY / UT) prefill of the gated delta rule.
//
// The recurrence S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t is evaluated chunk by chunk. Inside a chunk of n tokens
// r = 0..n-1 that enters with state S0, with g_r = sum_{s<=r} log a_s:
//   u_r := b_r (v_r - a_r S_{r-1} k_r)  gives  S_r = a_r S_{r-1} + u_r k_r^T;
//   A_rs = b_r e^{g_r - g_s} (k_r . k_s) for s < r (strictly lower);
//   Tm = (I + A)^{-1}  (unit lower triangular, forward substitution);
//   W = Tm diag(b e^g) K,   U = Tm diag(b) V;
//   Delta = U - W S0^T      (the u_r of the chunk, as rows);
//   O = diag(e^g) Q S0^T + (M o Q K^T) Delta,  M_rs = e^{g_r - g_s} (s <= r);
//   S_n = e^{g_{n-1}} S0 + Delta^T diag(e^{g_{n-1} - g}) K.
// Chunks start at each sequence's first token and never cross sequences.
//
// Three launches:
//   1. descriptors of the 64-token chunks (the conv descriptor builder, with
//      chunk_tokens = 64) into the workspace;
//   2. intra-chunk kernel, one CTA per (chunk, v-head): g, A, Tm, W and U,
//      written to the workspace by token row;
//   3. state pass, one CTA per (sequence, v-head, 32-row slice of S): walks the
//      chunks in order, forms Delta, the outputs and the next state. Rows of S
//      (dv index) evolve independently, so slices need no exchange.
// This file holds the float32 CUDA-core version, used for head dims 16, 32
// and 64; head dim 128 runs on the tensor cores (prefill_tc.cu).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kChunk = 64;
constexpr int kThreads = 256;
constexpr int kSlice = 32;  // rows of S per state-pass CTA (dv >= 32), else dv

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t desc_off, g_off, w_off, u_off, total;
  int capacity;
};

__host__ __device__ inline WsLayout ws_layout(int T, int N, int Hv, int dk, int dv) {
  WsLayout L;
  L.capacity = T / kChunk + N + 1;
  size_t off = 256;  // [0]: descriptor count, [1]: builder status
  L.desc_off = off;
  off += align256((size_t)L.capacity * sizeof(gdn_conv_chunk_t));
  L.g_off = off;
  off += align256((size_t)T * Hv * sizeof(float));
  L.w_off = off;
  off += align256((size_t)T * Hv * dk * sizeof(float));
  L.u_off = off;
  off += align256((size_t)T * Hv * dv * sizeof(float));
  L.total = off;
  return L;
}

// Rows of length D (BF16, contiguous in global) -> float smem rows with pitch
// P, optionally L2-normalised. One warp per row.
template <int D, int P>
__device__ __forceinline__ void load_rows_bf16(float* dst, const __nv_bfloat16* src,
                                               int64_t row_stride, int rows, int l2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = warp; r < kChunk; r += kThreads / 32) {
    float vals[(D + 31) / 32];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < (D + 31) / 32; ++e) {
      const int j = lane + 32 * e;
      float x = 0.f;
      if (r < rows && j < D) x = __bfloat162float(src[r * row_stride + j]);
      vals[e] = x;
      ss += x * x;
    }
    if (l2) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rn = 1.0f / sqrtf(ss + 1e-6f);
#pragma unroll
      for (int e = 0; e < (D + 31) / 32; ++e) vals[e] *= rn;
    }
#pragma unroll
    for (int e = 0; e < (D + 31) / 32; ++e) {
      const int j = lane + 32 * e;
      if (j < D) dst[r * P + j] = vals[e];
    }
  }
}

// ---------------------------------------------------------------------------
// Intra-chunk kernel: one CTA per (chunk, v-head).
// ---------------------------------------------------------------------------
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads)
intra_chunk_kernel(const __nv_bfloat16* __restrict__ k, int64_t qk_stride,
                   const __nv_bfloat16* __restrict__ v, int64_t v_stride,
                   const float* __restrict__ a, const float* __restrict__ b,
                   const int32_t* __restrict__ count, const gdn_conv_chunk_t* __restrict__ desc,
                   int T, int Hk, int Hv, int flags, float* __restrict__ g_ws,
                   float* __restrict__ w_ws, float* __restrict__ u_ws) {
  constexpr int PK = DK + 1, PV = DV + 1, PT = kChunk + 1;
  extern __shared__ float smem[];
  float* Ks = smem;                    // [64][PK]
  float* Vs = Ks + kChunk * PK;        // [64][PV]
  float* As = Vs + kChunk * PV;        // [64][PT]
  float* Tm = As + kChunk * PT;        // [64][PT]
  float* gs = Tm + kChunk * PT;        // [64]
  float* bs = gs + kChunk;             // [64]
  float* cwk = bs + kChunk;            // [64]  b_s e^{g_s}

  if ((int)blockIdx.x >= *count) return;
  const int4 d = reinterpret_cast<const int4*>(desc)[blockIdx.x];
  const int tok0 = d.y, n = d.z;
  if (tok0 < 0 || n <= 0 || n > kChunk || tok0 + n > T) return;
  const int h = blockIdx.y, g = h / (Hv / Hk);
  const int tid = threadIdx.x;

  load_rows_bf16<DK, PK>(Ks, k + tok0 * qk_stride + (int64_t)g * DK, qk_stride, n, flags & kFlagL2);
  load_rows_bf16<DV, PV>(Vs, v + tok0 * v_stride + (int64_t)h * DV, v_stride, n, 0);
  if (tid < kChunk) {
    const bool in = tid < n;
    const bool gl = (flags & kFlagGateLogits) != 0;
    gs[tid] = in ? gate_ln_decay(a[(int64_t)(tok0 + tid) * Hv + h], gl) : 0.f;
    bs[tid] = in ? gate_write(b[(int64_t)(tok0 + tid) * Hv + h], gl) : 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f;
    for (int r = 0; r < n; ++r) { acc += gs[r]; gs[r] = acc; }
  }
  __syncthreads();
  if (tid < kChunk) cwk[tid] = bs[tid] * expf(gs[tid]);
  // A (strictly lower) and Tm = I on the diagonal.
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
    const int r = idx / kChunk, s = idx % kChunk;
    float val = 0.f;
    if (s < r && r < n) {
      float dot = 0.f;
#pragma unroll 8
      for (int j = 0; j < DK; ++j) dot = fmaf(Ks[r * PK + j], Ks[s * PK + j], dot);
      val = bs[r] * expf(gs[r] - gs[s]) * dot;
    }
    As[r * PT + s] = val;
    Tm[r * PT + s] = (r == s) ? 1.f : 0.f;
  }
  __syncthreads();
  // Forward substitution: Tm_r = e_r - sum_{s<r} A_rs Tm_s (column j per thread).
  for (int r = 1; r < n; ++r) {
    if (tid < r) {
      const int j = tid;
      float acc = 0.f;
      for (int s = j; s < r; ++s) acc = fmaf(As[r * PT + s], Tm[s * PT + j], acc);
      Tm[r * PT + j] = -acc;
    }
    __syncthreads();
  }
  // W = Tm diag(b e^g) K and U = Tm diag(b) V, rows r < n, to the workspace.
  for (int idx = tid; idx < n * DK; idx += kThreads) {
    const int r = idx / DK, j = idx % DK;
    float acc = 0.f;
    for (int s = 0; s <= r; ++s) acc = fmaf(Tm[r * PT + s] * cwk[s], Ks[s * PK + j], acc);
    w_ws[((int64_t)(tok0 + r) * Hv + h) * DK + j] = acc;
  }
  for (int idx = tid; idx < n * DV; idx += kThreads) {
    const int r = idx / DV, j = idx % DV;
    float acc = 0.f;
    for (int s = 0; s <= r; ++s) acc = fmaf(Tm[r * PT + s] * bs[s], Vs[s * PV + j], acc);
    u_ws[((int64_t)(tok0 + r) * Hv + h) * DV + j] = acc;
  }
  if (tid < n) g_ws[(int64_t)(tok0 + tid) * Hv + h] = gs[tid];
}

// ---------------------------------------------------------------------------
// State pass: one CTA per (sequence, v-head, slice of SL rows of S).
// ---------------------------------------------------------------------------
template <int DK, int DV, int SL>
__global__ void __launch_bounds__(kThreads)
state_pass_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  int64_t qk_stride, const int32_t* __restrict__ cu, int T,
                  float* __restrict__ S, const uint8_t* __restrict__ has_init,
                  __nv_bfloat16* __restrict__ o, int Hk, int Hv, int flags,
                  const float* __restrict__ g_ws, const float* __restrict__ w_ws,
                  const float* __restrict__ u_ws, const int32_t* __restrict__ bstatus,
                  const StateSlots slots) {
  constexpr int PK = DK + 1, PT = kChunk + 1, PS = SL + 1;
  extern __shared__ float smem[];
  float* Ss = smem;                  // [SL][PK]   state rows i (slice), columns j
  float* Ws = Ss + SL * PK;          // [64][PK]
  float* Qs = Ws + kChunk * PK;      // [64][PK]
  float* Ks = Qs + kChunk * PK;      // [64][PK]
  float* Us = Ks + kChunk * PK;      // [64][PS]
  float* Ds = Us + kChunk * PS;      // [64][PS]   Delta
  float* Ps = Ds + kChunk * PS;      // [64][PT]   M o Q K^T
  float* gs = Ps + kChunk * PT;      // [64]

  const int seq = blockIdx.x, h = blockIdx.y, i0 = blockIdx.z * SL;
  const int g = h / (Hv / Hk);
  const int tid = threadIdx.x;
  const int start = cu[seq], end = cu[seq + 1];
  if (end <= start || start < 0 || end > T) return;
  const int slot = state_slot(slots, seq);
  if (slot < 0) return;   // a padding entry: state and outputs untouched
  // Malformed cu_seqlens: the builder produced no chunks, so the per-token
  // workspace rows were never written; leave state and outputs untouched.
  if (*bstatus != GDN_OK) return;
  float* Sg = S + ((size_t)slot * Hv + h) * DV * DK + (size_t)i0 * DK;
  const bool init = has_init != nullptr && has_init[seq] != 0;
  for (int idx = tid; idx < SL * DK; idx += kThreads) {
    const int i = idx / DK, j = idx % DK;
    Ss[i * PK + j] = init ? Sg[(size_t)i * DK + j] : 0.f;
  }
  for (int c0 = start; c0 < end; c0 += kChunk) {
    const int n = min(kChunk, end - c0);
    __syncthreads();
    load_rows_bf16<DK, PK>(Qs, q + c0 * qk_stride + (int64_t)g * DK, qk_stride, n, flags & kFlagL2);
    load_rows_bf16<DK, PK>(Ks, k + c0 * qk_stride + (int64_t)g * DK, qk_stride, n, flags & kFlagL2);
    for (int idx = tid; idx < kChunk * DK; idx += kThreads) {
      const int r = idx / DK, j = idx % DK;
      Ws[r * PK + j] = r < n ? w_ws[((int64_t)(c0 + r) * Hv + h) * DK + j] : 0.f;
    }
    for (int idx = tid; idx < kChunk * SL; idx += kThreads) {
      const int r = idx / SL, i = idx % SL;
      Us[r * PS + i] = r < n ? u_ws[((int64_t)(c0 + r) * Hv + h) * DV + i0 + i] : 0.f;
    }
    if (tid < kChunk) gs[tid] = tid < n ? g_ws[(int64_t)(c0 + tid) * Hv + h] : 0.f;
    __syncthreads();
    // Delta = U - W S^T ; P = M o Q K^T.
    for (int idx = tid; idx < kChunk * SL; idx += kThreads) {
      const int r = idx / SL, i = idx % SL;
      float acc = 0.f;
#pragma unroll 8
      for (int j = 0; j < DK; ++j) acc = fmaf(Ws[r * PK + j], Ss[i * PK + j], acc);
      Ds[r * PS + i] = Us[r * PS + i] - acc;
    }
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
      const int r = idx / kChunk, s = idx % kChunk;
      float val = 0.f;
      if (s <= r && r < n) {
        float acc = 0.f;
#pragma unroll 8
        for (int j = 0; j < DK; ++j) acc = fmaf(Qs[r * PK + j], Ks[s * PK + j], acc);
        val = expf(gs[r] - gs[s]) * acc;
      }
      Ps[r * PT + s] = val;
    }
    __syncthreads();
    // O = diag(e^g) Q S^T + P Delta.
    for (int idx = tid; idx < n * SL; idx += kThreads) {
      const int r = idx / SL, i = idx % SL;
      float qs = 0.f;
#pragma unroll 8
      for (int j = 0; j < DK; ++j) qs = fmaf(Qs[r * PK + j], Ss[i * PK + j], qs);
      float pd = 0.f;
      for (int s = 0; s <= r; ++s) pd = fmaf(Ps[r * PT + s], Ds[s * PS + i], pd);
      const float val = fmaf(expf(gs[r]), qs, pd);
      o[((int64_t)(c0 + r) * Hv + h) * DV + i0 + i] = __float2bfloat16_rn(val);
    }
    __syncthreads();
    // S <- e^{g_{n-1}} S + Delta^T diag(e^{g_{n-1} - g}) K.
    const float gl = gs[n - 1];
    const float decay = expf(gl);
    for (int idx = tid; idx < SL * DK; idx += kThreads) {
      const int i = idx / DK, j = idx % DK;
      float acc = 0.f;
      for (int s = 0; s < n; ++s) acc = fmaf(Ds[s * PS + i] * expf(gl - gs[s]), Ks[s * PK + j], acc);
      Ss[i * PK + j] = fmaf(decay, Ss[i * PK + j], acc);
    }
  }
  __syncthreads();
  for (int idx = tid; idx < SL * DK; idx += kThreads) {
    const int i = idx / DK, j = idx % DK;
    Sg[(size_t)i * DK + j] = Ss[i * PK + j];
  }
}

template <int D>
gdn_status_t launch_prefill_t(const void* q, const void* k, int64_t qk_stride, const void* v,
                              int64_t v_stride, const float* a, const float* b,
                              const int32_t* cu, int N, int T, float* S,
                              const uint8_t* has_init, void* o, int Hk, int Hv, int flags,
                              void* workspace, cudaStream_t st, StateSlots slots) {
  constexpr int DK = D, DV = D, SL = D < kSlice ? D : kSlice;
  const WsLayout L = ws_layout(T, N, Hv, DK, DV);
  char* ws = static_cast<char*>(workspace);
  int32_t* count = reinterpret_cast<int32_t*>(ws);
  int32_t* bstatus = count + 1;
  auto desc = reinterpret_cast<gdn_conv_chunk_t*>(ws + L.desc_off);
  float* g_ws = reinterpret_cast<float*>(ws + L.g_off);
  float* w_ws = reinterpret_cast<float*>(ws + L.w_off);
  float* u_ws = reinterpret_cast<float*>(ws + L.u_off);
  auto qp = static_cast<const __nv_bfloat16*>(q);
  auto kp = static_cast<const __nv_bfloat16*>(k);
  auto vp = static_cast<const __nv_bfloat16*>(v);

  // Word 2 of the workspace header: the state pass's status. This state pass
  // has no device-side waits, so it always reports GDN_OK.
  if (cudaMemsetAsync(count + 2, 0, sizeof(int32_t), st) != cudaSuccess) return check_launch();
  gdn_status_t rc = GDN_OK;
  if (!(flags & kFlagPlanned)) {
    rc = launch_build_chunks(cu, N, kChunk, desc, L.capacity, count, bstatus, st);
    if (rc != GDN_OK) return rc;
  }

  constexpr int PK = DK + 1, PV = DV + 1, PT = kChunk + 1, PS = SL + 1;
  constexpr size_t smem1 =
      sizeof(float) * (kChunk * PK + kChunk * PV + 2 * kChunk * PT + 3 * kChunk);
  constexpr size_t smem2 =
      sizeof(float) * (SL * PK + 3 * kChunk * PK + 2 * kChunk * PS + kChunk * PT + kChunk);
  auto k1 = intra_chunk_kernel<DK, DV>;
  auto k2 = state_pass_kernel<DK, DV, SL>;
  // Opt in to more than 48 KB of dynamic shared memory, once per process (not a
  // stream operation, so it is also safe while a stream is being captured).
  static const bool smem_attrs = [] {
    cudaFuncSetAttribute(intra_chunk_kernel<DK, DV>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    cudaFuncSetAttribute(state_pass_kernel<DK, DV, SL>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
    return true;
  }();
  (void)smem_attrs;
  k1<<<dim3(L.capacity, Hv), kThreads, smem1, st>>>(kp, qk_stride, vp, v_stride, a, b, count,
                                                     desc, T, Hk, Hv, flags, g_ws, w_ws, u_ws);
  if ((rc = check_launch()) != GDN_OK) return rc;
  k2<<<dim3(N, Hv, DV / SL), kThreads, smem2, st>>>(qp, kp, qk_stride, cu, T, S, has_init,
                                                    static_cast<__nv_bfloat16*>(o), Hk, Hv, flags,
                                                    g_ws, w_ws, u_ws, bstatus, slots);
  return check_launch();
}

}  // namespace

size_t prefill_workspace_bytes(int32_t T, int32_t N, int32_t Hv, int32_t dk, int32_t dv,
                               int32_t chunk) {
  if (T < 0 || N < 0 || Hv <= 0 || dk <= 0 || dv <= 0 || chunk != kChunk) return 0;
  if (dk == 128 && dv == 128) return prefill_tc_workspace_bytes(T, N, Hv);
  return ws_layout(T, N, Hv, dk, dv).total;
}

gdn_status_t launch_prefill_plan(const int32_t* cu, int32_t N, int32_t T, int32_t Hv,
                                 int32_t dk, void* workspace, cudaStream_t st) {
  if (dk == 128) return launch_prefill_tc_plan(cu, N, T, Hv, workspace, st);
  const WsLayout L = ws_layout(T, N, Hv, dk, dk);
  char* ws = static_cast<char*>(workspace);
  int32_t* count = reinterpret_cast<int32_t*>(ws);
  return launch_build_chunks(cu, N, kChunk, reinterpret_cast<gdn_conv_chunk_t*>(ws + L.desc_off),
                             L.capacity, count, count + 1, st);
}

gdn_status_t launch_delta_prefill(const void* q, const void* k, int64_t qk_stride,
                                  const void* v, int64_t v_stride, const float* a,
                                  const float* b, const int32_t* cu, int32_t N, int32_t T,
                                  float* S, const uint8_t* has_init, void* o, int32_t Hk,
                                  int32_t Hv, int32_t dk, int32_t dv, int32_t chunk,
                                  int32_t flags, void* workspace, cudaStream_t st,
                                  StateSlots slots) {
  (void)chunk;
  if (dk != dv) return GDN_ERR_UNSUPPORTED;
  switch (dk) {
    case 16: return launch_prefill_t<16>(q, k, qk_stride, v, v_stride, a, b, cu, N, T, S, has_init, o, Hk, Hv, flags, workspace, st, slots);
    case 32: return launch_prefill_t<32>(q, k, qk_stride, v, v_stride, a, b, cu, N, T, S, has_init, o, Hk, Hv, flags, workspace, st, slots);
    case 64: return launch_prefill_t<64>(q, k, qk_stride, v, v_stride, a, b, cu, N, T, S, has_init, o, Hk, Hv, flags, workspace, st, slots);
    case 128: return launch_prefill_tc(q, k, qk_stride, v, v_stride, a, b, cu, N, T, S, has_init, o, Hk, Hv, flags, workspace, st, slots);
  }
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
