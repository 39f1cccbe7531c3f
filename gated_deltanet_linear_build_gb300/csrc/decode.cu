// Single-token gated delta-rule update (decode).
//
// Source: "RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs vLLM",
// Existing evidence: the fused decode kernel, the register-resident state arm
// (each state element read once and written once per token), and the lesson
// that scalar state stores regress the kernel (vector stores kept).
//
// Per (sequence n, v-head h), with q/k-head g = h / (Hv / Hk):
//   S' = a S,  u = b (v - S' k),  S_new = S' + u k^T,  o = S_new q
//      = a (S q) + u (k . q).
// Rows of S (one per dv index) are independent: row i needs only S_i . k and
// S_i . q, then S_i <- a S_i + u_i k. So a row is one pass: a group of dk/4
// lanes loads it as float4 vectors, reduces both dot products with xor
// shuffles inside the group, updates the row in registers and stores it.
//
// GB300 mapping: the kernel is HBM-bound (dv * dk * 8 bytes of state traffic
// per (n, h), 128 KiB at dk = dv = 128). A CTA of up to 256 threads owns one
// (n, h); each lane keeps kRowBatch row vectors in flight before reducing, so
// a resident SM has ~128 KiB of loads outstanding. S is streamed with
// evict-first hints (it is touched once per step).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

template <int DK, int DV>
struct DecodeCfg {
  static constexpr int kLanesPerRow = DK / 4;                 // float4 per lane
  static constexpr int kRowsPerWarp = 32 / kLanesPerRow;      // rows per warp per pass
  static constexpr int kThreads = (DV * kLanesPerRow < 256) ? DV * kLanesPerRow : 256;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kRowsPerPass = kWarps * kRowsPerWarp;
  static constexpr int kPasses = DV / kRowsPerPass;
  static constexpr int kRowBatch = kPasses < 8 ? kPasses : 8;
  static_assert(DV % kRowsPerPass == 0, "row mapping");
  static_assert(kPasses % kRowBatch == 0, "row batching");
};

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float4 ld_bf16x4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
}

template <int DK, int DV>
__global__ void __launch_bounds__(DecodeCfg<DK, DV>::kThreads)
delta_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    int64_t qk_stride, const __nv_bfloat16* __restrict__ v, int64_t v_stride,
                    const float* __restrict__ a, const float* __restrict__ b,
                    float* __restrict__ S, __nv_bfloat16* __restrict__ o, int Hk, int Hv,
                    int qk_l2norm) {
  using Cfg = DecodeCfg<DK, DV>;
  constexpr int LPR = Cfg::kLanesPerRow;
  __shared__ float s_o[DV];

  const int nh = blockIdx.x;  // n * Hv + h
  const int n = nh / Hv, h = nh - n * Hv;
  const int g = h / (Hv / Hk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % LPR;              // float4 column of this lane
  const int row_in_warp = lane / LPR;

  float4 k4 = ld_bf16x4(k + n * qk_stride + (int64_t)g * DK + sub * 4);
  float4 q4 = ld_bf16x4(q + n * qk_stride + (int64_t)g * DK + sub * 4);
  if (qk_l2norm) {
    const float kk = group_sum<LPR>(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
    const float qq = group_sum<LPR>(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
    const float rk = 1.0f / sqrtf(kk + 1e-6f), rq = 1.0f / sqrtf(qq + 1e-6f);
    k4 = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
    q4 = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
  }
  const float kq = group_sum<LPR>(k4.x * q4.x + k4.y * q4.y + k4.z * q4.z + k4.w * q4.w);
  const float av = __ldg(a + nh), bv = __ldg(b + nh);

  float* Sh = S + (size_t)nh * DV * DK;
  const __nv_bfloat16* vh = v + n * v_stride + (int64_t)h * DV;

#pragma unroll 1
  for (int p0 = 0; p0 < Cfg::kPasses; p0 += Cfg::kRowBatch) {
    float4 s[Cfg::kRowBatch];
    float vv[Cfg::kRowBatch];
#pragma unroll
    for (int r = 0; r < Cfg::kRowBatch; ++r) {
      const int row = (p0 + r) * Cfg::kRowsPerPass + warp * Cfg::kRowsPerWarp + row_in_warp;
      s[r] = __ldcs(reinterpret_cast<const float4*>(Sh + (size_t)row * DK) + sub);
      vv[r] = __bfloat162float(vh[row]);
    }
#pragma unroll
    for (int r = 0; r < Cfg::kRowBatch; ++r) {
      const int row = (p0 + r) * Cfg::kRowsPerPass + warp * Cfg::kRowsPerWarp + row_in_warp;
      const float sk = group_sum<LPR>(s[r].x * k4.x + s[r].y * k4.y + s[r].z * k4.z + s[r].w * k4.w);
      const float sq = group_sum<LPR>(s[r].x * q4.x + s[r].y * q4.y + s[r].z * q4.z + s[r].w * q4.w);
      const float u = bv * (vv[r] - av * sk);
      float4 sn;
      sn.x = fmaf(u, k4.x, av * s[r].x);
      sn.y = fmaf(u, k4.y, av * s[r].y);
      sn.z = fmaf(u, k4.z, av * s[r].z);
      sn.w = fmaf(u, k4.w, av * s[r].w);
      __stcs(reinterpret_cast<float4*>(Sh + (size_t)row * DK) + sub, sn);
      if (sub == 0) s_o[row] = fmaf(u, kq, av * sq);
    }
  }
  __syncthreads();
  // Output row of this (n, h): DV BF16 values, written as 16-byte vectors.
  for (int c = threadIdx.x; c < DV / 8; c += blockDim.x)
    *reinterpret_cast<uint4*>(o + (size_t)nh * DV + c * 8) = pack8(s_o + c * 8);
}

template <int DK, int DV>
gdn_status_t launch_decode_t(const void* q, const void* k, int64_t qk_stride, const void* v,
                             int64_t v_stride, const float* a, const float* b, float* S,
                             void* o, int N, int Hk, int Hv, int qk_l2norm, cudaStream_t st) {
  using Cfg = DecodeCfg<DK, DV>;
  delta_decode_kernel<DK, DV><<<N * Hv, Cfg::kThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qk_stride,
      static_cast<const __nv_bfloat16*>(v), v_stride, a, b, S,
      static_cast<__nv_bfloat16*>(o), Hk, Hv, qk_l2norm);
  return check_launch();
}

template <int DK>
gdn_status_t launch_decode_dv(int dv, const void* q, const void* k, int64_t qk_stride,
                              const void* v, int64_t v_stride, const float* a, const float* b,
                              float* S, void* o, int N, int Hk, int Hv, int l2, cudaStream_t st) {
  switch (dv) {
    case 16: return launch_decode_t<DK, 16>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st);
    case 32: return launch_decode_t<DK, 32>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st);
    case 64: return launch_decode_t<DK, 64>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st);
    case 128: return launch_decode_t<DK, 128>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st);
  }
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace

gdn_status_t launch_delta_decode(const void* q, const void* k, int64_t qk_stride,
                                 const void* v, int64_t v_stride, const float* a,
                                 const float* b, float* S, void* o, int32_t N, int32_t Hk,
                                 int32_t Hv, int32_t dk, int32_t dv, int32_t qk_l2norm,
                                 cudaStream_t st) {
  switch (dk) {
    case 16: return launch_decode_dv<16>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
    case 32: return launch_decode_dv<32>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
    case 64: return launch_decode_dv<64>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
    case 128: return launch_decode_dv<128>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
  }
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
