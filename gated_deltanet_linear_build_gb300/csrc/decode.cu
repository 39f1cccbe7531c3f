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
#include "tc_ptx.cuh"

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

// ---------------------------------------------------------------------------
// dk = dv = 128: persistent, warp-specialized streaming kernel. The state is
// cut into units of 64 rows of one (sequence, v-head) -- 32 KB, contiguous --
// and each CTA (one per SM) walks its units through a ring of shared-memory
// stages. A producer warp issues, per unit, TMA bulk loads of the rows plus
// the unit's k, q (256 B each) and v (128 B) into a stage, and later the bulk
// stores of the updated rows and of the unit's 64 outputs; sixteen compute
// warps wait on the stage's "full" barrier, update four rows each in place,
// and arrive on its "empty" barrier. kDecStages units are in flight per SM.
// ---------------------------------------------------------------------------
constexpr int kDecRows = 64;                       // rows of S per unit
constexpr int kDecUnitBytes = kDecRows * 128 * 4;  // 32 KB
constexpr int kDecOffK = kDecUnitBytes, kDecOffQ = kDecOffK + 256, kDecOffV = kDecOffQ + 256;
constexpr int kDecOffO = kDecOffV + 2 * kDecRows;  // BF16 outputs of the unit's rows
constexpr int kDecStageBytes = kDecOffO + 2 * kDecRows;
constexpr int kDecStages = 6;
constexpr int kDecWarps = 16;                      // compute warps, 4 rows each
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + producer warp
constexpr int kDecSmem = kDecStages * kDecStageBytes + 2 * kDecStages * 8 + 64;
constexpr int kDecUnitsPerHead = 128 / kDecRows;

// Sum over the 32 lanes of eight per-lane values at once (transpose-reduce):
// after five exchange rounds lane l holds the full sum of value (l >> 2) & 7
// (lanes 4m..4m+3 hold value m); 9 shuffles instead of 40.
__device__ __forceinline__ float reduce8_transpose(const float (&x)[8], int lane) {
  float y4[4], y2[2], y1;
  const bool up16 = lane & 16, up8 = lane & 8, up4 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {   // keep values [0,4) on lanes without bit 16, [4,8) with it
    const float send = up16 ? x[i] : x[i + 4];
    const float keep = up16 ? x[i + 4] : x[i];
    y4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = up8 ? y4[i] : y4[i + 2];
    const float keep = up8 ? y4[i + 2] : y4[i];
    y2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const float send = up4 ? y2[0] : y2[1];
    const float keep = up4 ? y2[1] : y2[0];
    y1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
  y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
  return y1;   // value index m = 4 (lane & 16 ? 1 : 0) + 2 (lane & 8 ? 1 : 0) + (lane & 4 ? 1 : 0)
}

__global__ void __launch_bounds__(kDecThreads, 1)
delta_decode_stream_kernel(const __nv_bfloat16* __restrict__ q,
                           const __nv_bfloat16* __restrict__ k, int64_t qk_stride,
                           const __nv_bfloat16* __restrict__ v, int64_t v_stride,
                           const float* __restrict__ a, const float* __restrict__ b,
                           float* __restrict__ S, __nv_bfloat16* __restrict__ o, int Hk, int Hv,
                           int qk_l2norm, int units) {
  using namespace tc;
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kDecStages * kDecStageBytes);
  uint64_t* empty = full + kDecStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int my_units = (units - (int)blockIdx.x + G - 1) / G;   // units blockIdx.x + i G
  if (tid == 0) {
    for (int st = 0; st < kDecStages; ++st) {
      mbar_init(full + st, 1);
      mbar_init(empty + st, kDecWarps);
    }
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // Producer warp (lane 0 issues).
    if (lane == 0) {
      auto issue_load = [&](int i) {
        const int st = i % kDecStages;
        const int unit = blockIdx.x + i * G;
        const int nh = unit / kDecUnitsPerHead, part = unit - nh * kDecUnitsPerHead;
        const int n = nh / Hv, h = nh - n * Hv, g = h / (Hv / Hk);
        unsigned char* dst = sm + st * kDecStageBytes;
        mbar_arrive_expect_tx(full + st, kDecUnitBytes + 256 + 256 + 2 * kDecRows);
        bulk_g2s(dst, S + (size_t)unit * kDecRows * 128, kDecUnitBytes, full + st);
        bulk_g2s(dst + kDecOffK, k + n * qk_stride + (int64_t)g * 128, 256, full + st);
        bulk_g2s(dst + kDecOffQ, q + n * qk_stride + (int64_t)g * 128, 256, full + st);
        bulk_g2s(dst + kDecOffV, v + n * v_stride + (int64_t)h * 128 + part * kDecRows,
                 2 * kDecRows, full + st);
      };
      for (int i = 0; i < my_units && i < kDecStages; ++i) issue_load(i);
      for (int i = 0; i < my_units; ++i) {
        const int st = i % kDecStages;
        mbar_wait(empty + st, (i / kDecStages) & 1);
        const int unit = blockIdx.x + i * G;
        bulk_s2g(S + (size_t)unit * kDecRows * 128, sm + st * kDecStageBytes, kDecUnitBytes);
        bulk_s2g(o + (size_t)unit * kDecRows, sm + st * kDecStageBytes + kDecOffO, 2 * kDecRows);
        bulk_commit();
        // Refill the stage stored one unit ago (its store has had a unit's
        // time to read shared memory), keeping kDecStages - 1 loads in flight.
        if (i >= 1 && i - 1 + kDecStages < my_units) {
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          issue_load(i - 1 + kDecStages);
        }
      }
      bulk_wait_all();
    }
    return;
  }

  // Compute warps: rows 4 warp .. 4 warp + 3 of every unit.
  float a_nxt = 0.f, b_nxt = 0.f;
  if (my_units > 0) {
    a_nxt = __ldg(a + blockIdx.x / kDecUnitsPerHead);
    b_nxt = __ldg(b + blockIdx.x / kDecUnitsPerHead);
  }
  for (int i = 0; i < my_units; ++i) {
    const int st = i % kDecStages;
    const int unit = blockIdx.x + i * G;
    const float av = a_nxt, bv = b_nxt;
    if (i + 1 < my_units) {
      a_nxt = __ldg(a + (unit + G) / kDecUnitsPerHead);
      b_nxt = __ldg(b + (unit + G) / kDecUnitsPerHead);
    }
    mbar_wait(full + st, (i / kDecStages) & 1);
    unsigned char* stage = sm + st * kDecStageBytes;
    const uint2 ku = reinterpret_cast<const uint2*>(stage + kDecOffK)[lane];
    const uint2 qu = reinterpret_cast<const uint2*>(stage + kDecOffQ)[lane];
    const uint2 vu = reinterpret_cast<const uint2*>(stage + kDecOffV)[warp];
    float4 k4 = make_float4(bf16lo(ku.x), bf16hi(ku.x), bf16lo(ku.y), bf16hi(ku.y));
    float4 q4 = make_float4(bf16lo(qu.x), bf16hi(qu.x), bf16lo(qu.y), bf16hi(qu.y));
    const float vv[4] = {bf16lo(vu.x), bf16hi(vu.x), bf16lo(vu.y), bf16hi(vu.y)};
    float4* rows = reinterpret_cast<float4*>(stage) + warp * 4 * 32 + lane;
    float4 sr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sr[j] = rows[j * 32];
    // Per-lane partial dot products: values 0-3 = S_j . k, 4-7 = S_j . q
    // (with the raw k, q; the optional L2 norms are applied to the sums).
    float part[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      part[j] = sr[j].x * k4.x + sr[j].y * k4.y + sr[j].z * k4.z + sr[j].w * k4.w;
      part[4 + j] = sr[j].x * q4.x + sr[j].y * q4.y + sr[j].z * q4.z + sr[j].w * q4.w;
    }
    float kk = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
    float qq = q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w;
    float kq = k4.x * q4.x + k4.y * q4.y + k4.z * q4.z + k4.w * q4.w;
    const float red = reduce8_transpose(part, lane);
    kk = group_sum<32>(kk);
    qq = group_sum<32>(qq);
    kq = group_sum<32>(kq);
    // Lanes 4m..4m+3 hold value m: S_j.k for m = j, S_j.q for m = 4 + j.
    float sk[4], sq[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sk[j] = __shfl_sync(0xffffffffu, red, 4 * j);
      sq[j] = __shfl_sync(0xffffffffu, red, 16 + 4 * j);
    }
    float rk = 1.f, rq = 1.f;
    if (qk_l2norm) {
      rk = 1.0f / sqrtf(kk + 1e-6f);
      rq = 1.0f / sqrtf(qq + 1e-6f);
    }
    // With normalised k = rk k~, q = rq q~: S k = rk (S k~), S q = rq (S q~),
    // k . q = rk rq (k~ . q~).
    const float kqn = kq * rk * rq;
    float ov[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 s4 = sr[j];
      const float u = bv * (vv[j] - av * (sk[j] * rk));
      const float uk = u * rk;
      float4 sn;
      sn.x = fmaf(uk, k4.x, av * s4.x);
      sn.y = fmaf(uk, k4.y, av * s4.y);
      sn.z = fmaf(uk, k4.z, av * s4.z);
      sn.w = fmaf(uk, k4.w, av * s4.w);
      rows[j * 32] = sn;
      ov[j] = fmaf(u, kqn, av * (sq[j] * rq));
    }
    if (lane < 2) {
      // lane 0 writes rows 0-1, lane 1 rows 2-3 of this warp as BF16 pairs
      const uint32_t pr = lane == 0 ? pack_bf16x2(ov[0], ov[1]) : pack_bf16x2(ov[2], ov[3]);
      reinterpret_cast<uint32_t*>(stage + kDecOffO)[warp * 2 + lane] = pr;
    }
    fence_smem_to_async();   // rows and outputs just written are read by the bulk stores
    __syncwarp();
    if (lane == 0) {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(empty + st)) : "memory");
    }
  }
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
  if (dk == 128 && dv == 128) {
    static const int num_sms = [] {
      int dev = 0, n = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      cudaFuncSetAttribute(delta_decode_stream_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
      return n > 0 ? n : 1;
    }();
    const int units = N * Hv * kDecUnitsPerHead;
    const int grid = units < num_sms ? units : num_sms;
    delta_decode_stream_kernel<<<grid, kDecThreads, kDecSmem, st>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qk_stride,
        static_cast<const __nv_bfloat16*>(v), v_stride, a, b, S, static_cast<__nv_bfloat16*>(o),
        Hk, Hv, qk_l2norm, units);
    return check_launch();
  }
  switch (dk) {
    case 16: return launch_decode_dv<16>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
    case 32: return launch_decode_dv<32>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
    case 64: return launch_decode_dv<64>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
    case 128: return launch_decode_dv<128>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, qk_l2norm, st);
  }
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
