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
                    int flags, const StateSlots slots) {
  using Cfg = DecodeCfg<DK, DV>;
  constexpr int LPR = Cfg::kLanesPerRow;
  __shared__ float s_o[DV];
  pdl_wait();
  pdl_trigger();

  const int nh = blockIdx.x;  // n * Hv + h
  const int n = nh / Hv, h = nh - n * Hv;
  const int slot = state_slot(slots, n);
  if (slot < 0) return;      // a padding entry
  const int g = h / (Hv / Hk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % LPR;              // float4 column of this lane
  const int row_in_warp = lane / LPR;

  float4 k4 = ld_bf16x4(k + n * qk_stride + (int64_t)g * DK + sub * 4);
  float4 q4 = ld_bf16x4(q + n * qk_stride + (int64_t)g * DK + sub * 4);
  if (flags & kFlagL2) {
    const float kk = group_sum<LPR>(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
    const float qq = group_sum<LPR>(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
    const float rk = 1.0f / sqrtf(kk + 1e-6f), rq = 1.0f / sqrtf(qq + 1e-6f);
    k4 = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
    q4 = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
  }
  const float kq = group_sum<LPR>(k4.x * q4.x + k4.y * q4.y + k4.z * q4.z + k4.w * q4.w);
  const bool gl = (flags & kFlagGateLogits) != 0;
  const float av = gate_decay(__ldg(a + nh), gl), bv = gate_write(__ldg(b + nh), gl);

  float* Sh = S + ((size_t)slot * Hv + h) * DV * DK;
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
// stages. A producer warp issues, per unit, a TMA bulk load of the rows into a
// stage, and later the bulk stores of the updated rows and of the unit's 64
// outputs; sixteen compute warps wait on the stage's "full" barrier, update
// four rows each in place, and arrive on its "empty" barrier.
// The unit's k, q (128 values each) and v (64) sit beside its rows in the
// stage. Unfused, the producer bulk-loads them from the conv output. Fused,
// the conv update runs in the kernel: a second producer warp bulk-loads the
// unit's conv inputs (x, state, taps, bias of its 320 channels) into a small
// ring of their own, and ten conv warps (one channel per thread) convolve
// them, write the BF16 outputs into the stage and the new conv state to
// global memory, and arrive on the stage's "full" barrier: the compute warps
// then run exactly as in the unfused kernel, one unit behind the conv warps.
// ---------------------------------------------------------------------------
constexpr int kDecRows = 64;                       // rows of S per unit
constexpr int kDecUnitBytes = kDecRows * 128 * 4;  // 32 KB
constexpr int kDecOffO = kDecUnitBytes;            // BF16 outputs of the unit's rows
constexpr int kDecOffK = kDecOffO + 2 * kDecRows;  // k, q (256 B each) and v (128 B)
constexpr int kDecOffQ = kDecOffK + 256, kDecOffV = kDecOffQ + 256;
constexpr int kDecStageBytes = kDecOffV + 2 * kDecRows;
constexpr int kDecStages = 6;
constexpr int kDecWarps = 16;                      // compute warps, 4 rows each
constexpr int kDecUnitsPerHead = 128 / kDecRows;
// Fused mode: conv-input slots, per q / k / v block of the unit's channels
// (128 / 128 / 64): x and the state [ch][3]. Offsets in a slot. (The taps and
// bias, the same for every sequence, are read through the cache by the conv
// warps themselves.)
constexpr int kFxQ = 0, kFxK = kFxQ + 256, kFxV = kFxK + 256;
constexpr int kFsQ = kFxV + 128, kFsK = kFsQ + 768, kFsV = kFsK + 768;
constexpr int kFSlot = kFsV + 384;                 // 2560 bytes
constexpr int kFSlots = 8;
constexpr int kFConv = 320;                        // conv channels of a unit (q, k, v)
constexpr int kFConvWarps = kFConv / 32;           // 10
constexpr int kFYSlot = 640;                       // BF16 k | q | v of a unit (fused)
constexpr int kFYSlots = 8;
template <bool kFused>
struct DecStage {
  static constexpr int kConvOff = kDecStages * kDecStageBytes;            // fused: conv ring
  static constexpr int kYOff = kConvOff + (kFused ? kFSlots * kFSlot : 0);  // fused: y ring
  static constexpr int kBarOff = kYOff + (kFused ? kFYSlots * kFYSlot : 0);
  static constexpr int kAbortOff = kBarOff + 2 * (kDecStages + kFSlots + kFYSlots) * 8;
  static constexpr int kSmem = kAbortOff + 64;
  // compute warps, state producer, [conv-input producer, conv warps]
  static constexpr int kProdWarp = kDecWarps;
  static constexpr int kConvWarp0 = kDecWarps + 2;
  static constexpr int kWarps = kDecWarps + 1 + (kFused ? 1 + kFConvWarps : 0);
  static constexpr int kThreads = kWarps * 32;
};

// Arguments of the streaming decode kernels (both modes).
struct DecodeArgs {
  // unfused: q, k, v read from the conv output
  const __nv_bfloat16 *q, *k, *v;
  int64_t qk_stride, v_stride;
  // fused: the conv update runs in the kernel (x, taps, bias, states)
  const __nv_bfloat16 *x, *w, *bias, *st_in;
  __nv_bfloat16* st_out;
  int64_t x_stride;
  int C, silu;
  // both
  const float *a, *b;
  float* S;
  __nv_bfloat16* o;
  int Hk, Hv, flags, units;   // flags: GDN_FLAG_* bits
  StateSlots slots;   // unfused only: sequence -> state slot
};

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

template <bool kFused>
__global__ void __launch_bounds__(DecStage<kFused>::kThreads, 1)
delta_decode_stream_kernel(const DecodeArgs p) {
  using namespace tc;
  using Cfg = DecStage<kFused>;
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Cfg::kBarOff);
  uint64_t* empty = full + kDecStages;
  uint64_t* cfull = empty + kDecStages;    // fused: conv-input ring
  uint64_t* cempty = cfull + kFSlots;
  uint64_t* yfull = cempty + kFSlots;      // fused: conv-output ring
  uint64_t* yempty = yfull + kFYSlots;
  // Set by the first role whose bounded wait gives up; every other wait then
  // gives up at once, no role stores a unit it has not finished, and the
  // state producer drains its copies in flight before the CTA exits.
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Cfg::kAbortOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int Hv = p.Hv, ratio = p.Hv / p.Hk;
  const int my_units = (p.units - (int)blockIdx.x + G - 1) / G;   // units blockIdx.x + i G
  if (tid == 0) {
    *abort = 0;
    for (int st = 0; st < kDecStages; ++st) {
      mbar_init(full + st, 1);
      mbar_init(empty + st, kDecWarps);
    }
    if constexpr (kFused) {
      for (int cs = 0; cs < kFSlots; ++cs) {
        mbar_init(cfull + cs, 32);   // one arrival per producer lane
        mbar_init(cempty + cs, kFConvWarps);
      }
      for (int ys = 0; ys < kFYSlots; ++ys) {
        mbar_init(yfull + ys, kFConvWarps);
        mbar_init(yempty + ys, kDecWarps);
      }
    }
  }
  __syncthreads();
  auto unit_coords = [&](int unit, int& n, int& h, int& g, int& part) {
    const int nh = unit / kDecUnitsPerHead;
    part = unit - nh * kDecUnitsPerHead;
    n = nh / Hv;
    h = nh - n * Hv;
    g = h / ratio;
  };
  if (!kFused && warp == Cfg::kProdWarp && lane == 0) {
    // Warm L2 with the state rows of the first stages while the previous
    // kernel finishes.
    for (int i = 0; i < my_units && i < kDecStages; ++i) {
      int n, h, g, part;
      unit_coords(blockIdx.x + i * G, n, h, g, part);
      const int slot = state_slot(p.slots, n);
      if (slot >= 0)
        bulk_prefetch_l2(p.S + (((size_t)slot * Hv + h) * kDecUnitsPerHead + part) * kDecRows * 128,
                         kDecUnitBytes);
    }
  }
  pdl_wait();
  pdl_trigger();

  if constexpr (kFused) {
    if (warp == Cfg::kProdWarp + 1) {
      // Conv-input producer: x and state of the unit's q, k and v channels
      // into the conv ring as 160 16-byte asynchronous copies, five per lane
      // (the slot's regions are contiguous in this order, so chunk t lands at
      // byte 16 t); each lane arrives on the slot's barrier once its own
      // copies have landed. Small bulk copies would queue in the copy engine
      // behind the state rows.
      for (int i = 0; i < my_units; ++i) {
        const int cs = i % kFSlots;
        const bool ok = i < kFSlots || mbar_wait_abortable(cempty + cs, ((i / kFSlots) - 1) & 1, abort);
        if (!__all_sync(0xffffffffu, ok)) break;
        int n, h, g, part;
        unit_coords(blockIdx.x + i * G, n, h, g, part);
        unsigned char* dst = sm + Cfg::kConvOff + cs * kFSlot;
        const int cq = g * 128, ck = p.Hk * 128 + g * 128;
        const int cv = 2 * p.Hk * 128 + h * 128 + part * kDecRows;
        const __nv_bfloat16* xr = p.x + n * p.x_stride;
        const __nv_bfloat16* sr = p.st_in + (size_t)n * p.C * 3;
#pragma unroll
        for (int m = 0; m < 5; ++m) {
          const int t = lane + 32 * m;
          const __nv_bfloat16* src =
              t < 16 ? xr + cq + 8 * t
            : t < 32 ? xr + ck + 8 * (t - 16)
            : t < 40 ? xr + cv + 8 * (t - 32)
            : t < 88 ? sr + (size_t)cq * 3 + 8 * (t - 40)
            : t < 136 ? sr + (size_t)ck * 3 + 8 * (t - 88)
                      : sr + (size_t)cv * 3 + 8 * (t - 136);
          cp_async16(dst + 16 * t, src, 16u);
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
                     :: "r"(smem_u32(cfull + cs)) : "memory");
      }
      cp_async_wait_all();   // no copy in flight when the warp exits
      return;
    }
    if (warp >= Cfg::kConvWarp0 && warp < Cfg::kConvWarp0 + kFConvWarps) {
      // Conv warps: channel t of the unit (q 0-127, k 128-255, v 256-319).
      const int t = tid - Cfg::kConvWarp0 * 32;
      const int blk = t < 128 ? 0 : (t < 256 ? 1 : 2);
      const int c = t - 128 * blk;
      const int offx = blk == 0 ? kFxQ : (blk == 1 ? kFxK : kFxV);
      const int offs = blk == 0 ? kFsQ : (blk == 1 ? kFsK : kFsV);
      // y slot: k 0-255, q 256-511, v 512-639 (BF16)
      const int offy = blk == 0 ? 256 : (blk == 1 ? 0 : 512);
      for (int i = 0; i < my_units; ++i) {
        const int cs = i % kFSlots, ys = i % kFYSlots;
        int n, h, g, part;
        unit_coords(blockIdx.x + i * G, n, h, g, part);
        const int cg = blk == 0 ? g * 128 + c
                                : (blk == 1 ? p.Hk * 128 + g * 128 + c
                                            : 2 * p.Hk * 128 + h * 128 + part * kDecRows + c);
        // taps 0-3 and bias of global channel cg (issued before the wait)
        const uint2 wu = __ldg(reinterpret_cast<const uint2*>(p.w) + cg);
        const float bias = p.bias ? __bfloat162float(p.bias[cg]) : 0.f;
        if (!mbar_wait_abortable(cfull + cs, (i / kFSlots) & 1, abort, 64)) break;
        const unsigned char* cslot = sm + Cfg::kConvOff + cs * kFSlot;
        const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(cslot + offx);
        const __nv_bfloat16* ss = reinterpret_cast<const __nv_bfloat16*>(cslot + offs);
        const __nv_bfloat16 s1 = ss[3 * c + 1], s2 = ss[3 * c + 2], xbf = xs[c];
        float acc = bias;
        acc = fmaf(bf16lo(wu.x), __bfloat162float(ss[3 * c]), acc);
        acc = fmaf(bf16hi(wu.x), __bfloat162float(s1), acc);
        acc = fmaf(bf16lo(wu.y), __bfloat162float(s2), acc);
        acc = fmaf(bf16hi(wu.y), __bfloat162float(xbf), acc);
        const __nv_bfloat16 y = __float2bfloat16_rn(p.silu ? silu_f(acc) : acc);
        __syncwarp();
        if (lane == 0)   // this warp's conv inputs are read
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(cempty + cs)) : "memory");
        // New state (s1, s2, x): v channels by every unit, q / k channels by
        // one unit per (sequence, q/k head).
        if (blk == 2 || (part == 0 && h % ratio == 0)) {
          __nv_bfloat16* d = p.st_out + ((size_t)n * p.C + cg) * 3;
          d[0] = s1;
          d[1] = s2;
          d[2] = xbf;
        }
        // The y slot is free once the compute warps have read its previous unit.
        if (i >= kFYSlots && !mbar_wait_abortable(yempty + ys, ((i / kFYSlots) - 1) & 1, abort, 64))
          break;
        reinterpret_cast<__nv_bfloat16*>(sm + Cfg::kYOff + ys * kFYSlot + offy)[c] = y;
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(yfull + ys)) : "memory");
      }
      return;
    }
  }

  if (warp == Cfg::kProdWarp) {
    // State producer (lane 0 issues).
    if (lane == 0) {
      auto issue_load = [&](int i) {
        const int st = i % kDecStages;
        const int unit = blockIdx.x + i * G;
        unsigned char* dst = sm + st * kDecStageBytes;
        if constexpr (kFused) {
          mbar_arrive_expect_tx(full + st, kDecUnitBytes);   // k, q, v: the conv warps
          bulk_g2s(dst, p.S + (size_t)unit * kDecRows * 128, kDecUnitBytes, full + st);
        } else {
          int n, h, g, part;
          unit_coords(unit, n, h, g, part);
          const int slot = state_slot(p.slots, n);
          // a padding entry: no state rows (the stage's stale rows are updated
          // and discarded, nothing is stored)
          mbar_arrive_expect_tx(full + st, (slot >= 0 ? kDecUnitBytes : 0) + 256 + 256 + 2 * kDecRows);
          if (slot >= 0)
            bulk_g2s(dst, p.S + (((size_t)slot * Hv + h) * kDecUnitsPerHead + part) * kDecRows * 128,
                     kDecUnitBytes, full + st);
          bulk_g2s(dst + kDecOffK, p.k + n * p.qk_stride + (int64_t)g * 128, 256, full + st);
          bulk_g2s(dst + kDecOffQ, p.q + n * p.qk_stride + (int64_t)g * 128, 256, full + st);
          bulk_g2s(dst + kDecOffV, p.v + n * p.v_stride + (int64_t)h * 128 + part * kDecRows,
                   2 * kDecRows, full + st);
        }
      };
      int issued = 0;   // units whose loads have been issued: [0, issued)
      for (; issued < my_units && issued < kDecStages; ++issued) issue_load(issued);
      int i = 0;
      for (; i < my_units; ++i) {
        const int st = i % kDecStages;
        // The compute warps stopped (or another role gave up): store nothing
        // more, the unit's rows are not all updated.
        if (!mbar_wait_abortable(empty + st, (i / kDecStages) & 1, abort)) break;
        const int unit = blockIdx.x + i * G;
        int n, h, g, part;
        unit_coords(unit, n, h, g, part);
        const int slot = kFused ? n : state_slot(p.slots, n);
        if (slot >= 0) {
          bulk_s2g(p.S + (((size_t)slot * Hv + h) * kDecUnitsPerHead + part) * kDecRows * 128,
                   sm + st * kDecStageBytes, kDecUnitBytes);
          bulk_s2g(p.o + (size_t)unit * kDecRows, sm + st * kDecStageBytes + kDecOffO, 2 * kDecRows);
        }
        bulk_commit();
        // Refill the stage stored one unit ago (its store has had a unit's
        // time to read shared memory), keeping kDecStages - 1 loads in flight.
        if (i >= 1 && i - 1 + kDecStages < my_units) {
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          issue_load(i - 1 + kDecStages);
          issued = i + kDecStages;
        }
      }
      // The stores' shared-memory reads are done before the CTA exits; their
      // global writes complete with the grid.
      bulk_wait_read();
      // After an abort, units [i, issued) may still have loads landing in
      // their stages (distinct stages: fewer than kDecStages of them); their
      // phases are the latest armed ones, so waiting for them is exact.
      // Bounded, not abortable: no copy may be in flight when the CTA exits.
      for (int j = i; j < issued; ++j)
        if (!mbar_wait(full + j % kDecStages, (j / kDecStages) & 1))
          record_device_status(GDN_ERR_TIMEOUT);
    }
    return;
  }

  // Compute warps: rows 4 warp .. 4 warp + 3 of every unit; lane l holds
  // columns 4 l .. 4 l + 3.
  const bool gl = (p.flags & kFlagGateLogits) != 0;
  float a_nxt = 0.f, b_nxt = 0.f;
  if (my_units > 0) {
    a_nxt = __ldg(p.a + blockIdx.x / kDecUnitsPerHead);
    b_nxt = __ldg(p.b + blockIdx.x / kDecUnitsPerHead);
  }
  for (int i = 0; i < my_units; ++i) {
    const int st = i % kDecStages;
    const int unit = blockIdx.x + i * G;
    const float av = gate_decay(a_nxt, gl), bv = gate_write(b_nxt, gl);
    if (i + 1 < my_units) {
      a_nxt = __ldg(p.a + (unit + G) / kDecUnitsPerHead);
      b_nxt = __ldg(p.b + (unit + G) / kDecUnitsPerHead);
    }
    // Waiting warps back off, so they take no issue slots from the producer
    // warps on their sub-partition. A wait that gives up stops this warp: it
    // no longer arrives on "empty", so the producer stores nothing more.
    if (!mbar_wait_abortable(full + st, (i / kDecStages) & 1, abort, 32)) break;
    unsigned char* stage = sm + st * kDecStageBytes;
    uint2 ku, qu, vu;
    if constexpr (kFused) {
      // k, q, v from the conv warps' ring (BF16, as the unfused stage holds them)
      const int ys = i % kFYSlots;
      if (!mbar_wait_abortable(yfull + ys, (i / kFYSlots) & 1, abort, 32)) break;
      const unsigned char* yslot = sm + Cfg::kYOff + ys * kFYSlot;
      ku = reinterpret_cast<const uint2*>(yslot)[lane];
      qu = reinterpret_cast<const uint2*>(yslot + 256)[lane];
      vu = reinterpret_cast<const uint2*>(yslot + 512)[warp];
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(yempty + ys)) : "memory");
    } else {
      ku = reinterpret_cast<const uint2*>(stage + kDecOffK)[lane];
      qu = reinterpret_cast<const uint2*>(stage + kDecOffQ)[lane];
      vu = reinterpret_cast<const uint2*>(stage + kDecOffV)[warp];
    }
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
    if (p.flags & kFlagL2) {
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
                             void* o, int N, int Hk, int Hv, int flags, cudaStream_t st,
                             StateSlots slots) {
  using Cfg = DecodeCfg<DK, DV>;
  return check_launch(launch_pdl(
      delta_decode_kernel<DK, DV>, dim3(N * Hv), dim3(Cfg::kThreads), 0, st,
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qk_stride,
      static_cast<const __nv_bfloat16*>(v), v_stride, a, b, S, static_cast<__nv_bfloat16*>(o),
      Hk, Hv, flags, slots));
}

template <int DK>
gdn_status_t launch_decode_dv(int dv, const void* q, const void* k, int64_t qk_stride,
                              const void* v, int64_t v_stride, const float* a, const float* b,
                              float* S, void* o, int N, int Hk, int Hv, int l2, cudaStream_t st,
                              StateSlots slots) {
  switch (dv) {
    case 16: return launch_decode_t<DK, 16>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st, slots);
    case 32: return launch_decode_t<DK, 32>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st, slots);
    case 64: return launch_decode_t<DK, 64>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st, slots);
    case 128: return launch_decode_t<DK, 128>(q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, l2, st, slots);
  }
  return GDN_ERR_UNSUPPORTED;
}

int decode_sm_count() {
  static const int n = [] {
    int dev = 0, c = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(delta_decode_stream_kernel<false>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, DecStage<false>::kSmem);
    cudaFuncSetAttribute(delta_decode_stream_kernel<true>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, DecStage<true>::kSmem);
    return c > 0 ? c : 1;
  }();
  return n;
}

template <bool kFused>
gdn_status_t launch_decode_stream(const DecodeArgs& p, cudaStream_t st) {
  const int sms = decode_sm_count();
  const int grid = p.units < sms ? p.units : sms;
  return check_launch(launch_pdl(delta_decode_stream_kernel<kFused>, dim3(grid),
                                dim3(DecStage<kFused>::kThreads), DecStage<kFused>::kSmem, st, p));
}

}  // namespace

gdn_status_t launch_decode_fused(const void* x, int64_t x_stride, const void* w,
                                 const void* bias, const void* st_in, void* st_out,
                                 const float* a, const float* b, float* S, void* o, int32_t N,
                                 int32_t Hk, int32_t Hv, int32_t silu, int32_t flags,
                                 cudaStream_t st) {
  DecodeArgs p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w = static_cast<const __nv_bfloat16*>(w);
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.st_in = static_cast<const __nv_bfloat16*>(st_in);
  p.st_out = static_cast<__nv_bfloat16*>(st_out);
  p.x_stride = x_stride;
  p.C = 2 * Hk * 128 + Hv * 128;
  p.silu = silu;
  p.a = a;
  p.b = b;
  p.S = S;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.Hk = Hk;
  p.Hv = Hv;
  p.flags = flags;
  p.units = N * Hv * kDecUnitsPerHead;
  return launch_decode_stream<true>(p, st);
}

gdn_status_t launch_delta_decode(const void* q, const void* k, int64_t qk_stride,
                                 const void* v, int64_t v_stride, const float* a,
                                 const float* b, float* S, void* o, int32_t N, int32_t Hk,
                                 int32_t Hv, int32_t dk, int32_t dv, int32_t flags,
                                 cudaStream_t st, StateSlots slots) {
  if (dk == 128 && dv == 128) {
    DecodeArgs p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.qk_stride = qk_stride;
    p.v_stride = v_stride;
    p.a = a;
    p.b = b;
    p.S = S;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.Hk = Hk;
    p.Hv = Hv;
    p.flags = flags;
    p.units = N * Hv * kDecUnitsPerHead;
    p.slots = slots;
    return launch_decode_stream<false>(p, st);
  }
  switch (dk) {
    case 16: return launch_decode_dv<16>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, flags, st, slots);
    case 32: return launch_decode_dv<32>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, flags, st, slots);
    case 64: return launch_decode_dv<64>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, flags, st, slots);
    case 128: return launch_decode_dv<128>(dv, q, k, qk_stride, v, v_stride, a, b, S, o, N, Hk, Hv, flags, st, slots);
  }
  return GDN_ERR_UNSUPPORTED;
}

GDN_DEFINE_STATUS_GATHER(gather_status_decode)

}  // namespace gdn
