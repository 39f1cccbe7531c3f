// Exact (sequence, chunk) descriptors and the width-4 depthwise causal conv1d
// (prefill over descriptors, and the single-token decode update).
//
// Sources: "perf(gdn): dispatch exact causal-conv chunks", What changed (one
// descriptor per (sequence, 8-token chunk), built once per step and reused by
// every layer; one conv program per descriptor; whole-sequence mapping kept as
// a rollback) and "RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs
// vLLM", Existing evidence (K=4 specialisation of the conv).
//
// GB300 mapping: the conv is HBM-bound (2 bytes in and 2 bytes out per element,
// 9 flops). In the prefill one thread owns 4 channels (an 8-byte vector) of one
// descriptor, keeps its taps and the 3-token window packed in registers,
// issues all of the descriptor's row loads before computing, and writes 8-byte
// vectors; a CTA covers 512 channels of one descriptor, so the 2048 x 8192
// prefill is 4096 small CTAs, about two resident waves on 152 SMs. The decode
// update keeps one thread per 8 channels.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;  // x 8 channels = 1024 channels per CTA
constexpr int kBuildThreads = 1024;

// ---------------------------------------------------------------------------
// Descriptor builder: one CTA. Validates cu_seqlens, checks the capacity, then
// walks the sequences in tiles of 1024: per tile, ceil(L / chunk) counts, a
// block-wide exclusive scan, and one thread per output descriptor (located by
// binary search over the tile's offsets).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int wv = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
    int winc = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += t;
    }
    s_warp[lane] = winc - wv;  // exclusive warp offsets
    if (lane == 31) *total = winc;
  }
  __syncthreads();
  int r = s_warp[warp] + inc - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kBuildThreads)
build_chunks_kernel(const int32_t* __restrict__ cu, int n, int chunk,
                    gdn_conv_chunk_t* __restrict__ out, int capacity,
                    int32_t* __restrict__ num_chunks, int32_t* __restrict__ status) {
  __shared__ int s_off[kBuildThreads + 1];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ int s_bad;
  __shared__ unsigned long long s_count;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (cu[0] != 0);
    s_count = 0;
  }
  __syncthreads();
  // Pass 1: validation and the total count.
  unsigned long long my = 0;
  bool bad = false;
  for (int s = tid; s < n; s += blockDim.x) {
    int L = cu[s + 1] - cu[s];
    if (L < 0) bad = true;
    else my += (unsigned long long)((L + chunk - 1) / chunk);
  }
  if (bad) atomicOr(&s_bad, 1);
  if (my) atomicAdd(&s_count, my);
  __syncthreads();
  if (s_bad || s_count > (unsigned long long)capacity) {
    if (tid == 0) {
      *num_chunks = 0;
      if (status) *status = s_bad ? GDN_ERR_INVALID_ARG : GDN_ERR_WORKSPACE;
    }
    return;
  }
  // Pass 2: emit descriptors, tile by tile.
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int s = base + tid;
    int L = (s < n) ? cu[s + 1] - cu[s] : 0;
    int cnt = (L + chunk - 1) / chunk;
    int off = block_exclusive_scan(cnt, s_warp, &s_total);
    s_off[tid] = off;
    if (tid == 0) s_off[blockDim.x] = s_total;
    __syncthreads();
    const int tile_total = s_off[blockDim.x];
    for (int i = tid; i < tile_total; i += blockDim.x) {
      // last j with s_off[j] <= i (that sequence is non-empty)
      int lo = 0, hi = blockDim.x - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const int seq = base + lo;
      const int local = i - s_off[lo];
      const int start = cu[seq];
      const int Ls = cu[seq + 1] - start;
      int4 d;
      d.x = seq;
      d.y = start + local * chunk;
      d.z = min(chunk, Ls - local * chunk);
      d.w = local * chunk;
      reinterpret_cast<int4*>(out)[carry + i] = d;
    }
    carry += tile_total;
    __syncthreads();
  }
  if (tid == 0) {
    *num_chunks = carry;
    if (status) *status = GDN_OK;
  }
}

// ---------------------------------------------------------------------------
// Conv prefill. Unit = one descriptor (kChunks) or one whole sequence.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load_taps(const __nv_bfloat16* __restrict__ w, int c0,
                                          float (&wf)[4][8]) {
  // w is [C, 4]: the 8 channels of this thread are 64 contiguous bytes.
  const uint4* wp = reinterpret_cast<const uint4*>(w + (size_t)c0 * 4);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u = ldg16(wp + q);  // channels 2q and 2q+1, taps 0..3 each
    wf[0][2 * q] = bf16lo(u.x);
    wf[1][2 * q] = bf16hi(u.x);
    wf[2][2 * q] = bf16lo(u.y);
    wf[3][2 * q] = bf16hi(u.y);
    wf[0][2 * q + 1] = bf16lo(u.z);
    wf[1][2 * q + 1] = bf16hi(u.z);
    wf[2][2 * q + 1] = bf16lo(u.w);
    wf[3][2 * q + 1] = bf16hi(u.w);
  }
}

// conv_state row of 8 channels: 24 BF16 (48 bytes) laid out [channel][3].
__device__ __forceinline__ void load_state8(const __nv_bfloat16* p, float (&st)[3][8]) {
  const uint4* sp = reinterpret_cast<const uint4*>(p);
  uint32_t wd[12];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    uint4 u = *(sp + q);
    wd[4 * q] = u.x; wd[4 * q + 1] = u.y; wd[4 * q + 2] = u.z; wd[4 * q + 3] = u.w;
  }
#pragma unroll
  for (int e = 0; e < 24; ++e) {
    uint32_t word = wd[e >> 1];
    st[e % 3][e / 3] = (e & 1) ? bf16hi(word) : bf16lo(word);
  }
}

__device__ __forceinline__ void store_state8(__nv_bfloat16* p, const float (&st)[3][8]) {
  uint32_t wd[12];
#pragma unroll
  for (int e = 0; e < 24; e += 2)
    wd[e >> 1] = pack_bf16x2(st[e % 3][e / 3], st[(e + 1) % 3][(e + 1) / 3]);
  uint4* sp = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int q = 0; q < 3; ++q) sp[q] = make_uint4(wd[4 * q], wd[4 * q + 1], wd[4 * q + 2], wd[4 * q + 3]);
}

// Element c (0..3) of 4 BF16 values packed in an 8-byte vector, as float.
__device__ __forceinline__ float elt4(const uint2& u, int c) {
  const uint32_t w = c < 2 ? u.x : u.y;
  return (c & 1) ? bf16hi(w) : bf16lo(w);
}

__device__ __forceinline__ uint2 ldg8(const void* p) {
  return __ldg(reinterpret_cast<const uint2*>(p));
}

// Prefill: one thread owns 4 channels (8-byte vectors) of one unit. The taps
// (4 channels x 4 taps, two 16-byte vectors), bias and the 3-token window stay
// packed as BF16 and are converted on use, so a thread needs few registers
// while it keeps all of a descriptor's rows in flight.
template <bool kChunks>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_kernel(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ bias,
                __nv_bfloat16* __restrict__ state, const uint8_t* __restrict__ has_init,
                const int32_t* __restrict__ cu, const gdn_conv_chunk_t* __restrict__ chunks,
                const int32_t* __restrict__ num_chunks, int T, int C, int N, int silu,
                __nv_bfloat16* __restrict__ y) {
  const int unit = blockIdx.x;
  int seq, tok0, len, pos;
  if (kChunks) {
    if (unit >= __ldg(num_chunks)) return;
    const int4 d = __ldg(reinterpret_cast<const int4*>(chunks) + unit);
    seq = d.x; tok0 = d.y; len = d.z; pos = d.w;
  } else {
    seq = unit; tok0 = __ldg(cu + unit); len = __ldg(cu + unit + 1) - tok0; pos = 0;
  }
  if (seq < 0 || seq >= N || len <= 0 || pos < 0 || tok0 < pos || (int64_t)tok0 + len > T) return;
  const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * 4;
  if (c0 >= C) return;

  // w[c0 .. c0+3][0..3]: 32 contiguous bytes.
  const uint4 w01 = ldg16(w + (size_t)c0 * 4), w23 = ldg16(w + (size_t)c0 * 4 + 8);
  auto tap = [&](int c, int j) {
    const uint4& u = c < 2 ? w01 : w23;
    const uint32_t wd = (c & 1) ? (j < 2 ? u.z : u.w) : (j < 2 ? u.x : u.y);
    return (j & 1) ? bf16hi(wd) : bf16lo(wd);
  };
  const uint2 bq = bias ? ldg8(bias + c0) : make_uint2(0, 0);

  // Window of the 3 tokens before the unit: slot j holds sequence position
  // pos - 3 + j (from x when >= 0, else from the initial state or zero).
  const bool init = has_init != nullptr && has_init[seq] != 0;
  __nv_bfloat16* st_row = state + ((size_t)seq * C + c0) * 3;   // 12 BF16: [channel][3]
  uint2 win[3] = {make_uint2(0, 0), make_uint2(0, 0), make_uint2(0, 0)};
  if (pos < 3 && init) {
    const uint2* sp = reinterpret_cast<const uint2*>(st_row);
    const uint2 s0 = sp[0], s1 = sp[1], s2 = sp[2];
    const uint32_t wd[6] = {s0.x, s0.y, s1.x, s1.y, s2.x, s2.y};
    float sv[3][4];
#pragma unroll
    for (int e = 0; e < 12; ++e) sv[e % 3][e / 3] = (e & 1) ? bf16hi(wd[e >> 1]) : bf16lo(wd[e >> 1]);
#pragma unroll
    for (int j = 0; j < 3; ++j)
      win[j] = make_uint2(pack_bf16x2(sv[j][0], sv[j][1]), pack_bf16x2(sv[j][2], sv[j][3]));
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    if (pos - 3 + j >= 0) win[j] = ldg8(x + (size_t)(tok0 - 3 + j) * x_stride + c0);
  }

  // The unit that starts the sequence is the only reader of the old state, so
  // it also writes the new one: the last 3 entries of (old state ++ x_seq).
  if (pos == 0) {
    const int L = kChunks ? (__ldg(cu + seq + 1) - __ldg(cu + seq)) : len;
    if (L < len || (int64_t)tok0 + L > T) return;  // descriptors inconsistent with cu_seqlens
    uint2 ns[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int p = L - 3 + j;
      ns[j] = p >= 0 ? ldg8(x + (size_t)(tok0 + p) * x_stride + c0)
                     : ((p == -3) ? win[0] : ((p == -2) ? win[1] : win[2]));
    }
    float nv[12];
#pragma unroll
    for (int e = 0; e < 12; ++e) nv[e] = elt4(ns[e % 3], e / 3);   // [channel][3] order
    uint2* sp = reinterpret_cast<uint2*>(st_row);
#pragma unroll
    for (int q = 0; q < 3; ++q)
      sp[q] = make_uint2(pack_bf16x2(nv[4 * q], nv[4 * q + 1]), pack_bf16x2(nv[4 * q + 2], nv[4 * q + 3]));
  }

  for (int base = 0; base < len; base += 8) {
    const int cnt = min(8, len - base);
    uint2 xr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < cnt) xr[i] = ldg8(x + (size_t)(tok0 + base + i) * x_stride + c0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < cnt) {
        float out[4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          float acc = elt4(bq, ch);
          acc = fmaf(tap(ch, 0), elt4(win[0], ch), acc);
          acc = fmaf(tap(ch, 1), elt4(win[1], ch), acc);
          acc = fmaf(tap(ch, 2), elt4(win[2], ch), acc);
          acc = fmaf(tap(ch, 3), elt4(xr[i], ch), acc);
          out[ch] = silu ? silu_f(acc) : acc;
        }
        win[0] = win[1];
        win[1] = win[2];
        win[2] = xr[i];
        *reinterpret_cast<uint2*>(y + (size_t)(tok0 + base + i) * C + c0) =
            make_uint2(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Conv decode update: one token per sequence.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kConvThreads)
conv_update_kernel(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                   const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ bias,
                   __nv_bfloat16* __restrict__ state, int C, int silu,
                   __nv_bfloat16* __restrict__ y) {
  const int n = blockIdx.y;
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
  if (c0 >= C) return;
  float wf[4][8], bf[8], win[3][8], xc[8], out[8];
  __nv_bfloat16* st_row = state + ((size_t)n * C + c0) * 3;
  const uint4 xv = ldg16(x + (size_t)n * x_stride + c0);
  load_state8(st_row, win);
  load_taps(w, c0, wf);
  if (bias) {
    unpack8(ldg16(bias + c0), bf);
  } else {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) bf[ch] = 0.f;
  }
  unpack8(xv, xc);
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    float acc = bf[ch];
    acc = fmaf(wf[0][ch], win[0][ch], acc);
    acc = fmaf(wf[1][ch], win[1][ch], acc);
    acc = fmaf(wf[2][ch], win[2][ch], acc);
    acc = fmaf(wf[3][ch], xc[ch], acc);
    out[ch] = silu ? silu_f(acc) : acc;
    win[0][ch] = win[1][ch];
    win[1][ch] = win[2][ch];
    win[2][ch] = xc[ch];
  }
  *reinterpret_cast<uint4*>(y + (size_t)n * C + c0) = pack8(out);
  store_state8(st_row, win);
}

}  // namespace

gdn_status_t launch_build_chunks(const int32_t* cu, int32_t n, int32_t chunk_tokens,
                                 gdn_conv_chunk_t* chunks, int32_t capacity,
                                 int32_t* num_chunks, int32_t* status, cudaStream_t st) {
  build_chunks_kernel<<<1, kBuildThreads, 0, st>>>(cu, n, chunk_tokens, chunks, capacity,
                                                   num_chunks, status);
  return check_launch();
}

gdn_status_t launch_conv_fwd(const void* x, int64_t x_stride, const void* w, const void* bias,
                             void* conv_state, const uint8_t* has_init, const int32_t* cu,
                             const gdn_conv_chunk_t* chunks, const int32_t* num_chunks,
                             int32_t units, int32_t T, int32_t C, int32_t N, int32_t silu,
                             void* y, cudaStream_t st) {
  if (units <= 0) return GDN_OK;
  dim3 grid(units, (C / 4 + kConvThreads - 1) / kConvThreads);
  auto xp = static_cast<const __nv_bfloat16*>(x);
  auto wp = static_cast<const __nv_bfloat16*>(w);
  auto bp = static_cast<const __nv_bfloat16*>(bias);
  auto sp = static_cast<__nv_bfloat16*>(conv_state);
  auto yp = static_cast<__nv_bfloat16*>(y);
  if (chunks)
    conv_fwd_kernel<true><<<grid, kConvThreads, 0, st>>>(xp, x_stride, wp, bp, sp, has_init, cu,
                                                         chunks, num_chunks, T, C, N, silu, yp);
  else
    conv_fwd_kernel<false><<<grid, kConvThreads, 0, st>>>(xp, x_stride, wp, bp, sp, has_init, cu,
                                                          nullptr, nullptr, T, C, N, silu, yp);
  return check_launch();
}

gdn_status_t launch_conv_update(const void* x, int64_t x_stride, const void* w,
                                const void* bias, void* conv_state, int32_t N, int32_t C,
                                int32_t silu, void* y, cudaStream_t st) {
  dim3 grid((C / 8 + kConvThreads - 1) / kConvThreads, N);
  conv_update_kernel<<<grid, kConvThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), x_stride, static_cast<const __nv_bfloat16*>(w),
      static_cast<const __nv_bfloat16*>(bias), static_cast<__nv_bfloat16*>(conv_state), C, silu,
      static_cast<__nv_bfloat16*>(y));
  return check_launch();
}

}  // namespace gdn
