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
// 9 flops and one SiLU). The prefill is a persistent stream: one CTA per SM
// walks a contiguous run of descriptors for one 2048-channel block, a producer
// warp keeps up to 192 KB of token rows in flight with bulk copies into a ring
// of shared-memory stages, and the compute warps convolve each stage from
// shared memory (the window of a continuing descriptor stays in registers).
// The whole-sequence mapping is the same kernel with one descriptor per
// sequence. The decode update keeps one thread per 8 channels.
#include <algorithm>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

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

// Buckets of the longest-first sequence order (chunk counts at or above the
// last bucket share it; the order only decides which sequences start first).
constexpr int kOrderBuckets = 1024;

// order[0 .. n): the sequences by descending chunk count (empty ones last; the
// order within one count is unspecified). A counting sort over chunk counts.
// `capacity` bounds every sequence's chunk count, so only that many buckets
// (at most kOrderBuckets) are used: a 2048-token step has about 36.
__device__ void longest_first_order(const int32_t* __restrict__ cu, int n, int chunk,
                                    int capacity, int32_t* __restrict__ order, int* s_hist,
                                    bool valid) {
  const int tid = threadIdx.x;
  if (!valid) {   // malformed offsets: any permutation will do (nothing runs)
    for (int s = tid; s < n; s += blockDim.x) order[s] = s;
    return;
  }
  const int nb = max(1, min(kOrderBuckets, capacity + 1));
  for (int b = tid; b < nb; b += blockDim.x) s_hist[b] = 0;
  __syncthreads();
  for (int s = tid; s < n; s += blockDim.x) {
    const int c = (cu[s + 1] - cu[s] + chunk - 1) / chunk;
    atomicAdd(&s_hist[min(max(c, 0), nb - 1)], 1);
  }
  __syncthreads();
  if (tid == 0) {   // start of each bucket, largest counts first
    int run = 0;
    for (int b = nb - 1; b >= 0; --b) {
      const int h = s_hist[b];
      s_hist[b] = run;
      run += h;
    }
  }
  __syncthreads();
  for (int s = tid; s < n; s += blockDim.x) {
    const int c = (cu[s + 1] - cu[s] + chunk - 1) / chunk;
    order[atomicAdd(&s_hist[min(max(c, 0), nb - 1)], 1)] = s;
  }
}

__global__ void __launch_bounds__(kBuildThreads)
build_chunks_kernel(const int32_t* __restrict__ cu, int n, int chunk,
                    gdn_conv_chunk_t* __restrict__ out, int capacity,
                    int32_t* __restrict__ num_chunks, int32_t* __restrict__ status,
                    int32_t* __restrict__ order) {
  __shared__ int s_off[kBuildThreads + 1];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ int s_bad;
  __shared__ unsigned long long s_count;
  __shared__ int s_hist[kOrderBuckets];
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
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
  if (order) longest_first_order(cu, n, chunk, capacity, order, s_hist, !s_bad);
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

// Prefill stream kernel. One CTA per SM: kCvGroups producer warps and
// kCvGroups groups of compute warps. The grid is NB channel blocks (kCvChan
// channels each) x R token groups; the CTA of (block cb, group r) owns
// descriptors [n r / R, n (r + 1) / R) of channel block cb. Every producer
// warp reads the CTA's descriptors up front (one per lane) and walks the same
// list of stages, kCvRows tokens each; stage i is posted by producer warp
// i % kCvGroups into that group's own ring of kCvSlotsPerGroup shared-memory
// stages, with bulk
// copies of the stage's rows, its 3-token halo (the 3 rows before it, or the
// initial conv_state at the start of a sequence) and, on the first stage of a
// sequence longer than the stage, the sequence's last 3 rows (the new
// conv_state). Several posting warps are needed because each mbarrier phase
// costs a posting thread a fixed time of the order of a few 2 KB copies. Every
// stage is self-contained, and stage i goes to compute group i % kCvGroups: a
// thread convolves 8 channels from shared memory (taps in registers, 16-byte
// loads and stores) and the group hands the stage back. No compute warp
// touches global memory except to store y and the new conv_state, so no load
// latency sits on the compute path.
constexpr int kCvGroups = 3;
constexpr int kCvGroupWarps = 8;
constexpr int kCvCpt = 4;                                // channels per compute thread
constexpr int kCvComputeWarps = kCvGroups * kCvGroupWarps;
constexpr int kCvThreads = (kCvComputeWarps + kCvGroups) * 32;   // + producer warps
constexpr int kCvChan = kCvGroupWarps * 32 * kCvCpt;     // 1024 channels per CTA
constexpr int kCvRows = 8;                               // tokens per stage
constexpr int kCvSlot = kCvChan * 2;                     // one token's row segment (bytes)
constexpr int kCvHalo = 0, kCvData = 3, kCvTail = 3 + kCvRows;   // slot indices
constexpr int kCvStageBytes = (3 + kCvRows + 3) * kCvSlot;        // 28 KB
// Each compute group has its own stages: a barrier is then only ever waited on
// by one group, for its next phase. (With stages shared round-robin between
// groups, a group that runs ahead can poll a barrier two phases before the one
// it wants, and a parity wait cannot tell those phases apart.)
constexpr int kCvSlotsPerGroup = 2;
constexpr int kCvStages = kCvGroups * kCvSlotsPerGroup;
constexpr int kCvMetaOff = kCvStages * kCvStageBytes;
constexpr int kCvBarOff = kCvMetaOff + kCvStages * 32;
constexpr int kCvSmem = kCvBarOff + 2 * kCvStages * 8;
// Stage i: group i % kCvGroups, its use number u = i / kCvGroups, slot
// g kCvSlotsPerGroup + u % kCvSlotsPerGroup, phase u / kCvSlotsPerGroup.
__device__ __forceinline__ int cv_slot(int i) {
  return (i % kCvGroups) * kCvSlotsPerGroup + (i / kCvGroups) % kCvSlotsPerGroup;
}
__device__ __forceinline__ int cv_round(int i) { return (i / kCvGroups) / kCvSlotsPerGroup; }
// Stage flags.
constexpr int kHaloX = 1;        // halo slots hold x rows tok-3 .. tok-1
constexpr int kHaloState = 2;    // halo slots hold the initial conv_state [ch][3]
constexpr int kFirst = 4;        // first stage of a sequence: writes the new conv_state
constexpr int kTailRows = 8;     // tail slots hold the sequence's last 3 rows

// One token of 4 channels (2 pairs): y = act(bias + w0 x[-3] + w1 x[-2] +
// w2 x[-1] + w3 x[0]) with the window win = (x[-3], x[-2], x[-1]), which then
// shifts by one. The products accumulate in this order in float32.
template <bool kSilu>
__device__ __forceinline__ void conv_row(const uint2 u, __nv_bfloat16* yd,
                                         const float2 (&wf)[4][2], const float2 (&bf)[2],
                                         float2 (&win)[3][2]) {
  const uint32_t xw[2] = {u.x, u.y};
  uint32_t ow[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float2 xc = bf16x2_f2(xw[q]);
    float2 acc = fma2(wf[0][q], win[0][q], bf[q]);
    acc = fma2(wf[1][q], win[1][q], acc);
    acc = fma2(wf[2][q], win[2][q], acc);
    acc = fma2(wf[3][q], xc, acc);
    ow[q] = f2_bf16x2(kSilu ? silu2(acc) : acc);
    win[0][q] = win[1][q];
    win[1][q] = win[2][q];
    win[2][q] = xc;
  }
  *reinterpret_cast<uint2*>(yd) = make_uint2(ow[0], ow[1]);
}

// conv_state of 4 channels ([channel][3], 24 bytes, 8-byte aligned) <-> floats.
__device__ __forceinline__ void state4_from_words(const uint2 (&u)[3], float (&st)[3][4]) {
  const uint32_t wd[6] = {u[0].x, u[0].y, u[1].x, u[1].y, u[2].x, u[2].y};
#pragma unroll
  for (int e = 0; e < 12; ++e) {
    const uint32_t word = wd[e >> 1];
    st[e % 3][e / 3] = (e & 1) ? bf16hi(word) : bf16lo(word);
  }
}
__device__ __forceinline__ void store_state4(__nv_bfloat16* p, const float (&st)[3][4]) {
  uint32_t wd[6];
#pragma unroll
  for (int e = 0; e < 12; e += 2)
    wd[e >> 1] = pack_bf16x2(st[e % 3][e / 3], st[(e + 1) % 3][(e + 1) / 3]);
  uint2* sp = reinterpret_cast<uint2*>(p);
#pragma unroll
  for (int q = 0; q < 3; ++q) sp[q] = make_uint2(wd[2 * q], wd[2 * q + 1]);
}
// a[i][ch] for a runtime i in 0..2, without indexing a register array.
__device__ __forceinline__ float sel3_4(const float (&a)[3][4], int i, int ch) {
  return i == 0 ? a[0][ch] : (i == 1 ? a[1][ch] : a[2][ch]);
}

struct CvMeta {
  int seq, tok, rows, pos, flags, L, slot;
};

template <bool kSilu>
__global__ void __launch_bounds__(kCvThreads, 1)
conv_fwd_stream_kernel(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                       const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ bias,
                       __nv_bfloat16* __restrict__ state, const uint8_t* __restrict__ has_init,
                       const int32_t* __restrict__ cu, const gdn_conv_chunk_t* __restrict__ chunks,
                       const int32_t* __restrict__ num_chunks, int units, int T, int C, int N,
                       __nv_bfloat16* __restrict__ y, const StateSlots slots) {
  using namespace tc;
  extern __shared__ __align__(128) unsigned char sm[];
  CvMeta* meta = reinterpret_cast<CvMeta*>(sm + kCvMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kCvBarOff);
  uint64_t* empty = full + kCvStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NB = (C + kCvChan - 1) / kCvChan;
  const int R = gridDim.x / NB;
  const int cb = blockIdx.x % NB, grp = blockIdx.x / NB;
  const int c_base = cb * kCvChan;
  const int nch = min(kCvChan, C - c_base);
  if (tid == 0) {
    for (int st = 0; st < kCvStages; ++st) {
      mbar_init(full + st, 1);
      mbar_init(empty + st, kCvGroupWarps);
    }
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  if (warp >= kCvComputeWarps) {
    // Producer warp pw. Lanes fetch and validate 32 descriptors at a time;
    // lane 0 posts the stages i with i % kCvGroups == pw, then the end marker
    // (rows = -1) of compute group pw.
    const int pw = warp - kCvComputeWarps;
    // The split over token groups uses the capacity, so the count and the
    // descriptors load together; entries at or past the count are skipped.
    const int d0 = (int)(((int64_t)units * grp) / R);
    const int d1 = (int)(((int64_t)units * (grp + 1)) / R);
    const uint32_t seg = (uint32_t)nch * 2u;
    int it = 0;
    bool ok = true;
    auto post = [&](const CvMeta& m, uint32_t bytes, int st) {
      meta[st] = m;
      if (bytes)
        mbar_arrive_expect_tx(full + st, bytes);
      else
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(full + st))
                     : "memory");
    };
    for (int base = d0; base < d1 && ok; base += 32) {
      const int d = base + lane;
      int4 dd = make_int4(-1, 0, 0, 0);
      int L = 0, init = 0, slot = 0;
      if (d < d1) {
        int n;
        if (chunks) {
          n = __ldg(num_chunks);
          dd = __ldg(reinterpret_cast<const int4*>(chunks) + d);
        } else {
          n = N;
          const int t0 = __ldg(cu + d);
          dd = make_int4(d, t0, __ldg(cu + d + 1) - t0, 0);
        }
        const int seq = dd.x, tok0 = dd.y, len = dd.z, pos = dd.w;
        bool valid = d < n && seq >= 0 && seq < N && len > 0 && (pos == 0 || pos >= 3) &&
                     tok0 >= pos && (int64_t)tok0 + len <= T;
        if (valid) {
          slot = state_slot(slots, seq);   // padding entries are skipped
          valid = slot >= 0;
        }
        if (valid && pos == 0) {
          // Only the first descriptor of a sequence needs the sequence
          // length (for the new state) and the initial-state flag.
          L = __ldg(cu + seq + 1) - __ldg(cu + seq);
          init = has_init != nullptr && has_init[seq] != 0;
          // descriptors inconsistent with cu_seqlens are skipped
          if (L < len || (int64_t)tok0 + L > T) valid = false;
        }
        if (!valid) dd.x = -1;
      }
      const int cnt = min(32, d1 - base);
      for (int j = 0; j < cnt; ++j) {
        const int seq = __shfl_sync(0xffffffffu, dd.x, j);
        const int tok0 = __shfl_sync(0xffffffffu, dd.y, j);
        const int len = __shfl_sync(0xffffffffu, dd.z, j);
        const int pos = __shfl_sync(0xffffffffu, dd.w, j);
        const int Lj = __shfl_sync(0xffffffffu, L, j);
        const int initj = __shfl_sync(0xffffffffu, init, j);
        const int slotj = __shfl_sync(0xffffffffu, slot, j);
        if (seq < 0) continue;
        if (lane == 0) {
          for (int r0 = 0; r0 < len && ok; r0 += kCvRows, ++it) {
            if (it % kCvGroups != pw) continue;
            const int st = cv_slot(it), rd = cv_round(it);
            if (rd > 0 && !mbar_wait_sleep(empty + st, (rd - 1) & 1, 128)) {
              record_device_status(GDN_ERR_TIMEOUT);   // the compute group stopped
              ok = false;
              break;
            }
            CvMeta m;
            m.seq = seq;
            m.tok = tok0 + r0;
            m.rows = min(kCvRows, len - r0);
            m.pos = pos + r0;
            m.L = Lj;
            m.slot = slotj;
            m.flags = 0;
            unsigned char* dst = sm + st * kCvStageBytes;
            const __nv_bfloat16* xr = x + (int64_t)m.tok * x_stride + c_base;
            uint32_t bytes = (uint32_t)m.rows * seg;
            if (m.pos >= 3) {
              m.flags |= kHaloX;
              bytes += 3 * seg;
            } else if (initj) {
              m.flags |= kHaloState;
              bytes += 3 * seg;
            }
            if (m.pos == 0) {
              m.flags |= kFirst;
              if (Lj > m.rows) {
                m.flags |= kTailRows;
                bytes += 3 * seg;
              }
            }
            post(m, bytes, st);
            for (int i = 0; i < m.rows; ++i)
              bulk_g2s(dst + (kCvData + i) * kCvSlot, xr + (int64_t)i * x_stride, seg, full + st);
            if (m.flags & kHaloX) {
              for (int i = 0; i < 3; ++i)
                bulk_g2s(dst + (kCvHalo + i) * kCvSlot, xr - (int64_t)(3 - i) * x_stride, seg,
                         full + st);
            } else if (m.flags & kHaloState) {
              bulk_g2s(dst + kCvHalo * kCvSlot, state + ((size_t)slotj * C + c_base) * 3, 3 * seg,
                       full + st);
            }
            if (m.flags & kTailRows) {
              const __nv_bfloat16* xt = x + (int64_t)(tok0 + Lj - 3) * x_stride + c_base;
              for (int i = 0; i < 3; ++i)
                bulk_g2s(dst + (kCvTail + i) * kCvSlot, xt + (int64_t)i * x_stride, seg,
                         full + st);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        it = __shfl_sync(0xffffffffu, it, 0);
      }
    }
    if (lane == 0 && ok) {
      while (it % kCvGroups != pw) ++it;
      const int st = cv_slot(it), rd = cv_round(it);
      if (rd == 0 || mbar_wait_sleep(empty + st, (rd - 1) & 1, 128)) {
        CvMeta m;
        m.rows = -1;
        post(m, 0, st);
      } else {
        record_device_status(GDN_ERR_TIMEOUT);
      }
    }
    return;
  }

  // Compute group g = warp / kCvGroupWarps takes stages g, g + kCvGroups, ...
  const int g = warp / kCvGroupWarps;
  const int gt = tid - g * kCvGroupWarps * 32;   // 0 .. 255
  const int c0 = c_base + gt * kCvCpt;
  const bool active = gt * kCvCpt < nch;
  float2 wf[4][2], bf[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    bf[q] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) wf[j][q] = make_float2(0.f, 0.f);
  }
  if (active) {
    // w is [C, 4]: 4 channels x 4 taps = 32 contiguous bytes.
    const uint4 w01 = ldg16(w + (size_t)c0 * 4), w23 = ldg16(w + (size_t)c0 * 4 + 8);
    const uint32_t tw[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
    // word 2 ch + (j >> 1) holds taps j (even: low half) of channel ch
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a0 = tw[2 * (2 * q) + (j >> 1)], a1 = tw[2 * (2 * q + 1) + (j >> 1)];
        wf[j][q] = (j & 1) ? make_float2(bf16hi(a0), bf16hi(a1)) : make_float2(bf16lo(a0), bf16lo(a1));
      }
    if (bias) {
      const uint2 bu = *reinterpret_cast<const uint2*>(bias + c0);
      bf[0] = bf16x2_f2(bu.x);
      bf[1] = bf16x2_f2(bu.y);
    }
  }
  for (int it = g;; it += kCvGroups) {
    const int st = cv_slot(it);
    // A wait that gives up (the producer stopped) ends the stream; only stages
    // whose copies have all landed are ever computed and stored.
    if (!mbar_wait_sleep(full + st, cv_round(it) & 1)) {
      record_device_status(GDN_ERR_TIMEOUT);
      break;
    }
    const CvMeta m = meta[st];
    if (m.rows < 0) break;
    const unsigned char* stage = sm + st * kCvStageBytes;
    if (active) {
      // Window slot j holds sequence position m.pos - 3 + j: an x row from the
      // halo slots, else the initial state (slot p + 3) or zero.
      float2 win[3][2];
      float sv[3][4];
      if (m.flags & kHaloState) {
        const uint2* sp = reinterpret_cast<const uint2*>(stage + kCvHalo * kCvSlot + gt * 24);
        const uint2 su[3] = {sp[0], sp[1], sp[2]};
        state4_from_words(su, sv);
      } else {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) sv[0][ch] = sv[1][ch] = sv[2][ch] = 0.f;
      }
      if (m.flags & kHaloX) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const uint2 u = *reinterpret_cast<const uint2*>(stage + (kCvHalo + j) * kCvSlot + gt * 8);
          win[j][0] = bf16x2_f2(u.x);
          win[j][1] = bf16x2_f2(u.y);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
          for (int q = 0; q < 2; ++q) win[j][q] = make_float2(sv[j][2 * q], sv[j][2 * q + 1]);
      }
      if (m.flags & kFirst) {
        // The first stage of a sequence is the only reader of the old state,
        // so it also writes the new one: the last 3 entries of (old ++ x_seq).
        float ns[3][4];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int p = m.L - 3 + j;
          if (p < 0) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) ns[j][ch] = sel3_4(sv, p + 3, ch);
          } else {
            const int slot = (m.flags & kTailRows) ? kCvTail + j : kCvData + p;
            const uint2 u = *reinterpret_cast<const uint2*>(stage + slot * kCvSlot + gt * 8);
            ns[j][0] = bf16lo(u.x);
            ns[j][1] = bf16hi(u.x);
            ns[j][2] = bf16lo(u.y);
            ns[j][3] = bf16hi(u.y);
          }
        }
        store_state4(state + ((size_t)m.slot * C + c0) * 3, ns);
      }
      const unsigned char* src = stage + kCvData * kCvSlot + gt * 8;
      __nv_bfloat16* dst = y + (int64_t)m.tok * C + c0;
      if (m.rows == kCvRows) {
        // Full stage: all rows are read from shared memory before the first
        // store (so no load waits behind a store), then straight-line code
        // in which the window shifts by renaming.
        uint2 xr[kCvRows];
#pragma unroll
        for (int i = 0; i < kCvRows; ++i)
          xr[i] = *reinterpret_cast<const uint2*>(src + i * kCvSlot);
#pragma unroll
        for (int i = 0; i < kCvRows; ++i)
          conv_row<kSilu>(xr[i], dst + (int64_t)i * C, wf, bf, win);
      } else {
        for (int i = 0; i < m.rows; ++i)
          conv_row<kSilu>(*reinterpret_cast<const uint2*>(src + i * kCvSlot),
                          dst + (int64_t)i * C, wf, bf, win);
      }
    }
    __syncwarp();
    if (lane == 0)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(empty + st))
                   : "memory");
  }
}

// ---------------------------------------------------------------------------
// Conv decode update: one token per sequence.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kConvThreads)
conv_update_kernel(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                   const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ bias,
                   __nv_bfloat16* __restrict__ state, int C, int silu,
                   __nv_bfloat16* __restrict__ y, const StateSlots slots) {
  const int n = blockIdx.y;
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
  if (c0 < C) {
    // Warm L2 with this thread's taps, bias and state while the previous
    // kernel finishes.
    const int s0 = state_slot(slots, n);
    prefetch_l2(w + (size_t)c0 * 4);
    if (bias) prefetch_l2(bias + c0);
    if (s0 >= 0) {
      const __nv_bfloat16* sp = state + ((size_t)s0 * C + c0) * 3;
      prefetch_l2(sp);
      prefetch_l2(sp + 23);
    }
  }
  pdl_wait();
  pdl_trigger();
  const int slot = state_slot(slots, n);
  if (c0 >= C || slot < 0) return;
  float wf[4][8], bf[8], win[3][8], xc[8], out[8];
  __nv_bfloat16* st_row = state + ((size_t)slot * C + c0) * 3;
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
                                 int32_t* num_chunks, int32_t* status, cudaStream_t st,
                                 int32_t* order) {
  return check_launch(launch_pdl(build_chunks_kernel, dim3(1), dim3(kBuildThreads), 0, st, cu, n,
                                chunk_tokens, chunks, capacity, num_chunks, status, order));
}

gdn_status_t launch_conv_fwd(const void* x, int64_t x_stride, const void* w, const void* bias,
                             void* conv_state, const uint8_t* has_init, const int32_t* cu,
                             const gdn_conv_chunk_t* chunks, const int32_t* num_chunks,
                             int32_t units, int32_t T, int32_t C, int32_t N, int32_t silu,
                             void* y, cudaStream_t st, StateSlots slots) {
  if (units <= 0) return GDN_OK;
  static const int num_sms = [] {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(conv_fwd_stream_kernel<true>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, kCvSmem);
    cudaFuncSetAttribute(conv_fwd_stream_kernel<false>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, kCvSmem);
    return n > 0 ? n : 1;
  }();
  const int NB = (C + kCvChan - 1) / kCvChan;
  const int R = std::max(1, std::min(num_sms / NB, (int)units));
  auto kern = silu ? conv_fwd_stream_kernel<true> : conv_fwd_stream_kernel<false>;
  return check_launch(launch_pdl(
      kern, dim3(NB * R), dim3(kCvThreads), kCvSmem, st, static_cast<const __nv_bfloat16*>(x),
      x_stride, static_cast<const __nv_bfloat16*>(w), static_cast<const __nv_bfloat16*>(bias),
      static_cast<__nv_bfloat16*>(conv_state), has_init, cu, chunks, num_chunks, (int)units,
      (int)T, (int)C, (int)N, static_cast<__nv_bfloat16*>(y), slots));
}

gdn_status_t launch_conv_update(const void* x, int64_t x_stride, const void* w,
                                const void* bias, void* conv_state, int32_t N, int32_t C,
                                int32_t silu, void* y, cudaStream_t st, StateSlots slots) {
  dim3 grid((C / 8 + kConvThreads - 1) / kConvThreads, N);
  return check_launch(launch_pdl(
      conv_update_kernel, grid, dim3(kConvThreads), 0, st, static_cast<const __nv_bfloat16*>(x),
      x_stride, static_cast<const __nv_bfloat16*>(w), static_cast<const __nv_bfloat16*>(bias),
      static_cast<__nv_bfloat16*>(conv_state), (int)C, (int)silu,
      static_cast<__nv_bfloat16*>(y), slots));
}

GDN_DEFINE_STATUS_GATHER(gather_status_conv)

}  // namespace gdn
