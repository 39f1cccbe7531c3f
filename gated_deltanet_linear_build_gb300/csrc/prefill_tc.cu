// Chunked prefill of the gated delta rule on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM), head dimension 128.
//
// The chunk algebra is the one described in prefill.cu. Everything is laid out
// so that every product has M = 128 (the head dimension) and K-major operands:
//
//   chunk kernel, one CTA per (64-token chunk, v-head):
//     G    = [K; Q] K^T                        (M=128: K rows then Q rows, N=64, K=128)
//     A_rs = b_r e^{g_r-g_s} (k_r.k_s), P_rs = e^{g_r-g_s} (q_r.k_s)     (CUDA cores)
//     Tm   = (I + A)^{-1}: one column per thread, forward substitution  (CUDA cores)
//     W^T  = K^T (Tm diag(b e^g))^T,  U^T = V^T (Tm diag(b))^T          (M=128, N=64, K=64)
//   and writes, per (chunk, v-head), a record with W (BF16 hi + lo), P, the
//   scaled queries e^{g_r} q_r, K^T (all in the tile layout the state kernel
//   feeds straight to the tensor core), U (float32) and g.
//
//   state kernel, one CTA per (sequence, v-head), S [dv=128 x dk=128] float32
//   resident in TMEM, chunks in order:
//     X^T  = S W^T                  (S and W split into BF16 hi + lo: 3 MMAs)
//     O^T  = S (e^g Q)^T            (single BF16: the output is BF16)
//     Delta^T = U^T - X^T           (CUDA cores, lane i holds row i)
//     O^T += Delta^T P^T            (single BF16)
//     S    = e^{g_last} S + (Delta^T diag(e^{g_last-g}))  K   (Delta split: 2 MMAs,
//            accumulated onto the rescaled S in TMEM)
//
// Precision: the products that feed the float32 state carry a hi/lo BF16 split
// of their float32 operand (hi = bf16(x), lo = bf16(x - hi)), which keeps about
// 16 mantissa bits; K, Q and V are exact BF16 inputs. With the optional q/k L2
// norm, the per-row factors are folded into the float32 side (A, P, Tm scaling,
// the Delta scaling and e^g Q) so that K stays exact in every product.
//
// Bounded waits: every mbarrier wait gives up after about two seconds, records
// GDN_ERR_TIMEOUT in workspace word 2 and unwinds (TMEM is always released).
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kC = 64;     // chunk tokens
constexpr int kD = 128;    // head dim (dk = dv)
constexpr int kThreads = 128;

// Record of one (chunk, v-head) written by the chunk kernel.
constexpr int kOffWhi = 0;          // W hi   [64 r][128 j] tile
constexpr int kOffWlo = 16384;      // W lo
constexpr int kOffP = 32768;        // P      [64 r][64 s] tile
constexpr int kOffGQ = 40960;       // e^g q  [64 r][128 j] tile
constexpr int kOffKT = 57344;       // K^T    [128 j][64 s] tile
constexpr int kTileBytes = 73728;   // the five tiles above, contiguous
constexpr int kOffU = 73728;        // U      [128 i][64 r] float32 rows
constexpr int kOffGK = 106496;      // g[64], rk[64] float32
constexpr int kRecBytes = 107008;

__host__ __device__ constexpr size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

struct TcLayout {
  int capacity;
  size_t desc_off, rec_off, total;
};

__host__ __device__ inline TcLayout tc_layout(int T, int N, int Hv) {
  TcLayout L;
  L.capacity = T / kC + N + 1;
  L.desc_off = 256;
  L.rec_off = L.desc_off + al256((size_t)L.capacity * sizeof(gdn_conv_chunk_t));
  L.total = L.rec_off + (size_t)L.capacity * Hv * kRecBytes;
  return L;
}

__device__ __forceinline__ void bf16_split(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// 8 floats -> hi and lo 16-byte vectors.
__device__ __forceinline__ void split8(const float* f, uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    __nv_bfloat16 a, b;
    bf16_split(f[e], a, b);
    h[e] = __bfloat162float(a);
    l[e] = __bfloat162float(b);
  }
  hi = pack8(h);   // exact: values are already BF16
  lo = pack8(l);
}

// ---------------------------------------------------------------------------
// Chunk kernel
// ---------------------------------------------------------------------------
// Shared memory map (bytes).
constexpr int kS1_A1 = 0;          // [K;Q] tile [128][128]          32768
constexpr int kS1_KT = 32768;      // K^T tile  [128 j][64 s]        16384
constexpr int kS1_VT = 49152;      // V^T tile  [128 i][64 s]        16384
constexpr int kS1_AF = 65536;      // A float32 [64][68] (rows 16-B aligned), also V staging
constexpr int kS1_SM = kS1_AF + 64 * 68 * 4;   // g, b, rk, rq, cw: 5 x 64 floats
constexpr int kS1_BAR = kS1_SM + 5 * 64 * 4;
constexpr int kS1_BYTES = kS1_BAR + 64;
// Aliases once [K;Q] has been consumed: Tm' hi/lo, Tm'' hi/lo tiles [64 r][64 s].
constexpr int kS1_TWH = 0, kS1_TWL = 8192, kS1_TUH = 16384, kS1_TUL = 24576;
// Aliases once the W/U products completed: W hi/lo staging tiles [64 r][128 j].
constexpr int kS1_WST = 32768;

__global__ void __launch_bounds__(kThreads)
tc_chunk_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ q,
                int64_t qk_stride, const __nv_bfloat16* __restrict__ v, int64_t v_stride,
                const float* __restrict__ a, const float* __restrict__ b,
                const int32_t* __restrict__ hdr, const gdn_conv_chunk_t* __restrict__ desc,
                int T, int Hk, int Hv, int l2, unsigned char* __restrict__ records,
                int32_t* __restrict__ status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  float* Af = reinterpret_cast<float*>(sm + kS1_AF);
  float* gs = reinterpret_cast<float*>(sm + kS1_SM);
  float* bs = gs + 64;
  float* rk = bs + 64;
  float* rq = rk + 64;
  float* cw = rq + 64;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + kS1_BAR);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kS1_BAR + 8);
  int* s_fail = reinterpret_cast<int*>(sm + kS1_BAR + 12);
  float* s_tot = reinterpret_cast<float*>(sm + kS1_BAR + 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if ((int)blockIdx.x >= hdr[0]) return;
  const int4 d = reinterpret_cast<const int4*>(desc)[blockIdx.x];
  const int tok0 = d.y, n = d.z;
  if (tok0 < 0 || n <= 0 || n > kC || tok0 + n > T) return;
  const int h = blockIdx.y, gh = h / (Hv / Hk);
  unsigned char* rec = records + ((size_t)blockIdx.x * Hv + h) * kRecBytes;

  if (tid == 0) {
    mbar_init(mbar, 1);
    *s_fail = 0;
  }
  if (warp == 0) {
    tmem_alloc(slot, 256);
    tmem_relinquish();
  }

  // Gates: g = inclusive prefix sum of log a over the chunk (0 past the end).
  if (tid < 64) {
    const bool in = tid < n;
    float x = in ? logf(fmaxf(a[(int64_t)(tok0 + tid) * Hv + h], 1e-30f)) : 0.f;
    bs[tid] = in ? b[(int64_t)(tok0 + tid) * Hv + h] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (tid == 31) *s_tot = x;
    gs[tid] = x;
  }
  // [K; Q] rows into the A1 tile, with row sums of squares for the L2 norm.
  for (int it = 0; it < 16; ++it) {
    const int c = tid + kThreads * it;
    const int row = c >> 4, kc = c & 15, rr = row & 63;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (rr < n) {
      const __nv_bfloat16* src = (row < 64 ? k : q) + (int64_t)(tok0 + rr) * qk_stride +
                                 (int64_t)gh * kD + kc * 8;
      u = ldg16(src);
    }
    *reinterpret_cast<uint4*>(sm + kS1_A1 + tile_off(row, kc * 8, 128)) = u;
    float f[8];
    unpack8(u, f);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += f[e] * f[e];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (kc == 0) {
      const float r = l2 ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
      if (row < 64) rk[rr] = r; else rq[rr] = r;
    }
  }
  // V rows (plain row-major staging in the A area, 256 bytes per row).
  for (int it = 0; it < 8; ++it) {
    const int c = tid + kThreads * it;
    const int s = c >> 4, kc = c & 15;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (s < n) u = ldg16(v + (int64_t)(tok0 + s) * v_stride + (int64_t)h * kD + kc * 8);
    *reinterpret_cast<uint4*>(sm + kS1_AF + s * 256 + kc * 16) = u;
  }
  __syncthreads();
  if (tid >= 32 && tid < 64) gs[tid] += *s_tot;
  // K^T and V^T tiles [128][64]: thread -> (row j = tid, 8-token group it).
  for (int it = 0; it < 8; ++it) {
    const int j = tid;
    float fk[8], fv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int s = it * 8 + e;
      fk[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
          sm + kS1_A1 + tile_off(s, j, 128)));
      fv[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
          sm + kS1_AF + s * 256 + j * 2));
    }
    *reinterpret_cast<uint4*>(sm + kS1_KT + tile_off(j, it * 8, 64)) = pack8(fk);
    *reinterpret_cast<uint4*>(sm + kS1_VT + tile_off(j, it * 8, 64)) = pack8(fv);
  }
  fence_smem_to_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t taddr = *slot;

  // G = [K; Q] K^T  -> TMEM columns [0, 64).
  if (tid == 0) {
    const uint32_t a1 = smem_u32(sm + kS1_A1);
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(taddr, tile_desc(a1, 128, kk), tile_desc(a1, 128, kk), idesc_bf16_f32(128, 64),
               kk > 0);
    mma_commit(mbar);
  }
  if (!mbar_wait(mbar, 0)) atomicExch(s_fail, 1);
  fence_after_sync();
  {
    float G0[32], G1[32];
    tmem_ld32(tmem_warp_addr(taddr, 0), G0);
    tmem_ld32(tmem_warp_addr(taddr, 32), G1);
    if (tid < 64) {
      const int r = tid;
      const float br = bs[r] * rk[r], gr = gs[r];
#pragma unroll
      for (int s0 = 0; s0 < 64; s0 += 4) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int s = s0 + e;
          const float gv = s < 32 ? G0[s & 31] : G1[s & 31];
          o[e] = (s < r && r < n) ? br * expf(gr - gs[s]) * rk[s] * gv : 0.f;
        }
        *reinterpret_cast<float4*>(Af + r * 68 + s0) = make_float4(o[0], o[1], o[2], o[3]);
      }
    } else {
      const int r = tid - 64;
      const float qr = rq[r], gr = gs[r];
#pragma unroll
      for (int s0 = 0; s0 < 64; s0 += 8) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = s0 + e;
          const float gv = s < 32 ? G0[s & 31] : G1[s & 31];
          pv[e] = (s <= r && r < n) ? expf(gr - gs[s]) * qr * rk[s] * gv : 0.f;
        }
        *reinterpret_cast<uint4*>(rec + kOffP + tile_off(r, s0, 64)) = pack8(pv);
      }
    }
  }
  // e^{g_r} rq_r q_r tile and K^T tile to the record.
  for (int it = 0; it < 8; ++it) {
    const int c = tid + kThreads * it;
    const int r = c >> 4, kc = c & 15;
    const uint4 u = *reinterpret_cast<const uint4*>(sm + kS1_A1 + tile_off(64 + r, kc * 8, 128));
    const float sc = r < n ? expf(gs[r]) * rq[r] : 0.f;
    float f[8];
    unpack8(u, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] *= sc;
    *reinterpret_cast<uint4*>(rec + kOffGQ + tile_off(r, kc * 8, 128)) = pack8(f);
  }
  for (int it = 0; it < 8; ++it) {
    const int c = tid + kThreads * it;
    reinterpret_cast<uint4*>(rec + kOffKT)[c] = reinterpret_cast<const uint4*>(sm + kS1_KT)[c];
  }
  if (tid < 64) cw[tid] = bs[tid] * expf(gs[tid]) * rk[tid];
  fence_before_sync();
  __syncthreads();

  // Tm = (I + A)^{-1}: thread t solves column j = t % 64 by forward substitution
  // (x_r = -sum_{s<r} A_rs x_s, x_j = 1); threads 0-63 write the W-side tiles
  // (Tm diag(b e^g rk)), threads 64-127 the U-side tiles (Tm diag(b)).
  {
    const int j = tid & 63;
    float x[64];
#pragma unroll
    for (int r = 0; r < 64; ++r) x[r] = 0.f;
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int s = 0; s < r; s += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(Af + r * 68 + s);
        acc0 = fmaf(a4.x, x[s], acc0);
        acc1 = fmaf(a4.y, x[s + 1], acc1);
        acc0 = fmaf(a4.z, x[s + 2], acc0);
        acc1 = fmaf(a4.w, x[s + 3], acc1);
      }
      x[r] = (r == j) ? 1.f : -(acc0 + acc1);
    }
    const float scale = (tid < 64) ? cw[j] : bs[j];
    unsigned char* th = sm + (tid < 64 ? kS1_TWH : kS1_TUH);
    unsigned char* tl = sm + (tid < 64 ? kS1_TWL : kS1_TUL);
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      __nv_bfloat16 hi, lo;
      bf16_split(x[r] * scale, hi, lo);
      *reinterpret_cast<__nv_bfloat16*>(th + tile_off(r, j, 64)) = hi;
      *reinterpret_cast<__nv_bfloat16*>(tl + tile_off(r, j, 64)) = lo;
    }
  }
  fence_smem_to_async();
  __syncthreads();
  fence_after_sync();

  // W^T = K^T Tm'^T -> cols [64, 128);  U^T = V^T Tm''^T -> cols [128, 192).
  if (tid == 0 && !*s_fail) {
    const uint32_t kt = smem_u32(sm + kS1_KT), vt = smem_u32(sm + kS1_VT);
    const uint32_t twh = smem_u32(sm + kS1_TWH), twl = smem_u32(sm + kS1_TWL);
    const uint32_t tuh = smem_u32(sm + kS1_TUH), tul = smem_u32(sm + kS1_TUL);
    const uint32_t id = idesc_bf16_f32(128, 64);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 64, tile_desc(kt, 64, kk), tile_desc(twh, 64, kk), id, kk > 0);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 64, tile_desc(kt, 64, kk), tile_desc(twl, 64, kk), id, 1);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 128, tile_desc(vt, 64, kk), tile_desc(tuh, 64, kk), id, kk > 0);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 128, tile_desc(vt, 64, kk), tile_desc(tul, 64, kk), id, 1);
    mma_commit(mbar);
  }
  __syncthreads();
  if (!*s_fail) {
    if (!mbar_wait(mbar, 1)) atomicExch(s_fail, 1);
  }
  fence_after_sync();
  __syncthreads();
  if (!*s_fail) {
    // Lane j holds W[r][j] for all r: split into the staging tiles [64 r][128 j].
    float w[32];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      tmem_ld32(tmem_warp_addr(taddr, 64 + 32 * half), w);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int r = 32 * half + e;
        __nv_bfloat16 hi, lo;
        bf16_split(w[e], hi, lo);
        *reinterpret_cast<__nv_bfloat16*>(sm + kS1_WST + tile_off(r, tid, 128)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sm + kS1_WST + 16384 + tile_off(r, tid, 128)) = lo;
      }
    }
    // Lane i holds U[r][i] for all r: row i of the U record (float32).
    float* urow = reinterpret_cast<float*>(rec + kOffU) + tid * 64;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      tmem_ld32(tmem_warp_addr(taddr, 128 + 32 * half), w);
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(urow + 32 * half + e) = make_float4(w[e], w[e + 1], w[e + 2], w[e + 3]);
    }
    if (tid < 64) {
      float* gk = reinterpret_cast<float*>(rec + kOffGK);
      gk[tid] = gs[tid];
      gk[64 + tid] = rk[tid];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (!*s_fail) {
    for (int it = 0; it < 16; ++it) {
      const int c = tid + kThreads * it;
      reinterpret_cast<uint4*>(rec + kOffWhi)[c] =
          reinterpret_cast<const uint4*>(sm + kS1_WST)[c];
    }
  } else if (tid == 0) {
    atomicExch(status + 2, (int)GDN_ERR_TIMEOUT);
  }
  if (warp == 0) tmem_dealloc(taddr, 256);
}

// ---------------------------------------------------------------------------
// State kernel
// ---------------------------------------------------------------------------
constexpr int kS2_SAH = 0;          // S hi  [128 i][128 j]   32768
constexpr int kS2_SAL = 32768;      // S lo                   32768
constexpr int kS2_DA = 65536;       // Delta^T hi [128 i][64 s] 16384
constexpr int kS2_DDH = 81920;      // (Delta^T D) hi           16384
constexpr int kS2_DDL = 98304;      // (Delta^T D) lo           16384
constexpr int kS2_B = 114688;       // record tiles (Whi, Wlo, P, GQ, KT) 73728
constexpr int kS2_WH = kS2_B + kOffWhi, kS2_WL = kS2_B + kOffWlo, kS2_P = kS2_B + kOffP;
constexpr int kS2_GQ = kS2_B + kOffGQ, kS2_KT = kS2_B + kOffKT;
constexpr int kS2_GK = kS2_B + kTileBytes;        // g[64], rk[64]
constexpr int kS2_DK = kS2_GK + 512;              // D_s rk_s [64]
constexpr int kS2_BAR = kS2_DK + 256;
constexpr int kS2_BYTES = kS2_BAR + 64;

__global__ void __launch_bounds__(kThreads, 1)
tc_state_kernel(const int32_t* __restrict__ cu, int T, int N, float* __restrict__ S,
                const uint8_t* __restrict__ has_init, __nv_bfloat16* __restrict__ o, int Hv,
                const unsigned char* __restrict__ records, int32_t* __restrict__ hdr) {
  extern __shared__ __align__(1024) unsigned char sm[];
  float* gk = reinterpret_cast<float*>(sm + kS2_GK);
  float* dks = reinterpret_cast<float*>(sm + kS2_DK);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + kS2_BAR);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kS2_BAR + 8);
  int* s_first = reinterpret_cast<int*>(sm + kS2_BAR + 12);
  int* s_fail = reinterpret_cast<int*>(sm + kS2_BAR + 16);

  const int seq = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int start = cu[seq], end = cu[seq + 1];
  if (start < 0 || end <= start || end > T) return;
  const int nchunks = (end - start + kC - 1) / kC;

  if (tid == 0) {
    *s_first = 0;
    *s_fail = 0;
    mbar_init(mbar, 1);
  }
  __syncthreads();
  {
    int cnt = 0;
    for (int s = tid; s < seq; s += kThreads) {
      const int L = cu[s + 1] - cu[s];
      if (L > 0) cnt += (L + kC - 1) / kC;
    }
    if (cnt) atomicAdd(s_first, cnt);
  }
  if (warp == 0) {
    tmem_alloc(slot, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t taddr = *slot;
  const int first = *s_first;
  const bool records_ok = first + nchunks <= hdr[0];

  float* Sg = S + (((size_t)seq * Hv + h) * kD + tid) * kD;
  const bool init = has_init != nullptr && has_init[seq] != 0;
  {
    float vbuf[32];
    for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float4 f4 = init ? *reinterpret_cast<const float4*>(Sg + blk * 32 + e)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        vbuf[e] = f4.x; vbuf[e + 1] = f4.y; vbuf[e + 2] = f4.z; vbuf[e + 3] = f4.w;
      }
      tmem_st32(tmem_warp_addr(taddr, blk * 32), vbuf);
    }
  }

  uint32_t phase = 0;
  const uint32_t id64 = idesc_bf16_f32(128, 64), id128 = idesc_bf16_f32(128, 128);
  for (int ci = 0; ci < nchunks && records_ok; ++ci) {
    const int c0 = start + ci * kC;
    const int n = min(kC, end - c0);
    const unsigned char* rec = records + ((size_t)(first + ci) * Hv + h) * kRecBytes;
    // (a) this chunk's tiles, gates and U row.
    for (int it = 0; it < kTileBytes / 16 / kThreads; ++it) {
      const int c = tid + kThreads * it;
      reinterpret_cast<uint4*>(sm + kS2_B)[c] = __ldg(reinterpret_cast<const uint4*>(rec) + c);
    }
    if (tid < 32)
      reinterpret_cast<uint4*>(sm + kS2_GK)[tid] =
          __ldg(reinterpret_cast<const uint4*>(rec + kOffGK) + tid);
    float u[64];
    {
      const float4* up = reinterpret_cast<const float4*>(rec + kOffU) + tid * 16;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float4 f = __ldg(up + e);
        u[4 * e] = f.x; u[4 * e + 1] = f.y; u[4 * e + 2] = f.z; u[4 * e + 3] = f.w;
      }
    }
    __syncthreads();
    const float glast = gk[n - 1];
    const float gamma_c = expf(glast);
    if (tid < 64) dks[tid] = tid < n ? expf(glast - gk[tid]) * gk[64 + tid] : 0.f;
    // (b) S -> hi/lo A tiles (row i = tid), then S <- e^{g_last} S in TMEM.
    for (int blk = 0; blk < 4; ++blk) {
      float sv[32];
      tmem_ld32(tmem_warp_addr(taddr, blk * 32), sv);
#pragma unroll
      for (int e8 = 0; e8 < 4; ++e8) {
        uint4 hi, lo;
        split8(sv + 8 * e8, hi, lo);
        const int j0 = blk * 32 + e8 * 8;
        *reinterpret_cast<uint4*>(sm + kS2_SAH + tile_off(tid, j0, 128)) = hi;
        *reinterpret_cast<uint4*>(sm + kS2_SAL + tile_off(tid, j0, 128)) = lo;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) sv[e] *= gamma_c;
      tmem_st32(tmem_warp_addr(taddr, blk * 32), sv);
    }
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // (c) X^T = S W^T (3 passes) -> cols [128,192);  O^T = S (e^g Q)^T -> cols [192,256).
    if (tid == 0) {
      const uint32_t sah = smem_u32(sm + kS2_SAH), sal = smem_u32(sm + kS2_SAL);
      const uint32_t wh = smem_u32(sm + kS2_WH), wl = smem_u32(sm + kS2_WL);
      const uint32_t gq = smem_u32(sm + kS2_GQ);
      for (int kk = 0; kk < 8; ++kk) mma_bf16(taddr + 128, tile_desc(sah, 128, kk), tile_desc(wh, 128, kk), id64, kk > 0);
      for (int kk = 0; kk < 8; ++kk) mma_bf16(taddr + 128, tile_desc(sah, 128, kk), tile_desc(wl, 128, kk), id64, 1);
      for (int kk = 0; kk < 8; ++kk) mma_bf16(taddr + 128, tile_desc(sal, 128, kk), tile_desc(wh, 128, kk), id64, 1);
      for (int kk = 0; kk < 8; ++kk) mma_bf16(taddr + 192, tile_desc(sah, 128, kk), tile_desc(gq, 128, kk), id64, kk > 0);
      mma_commit(mbar);
    }
    if (!mbar_wait(mbar, phase)) atomicExch(s_fail, 1);
    phase ^= 1;
    fence_after_sync();
    // (d) Delta^T = U^T - X^T for this lane's row i; A tiles for O and for S.
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float xv[32];
      tmem_ld32(tmem_warp_addr(taddr, 128 + 32 * half), xv);
#pragma unroll
      for (int e8 = 0; e8 < 4; ++e8) {
        float dl[8], dd[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = 32 * half + 8 * e8 + e;
          const float del = r < n ? u[r] - xv[8 * e8 + e] : 0.f;
          dl[e] = del;
          dd[e] = del * dks[r];
        }
        const int s0 = 32 * half + 8 * e8;
        uint4 hi, lo;
        *reinterpret_cast<uint4*>(sm + kS2_DA + tile_off(tid, s0, 64)) = pack8(dl);
        split8(dd, hi, lo);
        *reinterpret_cast<uint4*>(sm + kS2_DDH + tile_off(tid, s0, 64)) = hi;
        *reinterpret_cast<uint4*>(sm + kS2_DDL + tile_off(tid, s0, 64)) = lo;
      }
    }
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // (e) O^T += Delta^T P^T;  S += (Delta^T D) K  (hi and lo passes).
    if (tid == 0 && !*s_fail) {
      const uint32_t da = smem_u32(sm + kS2_DA), p = smem_u32(sm + kS2_P);
      const uint32_t ddh = smem_u32(sm + kS2_DDH), ddl = smem_u32(sm + kS2_DDL);
      const uint32_t kt = smem_u32(sm + kS2_KT);
      for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 192, tile_desc(da, 64, kk), tile_desc(p, 64, kk), id64, 1);
      for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr, tile_desc(ddh, 64, kk), tile_desc(kt, 64, kk), id128, 1);
      for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr, tile_desc(ddl, 64, kk), tile_desc(kt, 64, kk), id128, 1);
      mma_commit(mbar);
    }
    __syncthreads();
    if (*s_fail) break;
    if (!mbar_wait(mbar, phase)) atomicExch(s_fail, 1);
    phase ^= 1;
    fence_after_sync();
    // (f) outputs: lane i holds O[r][i] for the chunk's tokens r.
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float ov[32];
      tmem_ld32(tmem_warp_addr(taddr, 192 + 32 * half), ov);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int r = 32 * half + e;
        if (r < n) o[((int64_t)(c0 + r) * Hv + h) * kD + tid] = __float2bfloat16_rn(ov[e]);
      }
    }
    fence_before_sync();
    __syncthreads();
    if (*s_fail) break;
  }
  if (!*s_fail && records_ok) {
    for (int blk = 0; blk < 4; ++blk) {
      float sv[32];
      tmem_ld32(tmem_warp_addr(taddr, blk * 32), sv);
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(Sg + blk * 32 + e) = make_float4(sv[e], sv[e + 1], sv[e + 2], sv[e + 3]);
    }
  } else if (tid == 0) {
    atomicExch(hdr + 2, (int)(*s_fail ? GDN_ERR_TIMEOUT : GDN_ERR_INVALID_ARG));
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, 256);
}

}  // namespace

size_t prefill_tc_workspace_bytes(int32_t T, int32_t N, int32_t Hv) {
  return tc_layout(T, N, Hv).total;
}

gdn_status_t launch_prefill_tc(const void* q, const void* k, int64_t qk_stride, const void* v,
                               int64_t v_stride, const float* a, const float* b,
                               const int32_t* cu, int32_t N, int32_t T, float* S,
                               const uint8_t* has_init, void* o, int32_t Hk, int32_t Hv,
                               int32_t qk_l2norm, void* workspace, cudaStream_t st) {
  const TcLayout L = tc_layout(T, N, Hv);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws);
  auto desc = reinterpret_cast<gdn_conv_chunk_t*>(ws + L.desc_off);
  unsigned char* records = ws + L.rec_off;
  static const bool attrs = [] {
    cudaFuncSetAttribute(tc_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kS1_BYTES);
    cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kS2_BYTES);
    return true;
  }();
  (void)attrs;
  if (cudaMemsetAsync(hdr + 2, 0, sizeof(int32_t), st) != cudaSuccess) return check_launch();
  gdn_status_t rc = launch_build_chunks(cu, N, kC, desc, L.capacity, hdr, hdr + 1, st);
  if (rc != GDN_OK) return rc;
  tc_chunk_kernel<<<dim3(L.capacity, Hv), kThreads, kS1_BYTES, st>>>(
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(q), qk_stride,
      static_cast<const __nv_bfloat16*>(v), v_stride, a, b, hdr, desc, T, Hk, Hv, qk_l2norm,
      records, hdr);
  if ((rc = check_launch()) != GDN_OK) return rc;
  tc_state_kernel<<<dim3(N, Hv), kThreads, kS2_BYTES, st>>>(
      cu, T, N, S, has_init, static_cast<__nv_bfloat16*>(o), Hv, records, hdr);
  return check_launch();
}

}  // namespace gdn
