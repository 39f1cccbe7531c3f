// Chunked prefill of the gated delta rule on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM), head dimension 128.
//
// The chunk algebra is the one described in prefill.cu. Everything is laid out
// so that every product has M = 128 (the head dimension); operand tiles use the
// K-major and MN-major layouts described in tc_ptx.cuh, or TMEM for A:
//
//   chunk kernel, one CTA per (64-token chunk, v-head):
//     G    = [K; Q] K^T                        (M=128: K rows then Q rows, N=64, K=128)
//     A_rs = b_r e^{g_r-g_s} (k_r.k_s), P_rs = e^{g_r-g_s} (q_r.k_s)     (CUDA cores)
//     Tm   = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution,
//            the blocks below them by blocked products          (CUDA cores)
//     W^T  = K^T (Tm diag(b e^g))^T,  U^T = V^T (Tm diag(b))^T          (M=128, N=64, K=64)
//   and writes, per (chunk, v-head), a record with W (BF16 hi + lo) and P (in
//   the tile layouts the state kernel feeds straight to the tensor core), U
//   (float32) and the gates and norms.
//
//   state kernel, one CTA per (sequence, v-head), S [dv=128 x dk=128] float32
//   resident in TMEM, and its BF16 hi + lo parts beside it in TMEM, where the
//   tensor core reads them as the A operand; chunks in order:
//     X^T  = S W^T                  (S and W split into BF16 hi + lo: 3 MMAs)
//     O1^T = S Q^T                  (single BF16: the output is BF16)
//     Delta^T = U^T - X^T           (CUDA cores, lane i holds row i)
//     O2^T = Delta^T P^T            (single BF16); o_r = e^{g_r} O1_r + O2_r,
//            transposed through shared memory and written out as whole
//            256-byte output rows
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

// Record of one (chunk, v-head) written by the chunk kernel and read, by bulk
// copy, by the state kernel.
// W hi and W lo as one MN-major B tile of N = 128 (rows 0-63: W hi of token r,
// rows 64-127: W lo of token r), K = j (128), so that S_hi [W hi; W lo]^T is a
// single N = 128 product.
constexpr int kOffW = 0;
constexpr int kOffP = 32768;        // P      K-major  [64 r][64 s]
constexpr int kOffU = 40960;        // U      [128 i][64 r] float32, 16-byte chunks XOR-swizzled
constexpr int kOffGK = 73728;       // g[64] (log2 of the cumulative decay), rk[64], rq[64]
constexpr int kRecBytes = 74496;    // 73728 + 768

__host__ __device__ constexpr size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

struct TcLayout {
  int capacity;
  size_t desc_off, order_off, rec_off, total;
};

__host__ __device__ inline TcLayout tc_layout(int T, int N, int Hv) {
  TcLayout L;
  L.capacity = T / kC + N + 1;
  L.desc_off = 256;
  L.order_off = L.desc_off + al256((size_t)L.capacity * sizeof(gdn_conv_chunk_t));
  L.rec_off = L.order_off + al256((size_t)N * sizeof(int32_t));
  L.total = L.rec_off + (size_t)L.capacity * Hv * kRecBytes;
  return L;
}

// 8 floats -> BF16 hi and lo parts (hi = bf16(x), lo = bf16(x - hi)) as 16-byte vectors.
// 2^x for x <= 0 (decay ratios), with the hardware base-2 exponential
// (ex2.approx.ftz: relative error ~2^-22; results below the normal range
// flush to zero).
__device__ __forceinline__ float exp2_nonpos(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(fminf(x, 0.f)));
  return y;
}

__device__ __forceinline__ void split8(const float* f, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    h[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
    l[e] = pack_bf16x2(f[2 * e] - bf16lo(h[e]), f[2 * e + 1] - bf16hi(h[e]));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// ---------------------------------------------------------------------------
// Chunk kernel: 128 threads, about 66 KB of shared memory and 128 TMEM columns,
// so three CTAs share an SM.
// ---------------------------------------------------------------------------
constexpr int kS1_A1 = 0;          // rows 0-63: K [s][j], rows 64-127: Q [r][j] (K-major, Kc 128)
constexpr int kS1_V = 32768;       // V [s][i] (K-major layout, read as MN-major A for V^T)
constexpr int kS1_AF = 49152;      // A float32 [64][68]
constexpr int kS1_SM = kS1_AF + 64 * 68 * 4;   // g2, b, rk, rq, cw: 5 x 64 floats
constexpr int kS1_RS = kS1_SM + 5 * 64 * 4;    // block-inverse scratch [3][16][16] float32
constexpr int kS1_BAR = kS1_RS + 3 * 256 * 4;
constexpr int kS1_BYTES = kS1_BAR + 64;
// Tm float32 [64][64] in the Q rows once they are consumed; the MN-major B
// tiles (N = r, K = s) of Tm diag(b e^g rk) go to the A area after the solve,
// those of Tm diag(b) to the Q rows after Tm has been read.
constexpr int kS1_TF = 16384;
constexpr int kS1_TWH = kS1_AF, kS1_TWL = kS1_AF + 8192;
constexpr int kS1_TUH = 16384, kS1_TUL = 24576;

// TC consecutive floats from shared memory (TC = 2 or 4).
template <int TC>
__device__ __forceinline__ void lds_vec(const float* p, float (&v)[TC]) {
  if constexpr (TC == 4) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
    const float2 f = *reinterpret_cast<const float2*>(p);
    v[0] = f.x; v[1] = f.y;
  }
}

// One distance of the blocked triangular inverse: for the tiles (i, j = i - D),
// R_ij = sum_{s in [16 j, 16 i)} A[16 i + rr][s] Tm[s][16 j + cc], then
// Tm_ij = -D_i R_ij. Thread t owns a TR x TC piece of one tile, accumulated in
// registers from vector loads (TR rows of A and four rows of Tm per step of
// four s), with the pieces sized so that nearly every thread has one at every
// distance (2 x 4 on 96 threads, 1 x 4 and 1 x 2 on 128); trip counts are
// compile-time.
template <int D, int TR, int TC>
__device__ __forceinline__ void tm_offdiag(const float* __restrict__ Af, float* __restrict__ Tf,
                                           float* __restrict__ Rs, int tid) {
  constexpr int kPerRow = 16 / TC, kPerTile = (16 / TR) * kPerRow;
  constexpr int kPieces = (4 - D) * kPerTile;
  const int blk = tid / kPerTile, t = tid - blk * kPerTile;
  const int i = D + blk, jb = i - D;
  const int r0 = TR * (t / kPerRow), c0 = TC * (t - (t / kPerRow) * kPerRow);
  if (tid < kPieces) {
    float acc[TR][TC];
#pragma unroll
    for (int rr = 0; rr < TR; ++rr)
#pragma unroll
      for (int cc = 0; cc < TC; ++cc) acc[rr][cc] = 0.f;
#pragma unroll
    for (int s4 = 0; s4 < 16 * D; s4 += 4) {
      const int s0 = 16 * jb + s4;
      float a[TR][4], tv[4][TC];
#pragma unroll
      for (int rr = 0; rr < TR; ++rr) lds_vec<4>(Af + (16 * i + r0 + rr) * 68 + s0, a[rr]);
#pragma unroll
      for (int e = 0; e < 4; ++e) lds_vec<TC>(Tf + (s0 + e) * 64 + 16 * jb + c0, tv[e]);
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int rr = 0; rr < TR; ++rr)
#pragma unroll
          for (int cc = 0; cc < TC; ++cc) acc[rr][cc] = fmaf(a[rr][e], tv[e][cc], acc[rr][cc]);
    }
#pragma unroll
    for (int rr = 0; rr < TR; ++rr)
#pragma unroll
      for (int cc = 0; cc < TC; ++cc) Rs[blk * 256 + (r0 + rr) * 16 + c0 + cc] = acc[rr][cc];
  }
  __syncthreads();
  if (tid < kPieces) {
    float acc[TR][TC];
#pragma unroll
    for (int rr = 0; rr < TR; ++rr)
#pragma unroll
      for (int cc = 0; cc < TC; ++cc) acc[rr][cc] = 0.f;
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      float d[TR][4], rv[4][TC];
#pragma unroll
      for (int rr = 0; rr < TR; ++rr) lds_vec<4>(Tf + (16 * i + r0 + rr) * 64 + 16 * i + k4, d[rr]);
#pragma unroll
      for (int e = 0; e < 4; ++e) lds_vec<TC>(Rs + blk * 256 + (k4 + e) * 16 + c0, rv[e]);
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int rr = 0; rr < TR; ++rr)
#pragma unroll
          for (int cc = 0; cc < TC; ++cc) acc[rr][cc] = fmaf(d[rr][e], rv[e][cc], acc[rr][cc]);
    }
#pragma unroll
    for (int rr = 0; rr < TR; ++rr)
#pragma unroll
      for (int cc = 0; cc < TC; ++cc)
        Tf[(16 * i + r0 + rr) * 64 + 16 * jb + c0 + cc] = -acc[rr][cc];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 3)
tc_chunk_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ q,
                int64_t qk_stride, const __nv_bfloat16* __restrict__ v, int64_t v_stride,
                const float* __restrict__ a, const float* __restrict__ b,
                const int32_t* __restrict__ hdr, const gdn_conv_chunk_t* __restrict__ desc,
                int T, int Hk, int Hv, int flags, unsigned char* __restrict__ records,
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
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x >= hdr[0]) return;
  const int4 d = reinterpret_cast<const int4*>(desc)[blockIdx.x];
  const int tok0 = d.y, n = d.z;
  if (tok0 < 0 || n <= 0 || n > kC || tok0 + n > T) return;
  const int h = blockIdx.y, gh = h / (Hv / Hk);
  unsigned char* rec = records + ((size_t)blockIdx.x * Hv + h) * kRecBytes;

  // K, Q and V rows as 16-byte asynchronous copies, all in flight together.
  // Lane l of a warp covers row (8 rg + l % 8) and chunk (4 kg + l / 8): eight
  // consecutive rows per quarter warp keep the shared-memory writes
  // conflict-free, four chunks per row keep the global reads in 64-byte runs.
#pragma unroll
  for (int it = 0; it < 16; ++it) {
    const int p = it * 4 + warp;
    const int row = (p >> 2) * 8 + (lane & 7), kc = (p & 3) * 4 + (lane >> 3);
    const int rr = row & 63;
    const bool valid = rr < n;
    const __nv_bfloat16* src = (row < 64 ? k : q) + (int64_t)(tok0 + (valid ? rr : 0)) * qk_stride +
                               (int64_t)gh * kD + kc * 8;
    cp_async16(sm + kS1_A1 + tile_off(row, kc * 8, 128), src, valid ? 16u : 0u);
  }
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int p = it * 4 + warp;
    const int s = (p >> 2) * 8 + (lane & 7), kc = (p & 3) * 4 + (lane >> 3);
    const bool valid = s < n;
    cp_async16(sm + kS1_V + tile_off(s, kc * 8, 128),
               v + (int64_t)(tok0 + (valid ? s : 0)) * v_stride + (int64_t)h * kD + kc * 8,
               valid ? 16u : 0u);
  }
  if (tid == 0) {
    mbar_init(mbar, 1);
    *s_fail = 0;
  }
  if (warp == 0) {
    tmem_alloc(slot, 128);
    tmem_relinquish();
  }
  // Gates: g = inclusive prefix sum of log a over the chunk (0 past the end).
  if (tid < 64) {
    const bool in = tid < n;
    // log2 of the decay, so that decay ratios are single exp2 evaluations.
    const bool gl = (flags & kFlagGateLogits) != 0;
    float x = in ? gate_log2_decay(a[(int64_t)(tok0 + tid) * Hv + h], gl) : 0.f;
    bs[tid] = in ? gate_write(b[(int64_t)(tok0 + tid) * Hv + h], gl) : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (tid == 31) *s_tot = x;
    gs[tid] = x;
  }
  cp_async_wait_all();
  __syncthreads();
  if (tid >= 32 && tid < 64) gs[tid] += *s_tot;
  // Row norms (thread = row; eight consecutive rows per quarter warp).
  {
    float ss = 0.f;
#pragma unroll
    for (int kc = 0; kc < 16; ++kc) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(sm + kS1_A1 + tile_off(tid, kc * 8, 128)), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
    const float r = (flags & kFlagL2) ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    if (tid < 64) rk[tid] = r; else rq[tid - 64] = r;
  }
  fence_smem_to_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t taddr = *slot;
  const uint32_t a1 = smem_u32(sm + kS1_A1);

  // G = [K; Q] K^T -> TMEM columns [0, 64).
  if (tid == 0) {
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(taddr, tile_desc(a1, 128, kk), tile_desc(a1, 128, kk), idesc_bf16_f32(128, 64),
               kk > 0);
    mma_commit(mbar);
  }
  if (tid < 64) cw[tid] = bs[tid] * exp2_nonpos(gs[tid]) * rk[tid];
  if (!mbar_wait(mbar, 0)) atomicExch(s_fail, 1);
  fence_after_sync();
  {
    // Row r of A = b_r e^{g_r - g_s} rk_r rk_s (k_r . k_s), strictly lower
    // (threads 0-63), and row r of P = e^{g_r - g_s} rq_r rk_s (q_r . k_s),
    // lower with the diagonal (threads 64-127); eight columns per step.
    const bool is_a = tid < 64;
    const int r = tid & 63;
    const float gr = gs[r];
    const float fr = is_a ? bs[r] * rk[r] : rq[r];
#pragma unroll 1
    for (int cb = 0; cb < 8; ++cb) {
      float gv[8], v8[8];
      // gates and norms of the 8 columns as vector loads, so the 8 entries
      // below are independent chains
      const float4 g0 = *reinterpret_cast<const float4*>(gs + 8 * cb);
      const float4 g1 = *reinterpret_cast<const float4*>(gs + 8 * cb + 4);
      const float4 k0 = *reinterpret_cast<const float4*>(rk + 8 * cb);
      const float4 k1 = *reinterpret_cast<const float4*>(rk + 8 * cb + 4);
      const float gsv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float rkv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
      tmem_ld8(tmem_warp_addr(taddr, 8 * cb), gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int s2 = 8 * cb + e;
        const bool keep = (is_a ? s2 < r : s2 <= r) && r < n;
        const float val = fr * exp2_nonpos(gr - gsv[e]) * rkv[e] * gv[e];
        v8[e] = keep ? val : 0.f;
      }
      if (is_a) {
        *reinterpret_cast<float4*>(Af + r * 68 + 8 * cb) = make_float4(v8[0], v8[1], v8[2], v8[3]);
        *reinterpret_cast<float4*>(Af + r * 68 + 8 * cb + 4) = make_float4(v8[4], v8[5], v8[6], v8[7]);
      } else {
        *reinterpret_cast<uint4*>(rec + kOffP + tile_off(r, 8 * cb, 64)) = pack8(v8);
      }
    }
  }
  fence_before_sync();
  __syncthreads();

  // Tm = (I + A)^{-1}, blocked in 16 x 16 tiles. Diagonal tiles D_i =
  // (I + A_ii)^{-1} by forward substitution (thread = column); then, for
  // i - j = 1, 2, 3: Tm_ij = -D_i R_ij with R_ij = sum_{s in [16j, 16i)} A[., s] Tm[s, .]
  // (Tm is zero above the diagonal, so the sum runs over one contiguous range).
  float* Tf = reinterpret_cast<float*>(sm + kS1_TF);   // [64][64]
  float* Rs = reinterpret_cast<float*>(sm + kS1_RS);   // [3][16][16]
  if (tid < 64) {
    const int bi = tid >> 4, c = tid & 15, o0 = 16 * bi;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < r; ++s2) acc = fmaf(Af[(o0 + r) * 68 + o0 + s2], x[s2], acc);
      x[r] = (r == c) ? 1.f : (r < c ? 0.f : -acc);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Tf[(o0 + r) * 64 + o0 + c] = x[r];
  } else {
    // zero the strictly upper tiles (i < j): 6 tiles of 256
    for (int e = tid - 64; e < 6 * 256; e += 64) {
      const int t6 = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      const int ti = t6 < 3 ? 0 : (t6 < 5 ? 1 : 2);
      const int tj = t6 < 3 ? t6 + 1 : (t6 < 5 ? t6 - 1 : 3);
      Tf[(16 * ti + rr) * 64 + 16 * tj + cc] = 0.f;
    }
  }
  __syncthreads();
  tm_offdiag<1, 2, 4>(Af, Tf, Rs, tid);
  tm_offdiag<2, 1, 4>(Af, Tf, Rs, tid);
  tm_offdiag<3, 1, 2>(Af, Tf, Rs, tid);
  // B tiles: column s of Tm diag(b e^g rk) and of Tm diag(b), split hi/lo, as
  // MN-major tiles (N = r, K = s): eight consecutive r per 16 bytes. The W-side
  // tiles go to the (now free) A area at once; the U-side ones are held in
  // registers until every thread is done reading Tm, then overwrite it.
  {
    uint4 uh[4], ul[4];
    const int s_ = tid & 63, rg0 = (tid >> 6) * 4;
    const float cws = cw[s_], bss = bs[s_];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int rg = rg0 + q4;
      float t8[8], f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) t8[e] = Tf[(8 * rg + e) * 64 + s_];
      uint4 hi, lo;
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = t8[e] * cws;
      split8(f, hi, lo);
      *reinterpret_cast<uint4*>(sm + kS1_TWH + mn_off(8 * rg, s_, 64)) = hi;
      *reinterpret_cast<uint4*>(sm + kS1_TWL + mn_off(8 * rg, s_, 64)) = lo;
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = t8[e] * bss;
      split8(f, uh[q4], ul[q4]);
    }
    __syncthreads();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int rg = rg0 + q4;
      *reinterpret_cast<uint4*>(sm + kS1_TUH + mn_off(8 * rg, s_, 64)) = uh[q4];
      *reinterpret_cast<uint4*>(sm + kS1_TUL + mn_off(8 * rg, s_, 64)) = ul[q4];
    }
  }
  fence_smem_to_async();
  __syncthreads();
  fence_after_sync();

  // W^T = K^T Tm'^T -> cols [0, 64);  U^T = V^T Tm''^T -> cols [64, 128).
  if (tid == 0 && !*s_fail) {
    const uint32_t vt = smem_u32(sm + kS1_V);
    const uint32_t twh = smem_u32(sm + kS1_TWH), twl = smem_u32(sm + kS1_TWL);
    const uint32_t tuh = smem_u32(sm + kS1_TUH), tul = smem_u32(sm + kS1_TUL);
    const uint32_t id = idesc_bf16_f32(128, 64) | kTransA | kTransB;
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr, mn_desc(a1, 128, kk), mn_desc(twh, 64, kk), id, kk > 0);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr, mn_desc(a1, 128, kk), mn_desc(twl, 64, kk), id, 1);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 64, mn_desc(vt, 128, kk), mn_desc(tuh, 64, kk), id, kk > 0);
    for (int kk = 0; kk < 4; ++kk) mma_bf16(taddr + 64, mn_desc(vt, 128, kk), mn_desc(tul, 64, kk), id, 1);
    mma_commit(mbar);
  }
  __syncthreads();
  if (!*s_fail) {
    if (!mbar_wait(mbar, 1)) atomicExch(s_fail, 1);
  }
  fence_after_sync();
  __syncthreads();
  if (!*s_fail) {
    // Stage the record in shared memory in its global layout (W hi/lo over the
    // consumed K/Q rows, U over V and the A area, gates over the scratch), then
    // write it with three bulk stores.
    // Lane j holds W[r][j] for all r: MN-major B tiles (N = r, K = j).
    {
      float w0[32], w1[32];
      tmem_ld32x2(tmem_warp_addr(taddr, 0), tmem_warp_addr(taddr, 32), w0, w1);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* w = half ? w1 : w0;
#pragma unroll
        for (int rg = 0; rg < 4; ++rg) {
          uint4 hi, lo;
          split8(w + 8 * rg, hi, lo);
          *reinterpret_cast<uint4*>(sm + kS1_A1 + kOffW + mn_off(32 * half + 8 * rg, tid, 128)) = hi;
          *reinterpret_cast<uint4*>(sm + kS1_A1 + kOffW + mn_off(64 + 32 * half + 8 * rg, tid, 128)) =
              lo;
        }
      }
    }
    // Lane i holds U[r][i] for all r: row i (float32), its 16-byte chunk c at
    // position c ^ (i % 8) so that the state kernel reads one chunk per row
    // across a warp without bank conflicts.
    {
      float4* urow = reinterpret_cast<float4*>(sm + kS1_V) + tid * 16;
      float u0[32], u1[32];
      tmem_ld32x2(tmem_warp_addr(taddr, 64), tmem_warp_addr(taddr, 96), u0, u1);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* w = half ? u1 : u0;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          urow[(8 * half + e / 4) ^ (tid & 7)] = make_float4(w[e], w[e + 1], w[e + 2], w[e + 3]);
      }
    }
    if (tid < 64) {
      float* gk = reinterpret_cast<float*>(sm + kS1_RS);
      gk[tid] = gs[tid];          // log2 units
      gk[64 + tid] = rk[tid];
      gk[128 + tid] = rq[tid];
    }
    fence_smem_to_async();
  } else if (tid == 0) {
    atomicExch(status + 2, (int)GDN_ERR_TIMEOUT);
    record_device_status(GDN_ERR_TIMEOUT);
  }
  fence_before_sync();
  __syncthreads();
  if (tid == 0 && !*s_fail) {
    bulk_s2g(rec + kOffW, sm + kS1_A1 + kOffW, 32768);
    bulk_s2g(rec + kOffU, sm + kS1_V, 32768);
    bulk_s2g(rec + kOffGK, sm + kS1_RS, 768);
    bulk_commit();
    bulk_wait_all();
  }
  if (warp == 0) tmem_dealloc(taddr, 128);
}

// ---------------------------------------------------------------------------
// State kernel: one CTA per (sequence, v-head), S [dv = 128 x dk = 128]
// float32 resident in TMEM, chunks in order. The warp roles hand work to each
// other through mbarriers only, so that no role waits for another's
// instruction stream:
//   warps 0-7 (rows): warp w owns TMEM lanes 32 (w % 4) .. + 31 (row i of S)
//     and column half w / 4. Per chunk: S -> BF16 hi/lo parts (in TMEM) and
//     S <- e^{g_last} S; the previous chunk's outputs; Delta = U - X.
//   warp 8 (one lane): the recurrence's MMAs. X^T = S W^T (hi/lo) once the
//     S parts are ready (A operands read from TMEM, so S costs no shared
//     memory traffic); S += (Delta^T D) K (hi/lo) and O2^T = Delta^T P^T
//     once Delta is.
//   warp 9: the next chunk's record (W and gates, U, P) by bulk copies, each
//     as soon as the buffer it refills is free.
//   warps 10 and 11: the next chunk's raw Q and K rows (16-byte asynchronous
//     copies by all lanes) once the previous tile's readers are done; warp 10
//     also issues O1^T = S Q^T, so that the recurrence's MMA lane never waits
//     on the output products.
// TMEM: S [0, 128), S hi [128, 192) and S lo [192, 256) as BF16 pairs (dk j
// in column j / 2), X^T [256, 384) (two partial sums; once read, the Delta
// parts as BF16 pairs of tokens), O1^T [384, 448) and O2^T [448, 512) (dv i
// in lane i, token r in column r).
// ---------------------------------------------------------------------------
constexpr int kThreads2 = 384;
constexpr int kRowThreads = 256;
constexpr int kS2_STG = 0;          // output staging [64 r][128 dv] BF16     16384
constexpr int kS2_Q = 16384;        // Q rows [64 r][128 j] K-major B         16384
constexpr int kS2_K = 32768;        // K rows [64 s][128 j] (MN-major B)      16384
constexpr int kS2_R = 49152;        // the chunk's record
constexpr int kS2_W = kS2_R + kOffW, kS2_P = kS2_R + kOffP;
constexpr int kS2_U = kS2_R + kOffU, kS2_GK = kS2_R + kOffGK;
constexpr int kS2_QS = kS2_R + kRecBytes;         // e^{g_r} rq_r, two chunks [2][64]
constexpr int kS2_DK = kS2_QS + 512;              // e^{g_last - g_s} rk_s, two chunks [2][64]
constexpr int kS2_BAR = kS2_DK + 512;             // barriers, TMEM slot, flags
constexpr int kS2_BYTES = kS2_BAR + 128;

__global__ void __launch_bounds__(kThreads2, 1)
tc_state_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                int64_t qk_stride, const int32_t* __restrict__ cu, int T, int Hk,
                float* __restrict__ S, const uint8_t* __restrict__ has_init,
                __nv_bfloat16* __restrict__ o, int Hv, const unsigned char* __restrict__ records,
                int32_t* __restrict__ hdr, const int32_t* __restrict__ order, int N,
                const StateSlots slots) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const float* gk = reinterpret_cast<const float*>(sm + kS2_GK);
  const float4* us = reinterpret_cast<const float4*>(sm + kS2_U);
  float* qs = reinterpret_cast<float*>(sm + kS2_QS);
  float* dks = reinterpret_cast<float*>(sm + kS2_DK);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kS2_BAR);
  uint64_t* bW = bars + 0;    // W and gates landed        (bulk copy)
  uint64_t* bU = bars + 1;    // U landed                  (bulk copy)
  uint64_t* bP = bars + 2;    // P landed                  (bulk copy)
  uint64_t* bQ = bars + 3;    // Q rows landed             (32 loader lanes)
  uint64_t* bK = bars + 4;    // K rows landed             (32 loader lanes)
  uint64_t* bSr = bars + 5;   // S hi/lo parts written     (256 row threads)
  uint64_t* bDr = bars + 6;   // Delta tiles written       (256 row threads)
  uint64_t* bX = bars + 7;    // X MMAs done               (commit)
  uint64_t* bO1 = bars + 8;   // O1 MMAs done              (commit, warp 10)
  uint64_t* bS = bars + 9;    // S update done             (commit)
  uint64_t* bO = bars + 10;   // O2 MMAs (and all before) done (commit)
  uint64_t* bOr = bars + 11;  // outputs read from TMEM    (256 row threads)
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kS2_BAR + 104);
  int* s_first = reinterpret_cast<int*>(sm + kS2_BAR + 108);
  int* s_fail = reinterpret_cast<int*>(sm + kS2_BAR + 112);

  // CTA r * Hv + h runs head h of the r-th longest sequence, so that the
  // long chains start in the first wave.
  const int rank = blockIdx.x / Hv, h = blockIdx.x - rank * Hv, gh = h / (Hv / Hk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = 32 * (warp & 3) + lane;   // row warps: S row (dv index) = TMEM lane
  const int hf = (warp >> 2) & 1;           // row warps: column / token half
  pdl_wait();
  pdl_trigger();
  const int seq = order[rank];
  if (seq < 0 || seq >= N) return;
  const int start = cu[seq], end = cu[seq + 1];
  if (start < 0 || end <= start || end > T) return;
  const int sslot = state_slot(slots, seq);
  if (sslot < 0) return;   // a padding entry: state and outputs untouched
  const int nchunks = (end - start + kC - 1) / kC;

  if (tid == 0) {
    *s_first = 0;
    *s_fail = 0;
    for (int i = 0; i < 12; ++i) {
      const bool rows_in = bars + i == bQ || bars + i == bK;
      const bool rows_out = bars + i == bSr || bars + i == bDr || bars + i == bOr;
      mbar_init(bars + i, rows_in ? 32u : (rows_out ? (uint32_t)kRowThreads : 1u));
    }
  }
  __syncthreads();
  {
    int cnt = 0;
    for (int s = tid; s < seq; s += kThreads2) {
      const int L = cu[s + 1] - cu[s];
      if (L > 0) cnt += (L + kC - 1) / kC;
    }
    if (cnt) atomicAdd(s_first, cnt);
  }
  if (warp == 0) {
    tmem_alloc(slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t taddr = *slot;
  const int first = *s_first;
  const bool records_ok = first + nchunks <= hdr[0];
  float* Sg = S + (((size_t)sslot * Hv + h) * kD + row) * kD;

  // Wait for the phase of parity `par`. Returns false at once when the CTA is
  // aborting, and starts the abort after about two seconds; the roles then
  // run their remaining steps without waiting, so that every named barrier
  // is still reached by all of its threads.
  auto wait = [&](uint64_t* b, uint32_t par) -> bool {
    const long long t0 = clock64();
    while (!mbar_try_wait(b, par)) {
      if (*reinterpret_cast<volatile int*>(s_fail)) return false;
      if (clock64() - t0 > 4000000000LL) {
        atomicExch(s_fail, 1);
        return false;
      }
    }
    return true;
  };
  auto failed = [&]() { return *reinterpret_cast<volatile int*>(s_fail) != 0; };
  auto rec_of = [&](int ci) {
    return records + ((size_t)(first + ci) * Hv + h) * kRecBytes;
  };

  // 16-byte asynchronous copies of chunk ci's raw rows (Q or K) into a tile by
  // one warp, then one arrival per lane on `bar` once they have landed.
  auto rows = [&](int ci, const __nv_bfloat16* src, int tile, uint64_t* bar) {
    const int c0 = start + ci * kC;
    const int n = min(kC, end - c0);
    // Lane l covers row (8 rg + l % 8) and chunk (4 kg + l / 8): eight
    // consecutive rows per quarter warp keep the shared-memory writes
    // conflict-free, four chunks per row keep global reads in 64-byte runs.
#pragma unroll 4
    for (int p = 0; p < 32; ++p) {
      const int r = (p >> 2) * 8 + (lane & 7), kc = (p & 3) * 4 + (lane >> 3);
      const bool valid = r < n;
      cp_async16(sm + tile + tile_off(r, kc * 8, 128),
                 src + (int64_t)(c0 + (valid ? r : 0)) * qk_stride + (int64_t)gh * kD + kc * 8,
                 valid ? 16u : 0u);
    }
    cp_async_commit();
    cp_async_wait_group<0>();
    fence_smem_to_async();
    mbar_arrive(bar);
  };
  if (warp == 10) {
    // ---------------- Q rows and the O1 products (warp 10) ----------------
    // O1^T = S Q^T into [dv lane][token column] (single BF16: the output is
    // BF16), issued here, beside the recurrence's MMAs, once the chunk's Q
    // rows and S parts are in place and the row warps have read the previous
    // chunk's outputs; Q is reloaded once O1 has read it.
    bool issued = false;
    uint32_t last_par = 0;
    if (records_ok) {
      const uint32_t id64 = idesc_bf16_f32(128, 64);
      const uint32_t sah = taddr + 128, qt = smem_u32(sm + kS2_Q);
      // Operand descriptors do not change across chunks: computed once, so
      // that the issuing lane spends no time on them between MMAs.
      uint64_t dq[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) dq[kk] = tile_desc(qt, 128, kk);
      for (int ci = 0; ci < nchunks; ++ci) {
        const uint32_t par = ci & 1;
        if (ci > 0 && !wait(bO1, (ci - 1) & 1)) break;
        rows(ci, q, kS2_Q, bQ);
        bool ok = wait(bQ, par);
        ok = wait(bSr, par) && ok;
        if (ci > 0) ok = wait(bOr, (ci - 1) & 1) && ok;
        // Issued once the X products are done, so that O1 fills the tensor
        // pipe while the row warps compute Delta instead of delaying X.
        ok = wait(bX, par) && ok;
        __syncwarp();
        fence_after_sync();
        if (ok && lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_bf16_tmem_a(taddr + 384, sah + 8 * kk, dq[kk], id64, kk > 0);
          mma_commit(bO1);
          issued = true;
          last_par = par;
        }
        __syncwarp();
        if (!ok) break;
      }
    }
    // Bounded, not abortable: the MMAs in flight must finish before exit.
    if (lane == 0 && issued && !mbar_wait(bO1, last_par)) record_device_status(GDN_ERR_TIMEOUT);
    __syncwarp();
  } else if (warp == 11) {
    // ---------------- K rows (warp 11) ----------------
    if (records_ok) {
      rows(0, k, kS2_K, bK);
      for (int ci = 0; ci + 1 < nchunks; ++ci) {
        // K is free once the chunk's S update has read it.
        if (wait(bS, ci & 1)) rows(ci + 1, k, kS2_K, bK);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------- record copies and output stores ----------------
    // Outstanding bulk copies (lane 0's view), drained on exit.
    int pend_w = -1, pend_u = -1, pend_p = -1;
    auto copy_w = [&](int ci) {
      mbar_arrive_expect_tx(bW, 32768 + 768);
      bulk_g2s(sm + kS2_W, rec_of(ci) + kOffW, 32768, bW);
      bulk_g2s(sm + kS2_GK, rec_of(ci) + kOffGK, 768, bW);
      pend_w = ci;
    };
    auto copy_u = [&](int ci) {
      mbar_arrive_expect_tx(bU, 32768);
      bulk_g2s(sm + kS2_U, rec_of(ci) + kOffU, 32768, bU);
      pend_u = ci;
    };
    auto copy_p = [&](int ci) {
      mbar_arrive_expect_tx(bP, 8192);
      bulk_g2s(sm + kS2_P, rec_of(ci) + kOffP, 8192, bP);
      pend_p = ci;
    };
    if (records_ok) {
      if (lane == 0) {
        copy_w(0);
        copy_u(0);
        copy_p(0);
      }
      for (int ci = 0; ci + 1 < nchunks; ++ci) {
        const uint32_t par = ci & 1;
        // Each buffer is refilled once the chunk's last reader of it is
        // done; these events happen in this order.
        if (wait(bX, par) && lane == 0) copy_w(ci + 1);
        if (wait(bDr, par) && lane == 0) copy_u(ci + 1);
        if (wait(bO, par) && lane == 0) copy_p(ci + 1);
      }
    }
    if (lane == 0) {
      // Bounded, not abortable: copies in flight must land before exit.
      bool drained = true;
      if (pend_w >= 0) drained = mbar_wait(bW, pend_w & 1) && drained;
      if (pend_u >= 0) drained = mbar_wait(bU, pend_u & 1) && drained;
      if (pend_p >= 0) drained = mbar_wait(bP, pend_p & 1) && drained;
      if (!drained) record_device_status(GDN_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---------------- MMAs (one lane) ----------------
    if (lane == 0 && records_ok) {
      const uint32_t id64 = idesc_bf16_f32(128, 64), id128 = idesc_bf16_f32(128, 128);
      const uint32_t sah = taddr + 128, sal = taddr + 192;   // S hi / lo in TMEM
      const uint32_t w = smem_u32(sm + kS2_W);
      const uint32_t p = smem_u32(sm + kS2_P), kt = smem_u32(sm + kS2_K);
      // TMEM column of K step kk (16 tokens) of a Delta part based at `col`
      auto dcol = [&](int col, int kk) { return taddr + col + 8 * kk + (kk >= 2 ? 16 : 0); };
      // Operand descriptors do not change across chunks: computed once, so
      // that the issuing lane spends no time on them between MMAs.
      uint64_t dw[8], dk4[4], dp4[4];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) dw[kk] = mn_desc(w, 128, kk);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        dk4[kk] = mn_desc(kt, 128, kk);
        dp4[kk] = tile_desc(p, 64, kk);
      }
      uint64_t* last = nullptr;
      uint32_t last_par = 0;
      for (int ci = 0; ci < nchunks; ++ci) {
        const uint32_t par = ci & 1;
        // X^T = S W^T: cols [256, 320) S_hi W_hi^T + S_lo W_hi^T, cols
        // [320, 384) S_hi W_lo^T (the record's W tile is [W hi; W lo], N = 128);
        // one K = 16 step of a TMEM A operand is 8 columns.
        bool ok = wait(bW, par);
        ok = wait(bSr, par) && ok;
        fence_after_sync();
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_bf16_tmem_a(taddr + 256, sah + 8 * kk, dw[kk], id128 | kTransB, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_bf16_tmem_a(taddr + 256, sal + 8 * kk, dw[kk], id64 | kTransB, 1);
          mma_commit(bX);
        }
        // S += (Delta^T D) K (hi and lo passes);  O2^T = Delta^T P^T.
        // The S update needs Delta and K only; O2 also needs P, whose copy
        // may still be landing: waited for after the S update is issued.
        ok = wait(bDr, par);
        ok = wait(bK, par) && ok;
        fence_after_sync();
        if (ok) {
          const uint32_t idk = id128 | kTransB;
          // A operands in TMEM: tokens 0-31 of each part in the hf = 0 columns,
          // tokens 32-63 in the hf = 1 columns (32 further on).
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16_tmem_a(taddr, dcol(256, kk), dk4[kk], idk, 1);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16_tmem_a(taddr, dcol(272, kk), dk4[kk], idk, 1);
          mma_commit(bS);
          last = bS;   // the last commit so far (drained on exit)
          last_par = par;
          ok = wait(bP, par);
          fence_after_sync();
        }
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16_tmem_a(taddr + 448, dcol(320, kk), dp4[kk], id64, kk > 0);
          mma_commit(bO);
          last = bO;
          last_par = par;
        }
      }
      // Bounded, not abortable: the MMAs in flight must finish before exit.
      if (last != nullptr && !mbar_wait(last, last_par)) record_device_status(GDN_ERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- rows (warps 0-7) ----------------
    const bool init = has_init != nullptr && has_init[seq] != 0;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const int c0 = 64 * hf + 32 * blk;
      float vbuf[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f4 = init ? *reinterpret_cast<const float4*>(Sg + c0 + e)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        vbuf[e] = f4.x; vbuf[e + 1] = f4.y; vbuf[e + 2] = f4.z; vbuf[e + 3] = f4.w;
      }
      tmem_st32(tmem_warp_addr(taddr, c0), vbuf);
    }
    auto row_sync = [&]() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    // Outputs of chunk cj: o_r = e^{g_r} rq_r O1_r + O2_r, in two parts.
    // stage_outputs: row thread (i, hf) holds output dv = i of tokens
    // [32 hf, 32 hf + 32); it releases the accumulators and stages the values
    // as [token][dv] BF16, 256 bytes per token with its 16-byte chunks
    // XOR-swizzled by the token (a warp's stores for one token fill 64
    // contiguous bytes). copy_outputs, after the next Delta (so that it
    // overlaps the S update instead of the X products) and a barrier of the
    // row threads: all of them write the staged rows out as whole 256-byte
    // rows of o (16 lanes per row), so that each warp store covers four full
    // lines.
    unsigned char* stg = sm + kS2_STG;
    auto stage_outputs = [&](int cj) {
      wait(bO1, cj & 1);
      wait(bO, cj & 1);
      __syncwarp();
      fence_after_sync();
      float o1[32], o2[32];
      tmem_ld32x2(tmem_warp_addr(taddr, 384 + 32 * hf), tmem_warp_addr(taddr, 448 + 32 * hf), o1, o2);
      fence_before_sync();
      mbar_arrive(bOr);
      const float4* qv = reinterpret_cast<const float4*>(qs + 64 * (cj & 1) + 32 * hf);
      const int jc = row >> 3, jb = (row & 7) * 2;
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 q4 = qv[e4];
        const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 32 * hf + 4 * e4 + e;
          *reinterpret_cast<__nv_bfloat16*>(stg + r * 256 + ((jc ^ (r & 15)) << 4) + jb) =
              __float2bfloat16_rn(fmaf(o1[4 * e4 + e], qq[e], o2[4 * e4 + e]));
        }
      }
    };
    auto copy_outputs = [&](int cj) {
      const int c0 = start + cj * kC;
      const int n = min(kC, end - c0);
      row_sync();   // every thread's staging is written
      if (!failed()) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int t = (p * kRowThreads + tid) >> 4, j = tid & 15;
          if (t < n)
            *reinterpret_cast<uint4*>(o + ((int64_t)(c0 + t) * Hv + h) * kD + 8 * j) =
                *reinterpret_cast<const uint4*>(stg + t * 256 + ((j ^ (t & 15)) << 4));
        }
      }
      // The next stage_outputs comes after the next chunk's first row
      // barrier, so the staging is read before it is overwritten.
    };

    for (int ci = 0; ci < nchunks && records_ok; ++ci) {
      const int c0 = start + ci * kC;
      const int n = min(kC, end - c0);
      const uint32_t par = ci & 1;
      // Once the previous chunk's S update is done, so are every row
      // thread's reads of the gate buffers this chunk refills (Delta two
      // chunks ago, the outputs of two chunks ago), and the MMAs that read
      // the previous S hi/lo parts. The record's gates are refilled only
      // after this chunk's X MMAs, which wait for the S parts below.
      if (ci > 0) wait(bS, (ci - 1) & 1);
      wait(bW, par);
      // The record's gates are read now (the buffer is refilled once this
      // chunk's X products, which wait for the split below, are done); the
      // per-token decay vectors are formed after the split, off its path.
      const float glast = gk[n - 1];
      float* dkb = dks + 64 * par;
      float g_t = 0.f, rk_t = 0.f, rq_t = 0.f;
      if (tid < 64) {
        g_t = gk[tid];
        rk_t = gk[64 + tid];
        rq_t = gk[128 + tid];
      }
      // (b) this thread's half of S row i -> BF16 hi/lo pairs in TMEM (the
      // X and O1 MMAs' A operands), then S <- e^{g_last} S.
      __syncwarp();
      fence_after_sync();
      {
        const int cb0 = 64 * hf, cb1 = 64 * hf + 32;
        float s0[32], s1[32];
        tmem_ld32x2(tmem_warp_addr(taddr, cb0), tmem_warp_addr(taddr, cb1), s0, s1);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const float* sv = part ? s1 : s0;
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            hi[e] = pack_bf16x2(sv[2 * e], sv[2 * e + 1]);
            lo[e] = pack_bf16x2(sv[2 * e] - bf16lo(hi[e]), sv[2 * e + 1] - bf16hi(hi[e]));
          }
          // The previous chunk's O1 (issued by warp 10) reads S hi until its
          // commit.
          if (part == 0 && ci > 0) {
            wait(bO1, (ci - 1) & 1);
            __syncwarp();
            fence_after_sync();
          }
          // dk j = 64 hf + 32 part + 2 e + {0, 1} -> column j / 2
          tmem_st16x2(tmem_warp_addr(taddr, 128 + 32 * hf + 16 * part),
                      tmem_warp_addr(taddr, 192 + 32 * hf + 16 * part), hi, lo);
        }
        fence_before_sync();
        mbar_arrive(bSr);
        if (tid < 64) {
          const bool in = tid < n;
          dkb[tid] = in ? exp2_nonpos(glast - g_t) * rk_t : 0.f;
          qs[64 * par + tid] = in ? exp2_nonpos(g_t) * rq_t : 0.f;
        }
        const float gamma_c = exp2_nonpos(glast);
        // S <- e^{g_last} S, off the X MMAs' path: only this chunk's S update
        // (after Delta, whose barrier also orders this store) touches S next.
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          s0[e] *= gamma_c;
          s1[e] *= gamma_c;
        }
        tmem_st32x2(tmem_warp_addr(taddr, cb0), tmem_warp_addr(taddr, cb1), s0, s1);
      }
      row_sync();   // dks and qs are written before they are read
      // The previous chunk's outputs released and staged while this chunk's
      // X MMAs run.
      if (ci > 0) stage_outputs(ci - 1);
      // (d) Delta^T = U^T - X^T for row i, tokens [32 hf, 32 hf + 32).
      wait(bX, par);
      __syncwarp();
      fence_after_sync();
      {
        float xv[32], xl[32];
        tmem_ld32x2(tmem_warp_addr(taddr, 256 + 32 * hf), tmem_warp_addr(taddr, 320 + 32 * hf),
                    xv, xl);
#pragma unroll
        for (int e = 0; e < 32; ++e) xv[e] += xl[e];
        wait(bU, par);
        // Delta and (Delta D) hi / lo as BF16 pairs of consecutive tokens,
        // written over this thread's own X columns (already read): (Delta D)
        // hi at [256 + 32 hf, + 16), lo at [272 + 32 hf, + 16), Delta at
        // [320 + 32 hf, + 16); the MMAs read them as A operands (K = tokens).
        uint32_t dl[16], dh[16], dlo[16];
#pragma unroll
        for (int e8 = 0; e8 < 4; ++e8) {
          const float4 u0 = us[row * 16 + ((8 * hf + 2 * e8) ^ (row & 7))];
          const float4 u1 = us[row * 16 + ((8 * hf + 2 * e8 + 1) ^ (row & 7))];
          const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          float del[8], dd[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int r = 32 * hf + 8 * e8 + e;
            del[e] = r < n ? uu[e] - xv[8 * e8 + e] : 0.f;
            dd[e] = del[e] * dkb[r];
          }
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            dl[4 * e8 + e2] = pack_bf16x2(del[2 * e2], del[2 * e2 + 1]);
            const uint32_t hv = pack_bf16x2(dd[2 * e2], dd[2 * e2 + 1]);
            dh[4 * e8 + e2] = hv;
            dlo[4 * e8 + e2] = pack_bf16x2(dd[2 * e2] - bf16lo(hv), dd[2 * e2 + 1] - bf16hi(hv));
          }
        }
        tmem_st16x2(tmem_warp_addr(taddr, 256 + 32 * hf), tmem_warp_addr(taddr, 272 + 32 * hf), dh,
                    dlo);
        tmem_st16(tmem_warp_addr(taddr, 320 + 32 * hf), dl);
      }
      fence_before_sync();
      mbar_arrive(bDr);
      if (ci > 0) copy_outputs(ci - 1);
    }
    if (records_ok && nchunks > 0) {
      row_sync();   // the last copy_outputs is done with the staging
      stage_outputs(nchunks - 1);
      copy_outputs(nchunks - 1);
      wait(bS, (nchunks - 1) & 1);
      __syncwarp();
      fence_after_sync();
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int cb = 64 * hf + 32 * blk;
        float sv[32];
        tmem_ld32(tmem_warp_addr(taddr, cb), sv);
        if (!failed()) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(Sg + cb + e) =
                make_float4(sv[e], sv[e + 1], sv[e + 2], sv[e + 3]);
        }
      }
    }
    if (tid == 0 && (failed() || !records_ok)) {
      atomicExch(hdr + 2, (int)(failed() ? GDN_ERR_TIMEOUT : GDN_ERR_INVALID_ARG));
      if (failed()) record_device_status(GDN_ERR_TIMEOUT);
    }
    __syncwarp();
  }
  cp_async_wait_all();
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, 512);
}

}  // namespace

size_t prefill_tc_workspace_bytes(int32_t T, int32_t N, int32_t Hv) {
  return tc_layout(T, N, Hv).total;
}

gdn_status_t launch_prefill_tc_plan(const int32_t* cu, int32_t N, int32_t T, int32_t Hv,
                                    void* workspace, cudaStream_t st) {
  const TcLayout L = tc_layout(T, N, Hv);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws);
  return launch_build_chunks(cu, N, kC, reinterpret_cast<gdn_conv_chunk_t*>(ws + L.desc_off),
                             L.capacity, hdr, hdr + 1, st,
                             reinterpret_cast<int32_t*>(ws + L.order_off));
}

gdn_status_t launch_prefill_tc(const void* q, const void* k, int64_t qk_stride, const void* v,
                               int64_t v_stride, const float* a, const float* b,
                               const int32_t* cu, int32_t N, int32_t T, float* S,
                               const uint8_t* has_init, void* o, int32_t Hk, int32_t Hv,
                               int32_t flags, void* workspace, cudaStream_t st,
                               StateSlots slots) {
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
  int32_t* order = reinterpret_cast<int32_t*>(ws + L.order_off);
  gdn_status_t rc = GDN_OK;
  if (!(flags & kFlagPlanned)) {
    rc = launch_build_chunks(cu, N, kC, desc, L.capacity, hdr, hdr + 1, st, order);
    if (rc != GDN_OK) return rc;
  }
  if ((rc = check_launch(launch_pdl(
           tc_chunk_kernel, dim3(L.capacity, Hv), dim3(kThreads), kS1_BYTES, st,
           static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(q), qk_stride,
           static_cast<const __nv_bfloat16*>(v), v_stride, a, b, (const int32_t*)hdr, desc, T, Hk,
           Hv, flags, records, hdr))) != GDN_OK)
    return rc;
  return check_launch(launch_pdl(
      tc_state_kernel, dim3(N * Hv), dim3(kThreads2), kS2_BYTES, st,
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qk_stride, cu,
      T, Hk, S, has_init, static_cast<__nv_bfloat16*>(o), Hv, (const unsigned char*)records,
      hdr, (const int32_t*)order, N, slots));
}

GDN_DEFINE_STATUS_GATHER(gather_status_prefill_tc)

}  // namespace gdn
