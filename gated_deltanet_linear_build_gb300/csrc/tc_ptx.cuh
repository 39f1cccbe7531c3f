// Thin inline-PTX wrappers for the Blackwell (sm_100 family) 5th-generation
// tensor core path: TMEM allocation, tcgen05.mma with shared-memory operand
// descriptors, commit to an mbarrier, TMEM <-> register moves, and the fences
// that order them. Written from the PTX ISA description of these instructions.
//
// Operand layout used throughout: K-major, no swizzle ("interleaved" core
// matrices). A tile of R rows (M or N index) by Kc columns (K index) of BF16 is
// stored as 8-row x 16-byte core matrices; core matrices adjacent along K are
// 128 bytes apart (the leading-dimension byte offset) and 8-row groups are
// Kc * 16 bytes apart (the stride-dimension byte offset):
//   byte(r, k) = (r / 8) * (Kc * 16) + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
// One MMA instruction consumes K = 16 (two core matrices along K), so the
// descriptor of K-step kk starts kk * 256 bytes after the tile base.
#pragma once

#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (r, k) inside a K-major no-swizzle tile with Kc columns.
__host__ __device__ __forceinline__ uint32_t tile_off(int r, int k, int Kc) {
  return (uint32_t)((r >> 3) * (Kc * 16) + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: start address, leading/stride byte offsets,
// descriptor version 1 (bits 46-47), no swizzle (bits 61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Descriptor of K-step kk of a K-major tile with Kc columns (rows from row0).
__device__ __forceinline__ uint64_t tile_desc(uint32_t tile_addr, int Kc, int kk, int row0 = 0) {
  return smem_desc(tile_addr + (uint32_t)(row0 >> 3) * (uint32_t)(Kc * 16) + (uint32_t)kk * 256u,
                   128u, (uint32_t)(Kc * 16));
}

// MN-major ("transposed") tile of R rows along M or N by Kc along K: core
// matrices are 8 K-rows x 16 bytes along MN; MN-adjacent core matrices are 128
// bytes apart (stride-dimension offset) and K-adjacent ones R * 16 bytes apart
// (leading-dimension offset):
//   byte(m, k) = (k / 8) * (R * 16) + (m / 8) * 128 + (k % 8) * 16 + (m % 8) * 2.
// Note byte(m, k) of an MN-major tile with R rows equals byte(k, m) of a K-major
// tile with Kc = R: a row-major [k][m] matrix stored as a K-major tile is, read
// with this descriptor, its own transpose.
__host__ __device__ __forceinline__ uint32_t mn_off(int m, int k, int R) {
  return (uint32_t)((k >> 3) * (R * 16) + (m >> 3) * 128 + (k & 7) * 16 + (m & 7) * 2);
}
__device__ __forceinline__ uint64_t mn_desc(uint32_t tile_addr, int R, int kk) {
  return smem_desc(tile_addr + (uint32_t)kk * 2u * (uint32_t)(R * 16), (uint32_t)(R * 16), 128u);
}
// Instruction-descriptor bits selecting MN-major A or B.
constexpr uint32_t kTransA = 1u << 15;
constexpr uint32_t kTransB = 1u << 16;

// Instruction descriptor, kind::f16: BF16 A and B (both K-major), float32 D,
// dense, no negation; N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ---- TMEM allocation (one full warp executes these) ------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(slot)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}

// ---- MMA issue and completion ----------------------------------------------
// D[tmem] (+)= A[smem desc] x B[smem desc]^T, one elected thread issues.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
      :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// D[tmem] (+)= A[tmem] x B[smem desc]^T: A in tensor memory, row m in lane m
// and its K elements as consecutive BF16 pairs along the columns (element k in
// column k / 2, the lower half for even k), so that one K = 16 step reads 8
// columns starting at a_tmem.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive (once) on the mbarrier when all previously issued MMAs complete.
__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      :: "r"(smem_u32(mbar)) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* mbar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
  return ok;
}

// Bounded wait that backs off with __nanosleep between polls, so that a
// waiting warp takes almost no issue slots from the working warps of its SM
// sub-partition (a plain poll loop issues several instructions per poll).
// Gives up after `max_polls` polls (each at least one poll instruction long;
// about 2 s at the sleep lengths used here) and returns false.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* mbar, uint32_t parity,
                                                unsigned sleep_ns = 32,
                                                unsigned max_polls = 1u << 26) {
  for (unsigned n = 0; n < max_polls; ++n) {
    if (mbar_try_wait(mbar, parity)) return true;
    __nanosleep(sleep_ns);
  }
  return false;
}

// Bounded wait for the phase with the given parity: gives up after about
// `max_cycles` SM clock cycles and returns false (the caller records
// GDN_ERR_TIMEOUT and unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity,
                                          long long max_cycles = 4000000000LL) {
  const long long t0 = clock64();
  while (!mbar_try_wait(mbar, parity)) {
    if (clock64() - t0 > max_cycles) return false;
  }
  return true;
}

// One plain arrival (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(mbar)) : "memory");
}

// ---- bulk (TMA, 1-D) and 16-byte asynchronous copies ----------------------
// Arm the mbarrier for `bytes` of incoming bulk copies (plus one arrival).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(mbar)), "r"(bytes) : "memory");
}
// Global -> shared bulk copy; completion is signalled on the mbarrier.
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(mbar)) : "memory");
}
// Shared -> global bulk copy (bulk-group completion). Addresses 16-byte
// aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(gmem_dst), "r"(smem_u32(smem_src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until this thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// 16-byte global -> shared copy; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src,
                                           uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N committed groups of this thread are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// ---- fences -----------------------------------------------------------------
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the tensor
// core (async proxy).
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMEM <-> registers (32 lanes x 32 columns per warp, 32-bit) ------------
// Warp w of a warpgroup may access TMEM lanes [32 (w % 4), 32 (w % 4) + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
         "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
         "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
         "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
         "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
         "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
         "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
         "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
         "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
         "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
         "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Two 32-column loads (possibly of different TMEM regions) and one wait, so
// that the second load's latency overlaps the first's.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&va)[32],
                                            float (&vb)[32]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb) : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[32 + i]);
  }
}

// Two 16-column stores of raw 32-bit words and one wait.
__device__ __forceinline__ void tmem_st16x2(uint32_t ta, uint32_t tb, const uint32_t (&va)[16],
                                            const uint32_t (&vb)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], "
      "{%18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(ta), "r"(tb), "r"(va[0]), "r"(va[1]), "r"(va[2]), "r"(va[3]), "r"(va[4]),
         "r"(va[5]), "r"(va[6]), "r"(va[7]), "r"(va[8]), "r"(va[9]), "r"(va[10]), "r"(va[11]),
         "r"(va[12]), "r"(va[13]), "r"(va[14]), "r"(va[15]), "r"(vb[0]), "r"(vb[1]), "r"(vb[2]),
         "r"(vb[3]), "r"(vb[4]), "r"(vb[5]), "r"(vb[6]), "r"(vb[7]), "r"(vb[8]), "r"(vb[9]),
         "r"(vb[10]), "r"(vb[11]), "r"(vb[12]), "r"(vb[13]), "r"(vb[14]), "r"(vb[15])
      : "memory");
}

// One 16-column store of raw 32-bit words and its wait.
__device__ __forceinline__ void tmem_st16(uint32_t ta, const uint32_t (&va)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(ta), "r"(va[0]), "r"(va[1]), "r"(va[2]), "r"(va[3]), "r"(va[4]), "r"(va[5]),
         "r"(va[6]), "r"(va[7]), "r"(va[8]), "r"(va[9]), "r"(va[10]), "r"(va[11]), "r"(va[12]),
         "r"(va[13]), "r"(va[14]), "r"(va[15])
      : "memory");
}

// Two 32-column stores and one wait.
__device__ __forceinline__ void tmem_st32x2(uint32_t ta, uint32_t tb, const float (&va)[32],
                                            const float (&vb)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], "
      "{%34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(ta), "r"(tb), "r"(__float_as_uint(va[0])), "r"(__float_as_uint(va[1])), "r"(__float_as_uint(va[2])), "r"(__float_as_uint(va[3])), "r"(__float_as_uint(va[4])), "r"(__float_as_uint(va[5])), "r"(__float_as_uint(va[6])), "r"(__float_as_uint(va[7])), "r"(__float_as_uint(va[8])), "r"(__float_as_uint(va[9])), "r"(__float_as_uint(va[10])), "r"(__float_as_uint(va[11])), "r"(__float_as_uint(va[12])), "r"(__float_as_uint(va[13])), "r"(__float_as_uint(va[14])), "r"(__float_as_uint(va[15])), "r"(__float_as_uint(va[16])), "r"(__float_as_uint(va[17])), "r"(__float_as_uint(va[18])), "r"(__float_as_uint(va[19])), "r"(__float_as_uint(va[20])), "r"(__float_as_uint(va[21])), "r"(__float_as_uint(va[22])), "r"(__float_as_uint(va[23])), "r"(__float_as_uint(va[24])), "r"(__float_as_uint(va[25])), "r"(__float_as_uint(va[26])), "r"(__float_as_uint(va[27])), "r"(__float_as_uint(va[28])), "r"(__float_as_uint(va[29])), "r"(__float_as_uint(va[30])), "r"(__float_as_uint(va[31])), "r"(__float_as_uint(vb[0])), "r"(__float_as_uint(vb[1])), "r"(__float_as_uint(vb[2])), "r"(__float_as_uint(vb[3])), "r"(__float_as_uint(vb[4])), "r"(__float_as_uint(vb[5])), "r"(__float_as_uint(vb[6])), "r"(__float_as_uint(vb[7])), "r"(__float_as_uint(vb[8])), "r"(__float_as_uint(vb[9])), "r"(__float_as_uint(vb[10])), "r"(__float_as_uint(vb[11])), "r"(__float_as_uint(vb[12])), "r"(__float_as_uint(vb[13])), "r"(__float_as_uint(vb[14])), "r"(__float_as_uint(vb[15])), "r"(__float_as_uint(vb[16])), "r"(__float_as_uint(vb[17])), "r"(__float_as_uint(vb[18])), "r"(__float_as_uint(vb[19])), "r"(__float_as_uint(vb[20])), "r"(__float_as_uint(vb[21])), "r"(__float_as_uint(vb[22])), "r"(__float_as_uint(vb[23])), "r"(__float_as_uint(vb[24])), "r"(__float_as_uint(vb[25])), "r"(__float_as_uint(vb[26])), "r"(__float_as_uint(vb[27])), "r"(__float_as_uint(vb[28])), "r"(__float_as_uint(vb[29])), "r"(__float_as_uint(vb[30])), "r"(__float_as_uint(vb[31]))
      : "memory");
}

// TMEM address of (lane quarter of this warp, column col).
__device__ __forceinline__ uint32_t tmem_warp_addr(uint32_t base, int col) {
  const uint32_t quarter = (threadIdx.x >> 5) & 3u;
  return base + ((quarter * 32u) << 16) + (uint32_t)col;
}

}  // namespace tc
}  // namespace gdn
