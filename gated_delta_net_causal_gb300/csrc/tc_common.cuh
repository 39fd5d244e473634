// Tensor-core (tcgen05 / TMEM) and TMA building blocks for sm_103a, as inline
// PTX. Layout conventions used throughout:
//
//  * Shared-memory operand tiles are K-major with the 128-byte swizzle: a tile
//    of R rows is stored as ceil(K*elem/128) "K atoms"; atom a holds bytes
//    [128a, 128a+128) of every row, rows 128 B apart, and inside each 8-row
//    group (1024 B) the 16-byte chunk j of row r sits at chunk (j ^ (r & 7)).
//    Tiles start on a 1024-byte boundary. This is the layout a TMA load with
//    CU_TENSOR_MAP_SWIZZLE_128B writes for a box whose inner extent is 128 B.
//  * One MMA instruction consumes 32 bytes of K (16 bf16/f16, 8 tf32), so the
//    descriptor of k-step s starts (s / 4) atoms and (s % 4) * 32 B in.
//  * TMEM addresses are (lane << 16) | column.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {
namespace tc {

// ------------------------------------------------------------ descriptors

// Byte offset of element (r, k) in a K-major SW128 tile of `rows` rows whose
// elements are `esize` bytes.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows, int esize) {
  const int kb = k * esize;               // byte position along K
  const int atom = kb >> 7;               // 128-byte K atom
  const int chunk = (kb >> 4) & 7;        // 16-byte chunk inside the atom
  const int within = kb & 15;
  return (uint32_t)(atom * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((chunk ^ (r & 7)) << 4) + within);
}

// Shared-memory matrix descriptor for a K-major SW128 tile (Blackwell form:
// start >> 4 in bits 0-13, leading offset 16-29 (unused here), stride offset
// 32-45 = 1024 B between 8-row groups, version 1 in bits 46-47, layout type
// SWIZZLE_128B (2) in bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (ignored for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
  return d;
}

// Descriptor of k-step `s` (32 bytes of K each) of a K-major SW128 tile.
__device__ __forceinline__ uint64_t sdesc_kstep(uint32_t tile_addr, int rows, int s) {
  return sdesc_sw128(tile_addr + (uint32_t)((s >> 2) * rows * 128 + (s & 3) * 32));
}

// Descriptor of k-step `s` advanced from a tile's base descriptor (the start
// address field is linear; shared addresses stay below 256 KB).
__device__ __forceinline__ uint64_t sdesc_at(uint64_t base, int rows, int s) {
  return base + (uint64_t)(((s >> 2) * rows * 128 + (s & 3) * 32) >> 4);
}

enum : uint32_t { kF16 = 0, kBF16 = 1, kTF32 = 2 };

// Instruction descriptor for kind::f16 / kind::tf32 with fp32 accumulation,
// both operands K-major: D format (bits 4-5) = F32, A/B formats in bits 7-9 /
// 10-12, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ __forceinline__ uint32_t idesc(uint32_t ab_format, int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;
  d |= ab_format << 7;
  d |= ab_format << 10;
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

// fp32 -> tf32 with round-to-nearest (ties away); the tensor cores would
// otherwise drop the low 13 mantissa bits of an fp32 operand (truncation).
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// ------------------------------------------------------------------ TMEM

// Allocates `ncols` TMEM columns (power of two >= 32) for the CTA; the base
// address is written to *dst (shared). Executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------- MMA

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (K = 32 bytes).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                        bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M rows x 16 bf16/f16 of K) sits in
// TMEM, row m in lane m, K elements 2c and 2c+1 packed in column c (low half
// first); k-step s of a K-major A starts 8 s columns in.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                           bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}
// mma_f16_ts and mma_commit issued by one elected lane of a converged warp
// (every lane calls them with the same arguments).
__device__ __forceinline__ void mma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                                 bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}
// mma_f16 (both operands in shared memory) issued by one elected lane of a
// converged warp.
__device__ __forceinline__ void mma_f16_elect(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                              bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}
// two consecutive k-steps into one accumulator (the second accumulates)
// issued by one elected lane of a converged warp
__device__ __forceinline__ void mma_f16_elect2(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint64_t a1,
                                               uint64_t b1, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %5, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %5, 1;\n\t}" ::"r"(d_tmem),
      "l"(a0), "l"(b0), "l"(a1), "l"(b1), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// -------------------------------------------------------------- TMEM I/O
// 32x32b shape: thread t of the warp reads/writes lane (quadrant base + t),
// consecutive 32-bit columns.

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------- TMA
// 2-D tiled load of box (x = inner coordinate, y = row) into shared memory,
// completing `bytes` on the mbarrier.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled store of a box from shared memory (16-byte aligned source),
// tracked by the executing thread's bulk async-groups (commit, then
// wait_group). Rows or columns outside the tensor are not written. The box
// must start at a non-negative coordinate with x * element size a multiple
// of 16 bytes.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap),
               "r"(x), "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}

// ------------------------------------------------------- host: tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on libcuda); nullptr if the driver lacks it.
inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D map over `rows` rows of `cols` elements of `esize` bytes, rows
// `stride` elements apart; boxes of box_cols x box_rows. Out-of-range box
// elements read as zero.
inline bool make_map_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                        int64_t stride, uint32_t esize, CUtensorMapDataType dt, uint32_t box_cols,
                        uint32_t box_rows, CUtensorMapSwizzle sw,
                        CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)stride * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace gdn
