// kda_umma.cuh -- 5th-generation tensor core (tcgen05) helpers for sm_103a, as inline PTX:
// tensor-memory allocation, shared-memory matrix descriptors for K-major tiles with 128-byte swizzle,
// instruction descriptors for kind::tf32 / kind::f16 (bf16) with fp32 accumulation, MMA issue and
// commit, and tensor-memory loads / stores.
//
// Operand tiles ("K-major, 128B swizzle"): a tile of R rows x K elements is stored as K / (128/esize)
// column chunks, each chunk R rows x 128 bytes; chunk c starts at c * R * 128 bytes (1024-byte aligned),
// and the 16-byte group g of row r sits at group g ^ (r % 8).  One MMA instruction consumes 32 bytes
// of K (8 tf32 or 16 bf16 elements); successive instructions advance the descriptor's start address by
// 32 bytes inside a chunk and by R * 128 bytes across chunks.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_device.cuh"

namespace kda {
namespace umma {

// Byte offset of element (r, k) of a K-major SW128 tile with R rows, for element size ESZ.
template <int ESZ>
__device__ __forceinline__ uint32_t sw128_offset(int R, int r, int k) {
    constexpr int KC = 128 / ESZ;  // elements per 128-byte row chunk
    const int c = k / KC;
    const int kb = (k - c * KC) * ESZ;
    return (uint32_t)(c * R * 128 + r * 128 + ((((kb >> 4) ^ (r & 7)) << 4) | (kb & 15)));
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t t;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(x));
    return t;
}

__device__ __forceinline__ void st_tf32(uint8_t *tile, int R, int r, int k, float x) {
    *reinterpret_cast<uint32_t *>(tile + sw128_offset<4>(R, r, k)) = to_tf32(x);
}

__device__ __forceinline__ void st_bf16(uint8_t *tile, int R, int r, int k, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(tile + sw128_offset<2>(R, r, k)) = __float2bfloat16_rn(x);
}

// 16-byte stores of 4 consecutive tf32 (k0 % 4 == 0) / 8 consecutive bf16 (k0 % 8 == 0) elements of a row.
__device__ __forceinline__ void st_tf32x4(uint8_t *tile, int R, int r, int k0, float x0, float x1, float x2,
                                          float x3) {
    *reinterpret_cast<uint4 *>(tile + sw128_offset<4>(R, r, k0)) = make_uint4(to_tf32(x0), to_tf32(x1), to_tf32(x2),
                                                                              to_tf32(x3));
}

// two floats rounded to bf16 (nearest even) in one conversion, lo in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void st_bf16x8(uint8_t *tile, int R, int r, int k0, const float *x) {
    *reinterpret_cast<uint4 *>(tile + sw128_offset<2>(R, r, k0)) =
        make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

// Shared-memory matrix descriptor: start address, leading / stride byte offsets, 128B swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(16 >> 4) << 16;     // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: 8 rows x 128 bytes
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

// Descriptor of the 32-byte K slice `ks` (0-based, in units of one instruction's K) of a tile.
__device__ __forceinline__ uint64_t sdesc_k(const uint8_t *tile, int R, int ks) {
    const int c = ks >> 2;  // 4 instructions per 128-byte chunk
    const uint32_t a = smem_addr(tile) + (uint32_t)(c * R * 128 + (ks & 3) * 32);
    return sdesc(a);
}

// Descriptor of K slice `ks` from the descriptor of slice 0 of the same tile: only the start-address field
// advances (by 32 bytes within a 128-byte chunk, by R * 128 bytes across chunks).  Shared-memory addresses
// stay below 2^18 bytes, so the 14-bit field (address / 16) never carries into the next field.
__device__ __forceinline__ uint64_t sdesc_at(uint64_t d0, int R, int ks) {
    return d0 + (uint64_t)((((ks >> 2) * R * 128) + (ks & 3) * 32) >> 4);
}

// Instruction descriptor: fp32 accumulate, K-major A and B, M x N; kind = 1 (bf16) or 2 (tf32).
__device__ __forceinline__ uint32_t idesc(int fmt, int M, int N, bool negate_a = false) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((negate_a ? 1u : 0u) << 13) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr int kBF16 = 1;
constexpr int kTF32 = 2;

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, bool acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc));
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, bool acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc));
}

// Arrive once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Warp-wide: allocate / free `ncols` tensor-memory columns (power of two >= 32).
__device__ __forceinline__ void alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Warp-wide: 32 lanes (this warp's quarter) x 32 consecutive columns -> r[32] per thread.
__device__ __forceinline__ void ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Warp-wide: store v[32] per thread into 32 lanes x 32 consecutive columns.
__device__ __forceinline__ void st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
        "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
        "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
        "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warp-wide, asynchronous: issue the load of 32 lanes x 32 consecutive columns into r[32].  The values are
// valid only after wait_ld(r), which ties r to the wait so that no use of them is scheduled above it.
__device__ __forceinline__ void ld32_issue(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// Warp-wide, asynchronous: 32 lanes x 16 consecutive columns into r[16]; valid after wait_ld16(r).
__device__ __forceinline__ void ld16_issue(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void wait_ld16(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void wait_ld(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                   "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Warp-wide, asynchronous: store v[32] into 32 lanes x 32 consecutive columns; wait_st() waits for every
// tensor-memory store this thread issued.
__device__ __forceinline__ void st32_issue(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]),
        "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]),
        "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace umma
}  // namespace kda
