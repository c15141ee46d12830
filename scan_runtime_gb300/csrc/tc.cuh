// tc.cuh -- fifth-generation tensor-core (tcgen05) helpers for sm_103a:
// tensor-memory allocation, shared-memory matrix descriptors, the tf32 MMA,
// commits to an mbarrier and loads from tensor memory.
//
// Operand layout used throughout: K-major with no swizzle.  A matrix with R
// rows and KD elements along K is stored as 8-row x 16-byte core matrices;
// element (r, k) sits at float offset kmajor_off(r, k, KD); the core matrices
// adjacent along K are 128 bytes apart (leading byte offset) and the 8-row
// groups (KD / 4) * 128 bytes apart (stride byte offset).  One kind::tf32
// MMA consumes 8 elements of K, i.e. the descriptor start advances 256 bytes.
// For M = 128 (cta_group::1) accumulator row r lives in tensor-memory lane r.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace sn {
namespace tc {

__device__ __forceinline__ int kmajor_off(int r, int k, int KD) {
    return (r >> 3) * (KD >> 2) * 32 + (k >> 2) * 32 + (r & 7) * 4 + (k & 3);
}

// Shared-memory matrix descriptor (no swizzle): start, leading and stride
// byte offsets in 16-byte units, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// 128-byte-swizzled K-major operand (the layout a TMA copy with 128-byte
// swizzle writes): atoms of 32 K elements (128 B) x R rows, rows 128 B apart,
// 8-row groups 1024 B apart, the 16-byte chunks of each row permuted by XOR
// with (row mod 8).  Atoms must start at 1024-byte boundaries.  Within an atom
// one kind::tf32 MMA (K = 8) advances the start by 32 bytes; the next atom is
// R * 128 bytes further.  Fields: leading offset 16 B (unused), stride offset
// 1024 B, version 1, swizzle mode 128 B (value 2 in bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::tf32: fp32 accumulator, tf32 A and B, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Round to the nearest tf32 value (kept in a 32-bit container).
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Whole warp: allocate `ncols` tensor-memory columns, address written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

// Whole warp: the same, keeping the CTA's permit to allocate again (a CTA
// that frees its columns and allocates once more, as the roles of one fused
// kernel do, must not have given it up; with one CTA per SM nothing waits on
// it).
__device__ __forceinline__ void tmem_alloc_keep(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols));
}

// Whole warp: release the allocation.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A * B^T, M x N x 8, one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// The mbarrier arrives once every tcgen05 operation this thread issued is done.
__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Issue the K/8 MMAs of D = A * B^T with A (M x KD) and B (N x KD) K-major.
__device__ __forceinline__ void gemm_tf32(uint32_t d_tmem, const float* A, const float* B, int KD, uint32_t idesc,
                                          bool accumulate) {
    const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
    const uint32_t sbo = (uint32_t)(KD >> 2) * 128u;
    for (int kk = 0; kk < KD / 8; ++kk)
        mma_tf32(d_tmem, smem_desc(a0 + kk * 256, 128, sbo), smem_desc(b0 + kk * 256, 128, sbo), idesc,
                 accumulate || kk > 0);
}

// D = A * B^T with K = 128, M = N = 128 rows, A and B both 128-byte-swizzled
// (four atoms of 32 K elements, 16 KB apart).
__device__ __forceinline__ void gemm_tf32_sw_sw(uint32_t d_tmem, const float* A, const float* B, uint32_t idesc,
                                                bool accumulate) {
    const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
    for (int kk = 0; kk < 16; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u;
        mma_tf32(d_tmem, smem_desc_sw128(a0 + off), smem_desc_sw128(b0 + off), idesc, accumulate || kk > 0);
    }
}

// D = A * B^T with K = 128: A 128-byte-swizzled (128 rows, atoms 16 KB apart),
// B in the plain K-major layout above.
__device__ __forceinline__ void gemm_tf32_sw_plain(uint32_t d_tmem, const float* A, const float* B, uint32_t idesc,
                                                   bool accumulate) {
    const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
    for (int kk = 0; kk < 16; ++kk) {
        const uint32_t aoff = (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u;
        mma_tf32(d_tmem, smem_desc_sw128(a0 + aoff), smem_desc(b0 + kk * 256, 128, 32 * 128), idesc,
                 accumulate || kk > 0);
    }
}

// Warp-collective load of 16 consecutive fp32 columns of this warp's 32 lanes.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

}  // namespace tc
}  // namespace sn
