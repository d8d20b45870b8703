// tc_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family)
// tensor-core path: TMEM allocation, tcgen05.mma with shared-memory operand
// descriptors, tcgen05.commit to an mbarrier, TMEM loads/stores, and bounded
// mbarrier waits. Written from the public PTX ISA description of tcgen05.
//
// Operand layout used throughout (no swizzle, K-major): a tile of R rows x Kd
// columns of 16-bit elements is stored as 8x8 "core matrices" of 128 bytes
// (8 rows x 16 bytes); element (r, k) lives at byte
//     (r / 8) * SBO + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2,
// SBO = (Kd / 8) * 128: core matrices adjacent along K are 128 bytes apart
// (the descriptor's leading-dimension offset), 8-row groups SBO apart (its
// stride-dimension offset).
#pragma once

#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__host__ __device__ constexpr uint32_t km_offset(int r, int k, int Kd)
{
    return (uint32_t)((r >> 3) * (Kd / 8) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: start address, leading byte offset (between
// core matrices along K), stride byte offset (between 8-row groups), the fixed
// descriptor version bits 46..48 = 0b001, base offset 0, no swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// 128-byte-swizzled K-major tile of 16-bit elements, `rows` x 128: atoms of 8
// rows x 64 elements (8 x 128 bytes, 1024-byte aligned) in which the 16-byte
// chunk index of a row is XOR-ed with address bits 7-9 (the row within the
// atom); atoms run down the rows 1024 bytes apart, and the two 64-element
// halves of K are rows * 128 bytes apart. Byte offset of element (r, k).
__host__ __device__ constexpr uint32_t sw128_offset(int r, int k, int rows)
{
    return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                      ((((k >> 3) & 7) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// Descriptor of such a tile starting at saddr (an atom row start plus the
// K offset within the 128-byte row): stride byte offset 1024 between 8-row
// groups, leading byte offset unused, version bits 46..48 = 0b001, base
// offset 0 (atoms are 1024-byte aligned), layout type 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, dense: D format bits 4-5 = 1 (f32), A format bits
// 7-9 = 1 (bf16), B format bits 10-12 = 1 (bf16), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive (once) on the mbarrier when every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(mbar), "r"(count));
}

// Wait for the phase with the given parity to complete, giving up after
// `limit` polls. Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, int limit)
{
    uint32_t done = 0;
    for (int it = 0; it < limit; ++it) {
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done)
            return true;
    }
    return false;
}

// TMEM allocation: executed by one whole warp; the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(slot_saddr), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_smem_to_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31; the lane offset is bits 16.. of the address).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                    "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                    "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                    "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                    "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                    "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                    "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace gdn
