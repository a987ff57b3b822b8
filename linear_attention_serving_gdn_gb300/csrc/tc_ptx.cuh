// Thin inline-PTX wrappers for the sm_100-family tensor-core path used by the
// chunked prefill: mbarriers, TMEM allocation, tcgen05.mma (kind::f16, A from
// shared memory or from TMEM), tcgen05.commit, tcgen05.ld / tcgen05.st and the
// shared-memory matrix
// descriptors of the canonical K-major and MN-major 128-byte-swizzled
// layouts.  Written from the PTX ISA description of these instructions.
#pragma once

#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe: true if the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// max_polls polls (each try_wait itself blocks for a bounded time) and
// returns false so the caller can report a timeout instead of hanging.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t max_polls) {
    for (uint32_t i = 0; i < max_polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---- fences -----------------------------------------------------------------

// Generic-proxy shared-memory writes become visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- TMEM allocation (one full warp) ------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- MMA ------------------------------------------------------------------------

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 operands, fp32 accumulation.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with the A operand in TMEM: row m of A is TMEM lane m, its K
// elements packed two per 32-bit column (the lower K index in the low half);
// a K step of 16 elements advances a_tmem by 8 columns.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on bar when every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(int M, int N) {
    return (1u << 4)                                 // D format: F32
           | (0u << 7) | (0u << 10)                  // A, B format: F16
           | (0u << 15) | (0u << 16)                 // A, B K-major
           | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// The same with B given MN-major (N contiguous in shared memory): the
// "transpose B" bit of the kind::f16 instruction descriptor.
__host__ __device__ constexpr uint32_t idesc_f16_f32acc_bmn(int M, int N) {
    return idesc_f16_f32acc(M, N) | (1u << 16);
}
// Modifier bits of the kind::f16 instruction descriptor: A given MN-major
// ("transpose A"), and both operands bf16 instead of fp16.
constexpr uint32_t kIdescAmn = 1u << 15;
constexpr uint32_t kIdescBmn = 1u << 16;
constexpr uint32_t kIdescBf16 = (1u << 7) | (1u << 10);

// Shared-memory descriptor of a K-major operand in the 128-byte-swizzle
// canonical layout: each row holds 64 fp16 (128 B) of the K dimension, rows
// are 128 B apart, 8-row groups 1024 B apart (the stride byte offset), and
// the 16-byte chunks of row r are stored XOR-permuted by (r % 8).  The tile
// base must be 1024-byte aligned; a K step of 16 elements inside the 128-byte
// row advances the start address by 32 B.
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                      // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
    return d;
}

// Shared-memory descriptor of an MN-major operand in the 128-byte-swizzle
// canonical layout: a 128-byte row holds 64 fp16 consecutive along M (or N)
// at one k, rows k .. k + 7 form one 1024-byte swizzle atom (16-byte chunk c
// of row k stored at chunk c ^ (k % 8)), 8-row groups along K are 1024 B
// apart (the stride byte offset) and the next 64 elements along M/N start
// mn_stride bytes further (the leading byte offset).  This is the layout a
// 128-byte-swizzled TMA box of 64-element rows lands in, read with the box
// rows as the K dimension.  The base must be 1024-byte aligned; a K step of
// 16 elements advances the start address by 2048 B.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t smem_addr, uint32_t mn_stride) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);     // start address
    d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;  // leading byte offset
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
    return d;
}

// Byte offset of element (r, k) in a K-major SW128 tile of `rows` rows.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t k, uint32_t rows) {
    const uint32_t kb = k >> 6, w = k & 63u;
    return kb * rows * 128u + (r >> 3) * 1024u + (r & 7u) * 128u + ((((w >> 3) ^ (r & 7u)) << 4)) +
           ((w & 7u) << 1);
}

// Byte offset of the 16-byte chunk c (8 fp16 along K, c in [0, K/8)) of row r.
__host__ __device__ __forceinline__ uint32_t sw128_chunk_offset(uint32_t r, uint32_t c, uint32_t rows) {
    const uint32_t kb = c >> 3, w = c & 7u;
    return kb * rows * 128u + (r >> 3) * 1024u + (r & 7u) * 128u + ((w ^ (r & 7u)) << 4);
}

// ---- TMEM <-> registers (32 lanes x 32 columns of 32 bits per warp) -------------

#define GDN_R32(r) "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), \
    "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),   \
    "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),            \
    "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),            \
    "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define GDN_W32(r) "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), \
    "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),         \
    "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),       \
    "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// Thread i of the warp receives columns [col, col + 32) of TMEM lane
// (warp's lane quarter base + i).  The load and its wait are one asm
// statement: tcgen05.ld writes its destination registers asynchronously until
// tcgen05.wait::ld, so the registers must not be visible to the compiler as
// defined (and free to copy out or reuse) before the wait has returned.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GDN_R32(r)
        : "r"(taddr)
        : "memory");
}
// The store and its wait are one asm statement, so the source registers stay
// reserved until the asynchronous read of them has completed.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        GDN_W32(r)
        : "memory");
}
// 16-column forms (thread i of the warp: columns [col, col + 16) of its lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

#undef GDN_R32
#undef GDN_W32

}  // namespace tc
}  // namespace gdn
