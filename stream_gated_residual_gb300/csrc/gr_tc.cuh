// tcgen05 wrappers (5th-generation tensor cores, sm_100-family): tensor-memory allocation, the
// shared-memory matrix descriptor, the instruction descriptor of kind::f16, the MMA, its commit to
// an mbarrier, and the tensor-memory loads and stores. Inline PTX, per the PTX ISA's tcgen05
// chapter; included after gr_ptx.cuh by the units that use tensor memory.
#pragma once

#include <stdint.h>

namespace gr {
namespace {

// ---- tensor memory (TMEM): 128 lanes × 512 columns of 32 bits per SM -------------------------
// Allocation by one whole warp; the column base is written to `slot` in shared memory. ncols is a
// power of two >= 32.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
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
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Writes of shared memory by threads, made visible to the tensor cores (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- descriptors --------------------------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzled layout that a TMA
// load with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128 bytes (64 bf16 of K), groups of 8 rows
// (1024 bytes, the swizzle atom) one after another. Start address (>> 4) in bits 0-13, leading
// byte offset (>> 4, unused for this layout) in 16-29, stride byte offset (>> 4: 1024 between
// 8-row groups) in 32-45, descriptor version 1 in 46-47, base offset 0 (atoms 1024-byte aligned)
// in 49-51, layout type 2 (128-byte swizzle) in 61-63. A K step of 16 elements inside the
// 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t(1u) << 16;                   // leading byte offset (ignored here)
    d |= uint64_t((1024u >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1u) << 46;
    d |= uint64_t(2u) << 61;
    return d;
}
// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits 7-9
// and 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
           (uint32_t(M >> 4) << 24);
}

// ---- MMA ----------------------------------------------------------------------------------------
// D[tmem] (+)= A[smem] · B[smem]ᵀ, issued by one thread; accumulate = 0 overwrites D.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] · B[smem]ᵀ: A's row m in lane m, two 16-bit elements of consecutive k in
// each 32-bit column (the lower k in the low half), so one K = 16 step reads 8 columns.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---- epilogue loads: a warp reads 32 lanes (its quadrant: warp % 4) × 16 columns -------------
// Without the wait: several loads may be in flight; tmem_wait_ld() before using any of them.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// Waits for this thread's tensor-memory loads; `r` (one load's destination) passes through the
// wait as in/out operands, so the compiler cannot move a use of it ahead of the wait. Call it
// once per destination array (the waits after the first return at once).
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}
// A warp writes 32 lanes (its quadrant) × 16 columns: thread l's r[k] to lane (taddr's lane
// + l), column (taddr's column + k). tmem_wait_st() before anything relies on the values.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16_nowait(taddr, r);
    tmem_wait_ld(r);
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
}

// ---- a bounded wait that never suspends ---------------------------------------------------------
// For producers that share a warp (lanes with waits of their own): a suspending try_wait would
// stop the whole warp. Spins on test_wait; records bit 0 of the status word if it runs out.
__device__ __forceinline__ bool spin_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n"
            " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitLimit) {
            atomicOr(&g_wait_status, 1u);
            return false;
        }
    }
}

// ---- TMA store of a 3-D box (the large-rank path's R' tiles) ---------------------------------
// From shared memory to the tensor (clipped to its extent), as one bulk group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
        : "memory");
}

}  // namespace
}  // namespace gr
