// Inline-PTX wrappers for sm_103a: mbarrier, cp.async (16 B, zero-fill),
// bulk async copy, tcgen05 (TMEM alloc, MMA, commit, load) and fences.
// Every wait is bounded: it gives up after kWaitNs of global time or when the
// block's abort flag is raised.
#pragma once
#include <cstdint>

namespace vg {
namespace ptx {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait until the phase with the given parity has completed.  Returns false if
// the block's abort flag is set or the time limit passes first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile uint32_t* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitNs) return false;
    }
}

// Time-bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool mbar_wait_timed(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitNs) return false;
    }
    return true;
}

// ---------------------------------------------------------------- copies
// 16-byte global->shared copy; src_bytes = 0 writes 16 zero bytes.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// Arrive on the mbarrier once all of this thread's earlier cp.async copies have
// landed (asynchronously; the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's completed generic-proxy shared-memory writes visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk (TMA engine) global->shared copy completing on an mbarrier transaction count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// 32-byte global store (p 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
// A warp stores one 128-byte line per lane: lane i holds its line as 32 words
// and its destination (null: nothing to store).  A 4 x 4
// transpose of 32-byte blocks inside each lane quad (two shuffle rounds) leaves
// lane 4g + d with block d of the lines of lanes 4g..4g+3, so each of the four
// stores writes eight whole lines -- eight requests per store instead of 32
// scattered 16-byte pieces when every lane writes its own line.  v8ok: the
// destinations are 32-byte aligned (one 32-byte store per block).
__device__ __forceinline__ void store_lines_quad(uint8_t* dst, uint32_t (&z)[32], int lane, bool v8ok) {
    const bool hi = (lane & 2) != 0, odd = (lane & 1) != 0;
    // round 1 (lanes d and d ^ 2): swap the off-diagonal 2 x 2 groups of blocks
#pragma unroll
    for (int sblk = 0; sblk < 2; ++sblk)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t send = hi ? z[8 * sblk + e] : z[8 * (2 + sblk) + e];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
            if (hi) z[8 * sblk + e] = recv;
            else z[8 * (2 + sblk) + e] = recv;
        }
    // round 2 (lanes d and d ^ 1): transpose each 2 x 2 group
#pragma unroll
    for (int t = 0; t < 4; t += 2)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t send = odd ? z[8 * t + e] : z[8 * (t + 1) + e];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
            if (odd) z[8 * t + e] = recv;
            else z[8 * (t + 1) + e] = recv;
        }
    const int d = lane & 3;
    const uint64_t mine = reinterpret_cast<uint64_t>(dst);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t pk = __shfl_sync(0xffffffffu, mine, (lane & ~3) | k);
        if (pk == 0) continue;  // the same for the four lanes of the quad
        uint8_t* p = reinterpret_cast<uint8_t*>(pk) + d * 32;
        if (v8ok) {
            st_global_v8(p, z + 8 * k);
        } else {
            uint4* d4 = reinterpret_cast<uint4*>(p);
            d4[0] = make_uint4(z[8 * k], z[8 * k + 1], z[8 * k + 2], z[8 * k + 3]);
            d4[1] = make_uint4(z[8 * k + 4], z[8 * k + 5], z[8 * k + 6], z[8 * k + 7]);
        }
    }
}

// Bring the 128-byte line holding p into L2 (no shared memory, no completion tracking).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, fp32 inputs read as TF32, fp32 accumulate (K = 8).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive (once) on the mbarrier when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout: rows of 128 B, 8-row groups 1024 B apart (stride byte offset), the
// tile 1024-byte aligned; start address advances by 32 B per K=16 step.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address, bits 0-13
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused here), bits 16-29
    d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset, bits 32-45
    d |= (uint64_t)1 << 46;                          // descriptor version, bits 46-47
    d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle, bits 61-63
    return d;
}

// Shared-memory matrix descriptor, MN-major operand in the 128-byte swizzle
// layout: each K row holds 64 consecutive M (or N) elements in 128 B, 8 K rows
// form a 1024-byte atom (stride byte offset between 8-row K groups = 1024),
// consecutive 64-element M/N blocks lie lbo bytes apart (leading byte offset);
// start address advances by 2048 B per K=16 step.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t lbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor for kind::f16 with both operands MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_mn(bool bf16, int n) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | (1u << 15) | (1u << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Instruction descriptor for kind::f16: D fp32, A/B fp16 (0) or bf16 (1), both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int n) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

// Instruction descriptor for kind::tf32: D fp32, A and B TF32 (format 2), both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_tf32(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

}  // namespace ptx
}  // namespace vg
