// fw_tc.cuh -- inline-PTX building blocks for the sm_103a tensor-core path:
// mbarriers, 1-D bulk (TMA) copies, tensor memory (TMEM) allocation and
// access, tcgen05.mma with shared-memory matrix descriptors, and the
// 128-byte-swizzled operand layouts those descriptors describe.
//
// Conventions used throughout:
//  * Operands are bf16, accumulators fp32 in TMEM, MMA shape M = 128
//    (cta_group::1): accumulator row m lives in TMEM lane m, column n in
//    TMEM column (base + n).  Warp w of a CTA may only touch lanes
//    [32 (w % 4), 32 (w % 4) + 32).
//  * "K-major, SW128" tile of R rows x K columns: K is split into 64-element
//    (128-byte) blocks; block kb starts at kb * R * 128 bytes; row r of a
//    block is 128 bytes at r * 128; the 16-byte chunk c of row r is stored at
//    chunk c ^ (r % 8).  Descriptor: start address of the 16-element K step,
//    stride byte offset (8-row group) 1024.  Every block starts 1024-aligned.
//  * "MN-major, SW128" view of the same bytes: for an operand whose
//    contraction index is the tile's row r and whose M/N index is the tile's
//    column, 64-column blocks are LBO bytes apart and 8-row groups SBO apart.
//  * Every wait is bounded: after about kWaitLimitNs the caller gets `false`
//    and the device status word records kStatusTimeout.
#pragma once

#include "fw_common.cuh"

namespace fw {
namespace tc {

constexpr uint64_t kWaitLimitNs = 1000000000ull; // a bounded wait gives up after ~1 s

FW_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ------------------------------------------------------------- mbarriers
FW_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

FW_DEV void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

FW_DEV bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(addr), "r"(parity)
                 : "memory");
    return ok != 0;
}

FW_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; false once limit_ns
// has passed (the device status word then records kStatusTimeout).
// try_wait itself suspends the thread for a while in hardware, so the loop
// only re-polls; the elapsed time is checked every 64 polls.
FW_DEV bool mbar_wait_ns(uint64_t *bar, uint32_t parity, unsigned *status, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity))
            return true;
        if ((i & 63) == 0 && globaltimer_ns() - t0 > limit_ns)
            break;
    }
    record_status(status, kStatusTimeout);
    return false;
}

FW_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *status) {
    return mbar_wait_ns(bar, parity, status, kWaitLimitNs);
}

// A plain arrival (release: this thread's earlier shared-memory accesses are
// ordered before it).
FW_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

FW_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// ------------------------------------------------------------ ready flags
// A flag in global memory that one CTA sets once what it guards is complete
// and another CTA of the same (cooperative) launch waits for.  The writer
// orders every write it guards (bulk copies included) before a release
// store; the reader's acquire load orders every later read, bulk copies
// included, after it.
// The writer has waited for its bulk copies to complete (their writes are
// then visible to it); the proxy fence orders those async-proxy writes
// before its later generic accesses, and the release store orders every
// earlier access of the thread before the flag.
FW_DEV void flag_set(unsigned *f) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(1u) : "memory");
}
FW_DEV unsigned flag_load(const unsigned *f) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
// Bounded wait for a flag: false after limit_ns, with kStatusTimeout
// recorded; on success later bulk copies observe what the writer released.
FW_DEV bool flag_wait_ns(const unsigned *f, unsigned *status, uint64_t limit_ns) {
    bool ok = flag_load(f) != 0;
    if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 1;; ++i) {
            __nanosleep(100);
            if (flag_load(f) != 0) {
                ok = true;
                break;
            }
            if ((i & 31) == 0 && globaltimer_ns() - t0 > limit_ns)
                break;
        }
    }
    if (!ok) {
        record_status(status, kStatusTimeout);
        return false;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}
FW_DEV bool flag_wait(const unsigned *f, unsigned *status) { return flag_wait_ns(f, status, kWaitLimitNs); }

// ------------------------------------------------ 1-D bulk copy (TMA engine)
// global -> shared, completion counted on `bar` in bytes.  dst, src and
// bytes must be multiples of 16.
FW_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 2-D TMA tensor copy of one box into shared memory, completion counted on
// `bar` in bytes.  x is the inner (contiguous) coordinate; x times the
// element size must be a multiple of 16 bytes.  `map` is a CUtensorMap
// (kernel parameter or global memory).
FW_DEV void tma_load_2d(void *dst, const void *map, int x, int y, uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
                 : "memory");
}

// shared -> global, tracked by this thread's bulk-async group.  dst, src and
// bytes must be multiples of 16.
FW_DEV void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
FW_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has finished reading
// its shared-memory source (the source may then be overwritten or released).
FW_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store of this thread has fully completed.
FW_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor core, bulk copies) once followed by a CTA barrier.
FW_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// (programmatic dependent launch: griddep_wait / griddep_launch_dependents
// and launch_pdl live in fw_common.cuh)

// ------------------------------------------------------------------- TMEM
FW_DEV void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) { // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
FW_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
FW_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) { // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
FW_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FW_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 bit, 16 consecutive columns: this thread gets lane
// (taddr.lane + laneid), columns taddr.col .. +15, into r[0..15].
FW_DEV void tmem_ld16(uint32_t taddr, float *r) {
    uint32_t u[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
                   "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
                   "=r"(u[14]), "=r"(u[15])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i)
        r[i] = __uint_as_float(u[i]);
}
FW_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Store r[0..15] to lane (taddr.lane + laneid), columns taddr.col .. +15.
FW_DEV void tmem_st16(uint32_t taddr, const float *r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])), "r"(__float_as_uint(r[2])),
                 "r"(__float_as_uint(r[3])), "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])),
                 "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])), "r"(__float_as_uint(r[8])),
                 "r"(__float_as_uint(r[9])), "r"(__float_as_uint(r[10])), "r"(__float_as_uint(r[11])),
                 "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])), "r"(__float_as_uint(r[14])),
                 "r"(__float_as_uint(r[15]))
                 : "memory");
}
FW_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Lane base of warp w's TMEM sub-partition, in the address's lane field.
FW_DEV uint32_t tmem_lane_base(int warp) { return (uint32_t)(32 * (warp & 3)) << 16; }

// -------------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, 128-byte swizzle.
FW_DEV uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46; // descriptor version for tcgen05
    d |= (uint64_t)2 << 61; // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator.
// a_mn / b_mn select MN-major (1) or K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T, issued by one thread.
FW_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
FW_DEV void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- layouts
// Byte offset of element (r, k) in a K-major SW128 tile of R rows.
FW_DEV uint32_t kmajor_off(int r, int k, int R) {
    return (uint32_t)((k >> 6) * R * 128 + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}
// Byte offset of the 16-byte chunk holding elements k .. k+7 (k % 8 == 0).
FW_DEV uint32_t kmajor_chunk(int r, int k, int R) {
    return (uint32_t)((k >> 6) * R * 128 + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4));
}
// Descriptor start offset of the 16-element K step s of a K-major SW128 tile.
FW_DEV uint32_t kmajor_step(int s, int R) { return (uint32_t)((s >> 2) * R * 128 + (s & 3) * 32); }

} // namespace tc
} // namespace fw
