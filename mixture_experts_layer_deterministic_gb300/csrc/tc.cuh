// tc.cuh -- inline-PTX building blocks for sm_103a: mbarriers, TMA tile loads, tcgen05
// (TMEM allocation, MMA, commit, TMEM loads) and the shared-memory / instruction
// descriptors the MMA reads. Written from the PTX ISA's descriptions of these instructions.
//
// Every wait is bounded: a wait that has not completed after WAIT_LIMIT_NS of wall time
// records MOK_ERR_TIMEOUT in the device status word and reports failure to its caller,
// which then stops issuing work, so a kernel can never spin forever.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mok {
namespace tc {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

MOK_DEV uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

MOK_DEV uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

MOK_DEV bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// ---------------------------------------------------------------- mbarrier
MOK_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
MOK_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOK_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
MOK_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
MOK_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait on phase `parity` of `bar`; gives up when another role has raised `abort`,
// or after limit_ns of wall time, when it records MOK_ERR_TIMEOUT in the status word and
// raises `abort` itself
MOK_DEV bool wait_bounded(uint64_t *bar, uint32_t parity, int *status, volatile int *abort,
                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++n & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                raise_status(status, MOK_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

// bounded spin until the global counter *ctr reaches `target` (an acquire load, so what its
// writers stored before raising it is visible after); gives up when another role has raised
// `abort`, or when the status word already holds a problem (another CTA gave up: raises
// `abort`), or after limit_ns of wall time (records MOK_ERR_TIMEOUT, raises `abort`)
MOK_DEV bool wait_count_bounded(const int32_t *ctr, int32_t target, int *status,
                                volatile int *abort, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 0;; ++n) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((n & 31u) == 31u) {
            if (*abort) return false;
            if (*(volatile int *)status != MOK_OK) {
                *abort = 1;
                return false;
            }
            if (globaltimer() - t0 > limit_ns) {
                raise_status(status, MOK_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
        __nanosleep(64);
    }
}

// ---------------------------------------------------------------- TMA
MOK_DEV void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)m) : "memory");
}
// 2D tile load into shared memory, completion counted on `bar` (transaction bytes)
MOK_DEV void tma_load_2d(void *smem_dst, const CUtensorMap *m, uint64_t *bar, int32_t x,
                         int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
// 5D tile load (coordinates innermost first), completion counted on `bar`
MOK_DEV void tma_load_5d(void *smem_dst, const CUtensorMap *m, uint64_t *bar, int32_t c0,
                         int32_t c1, int32_t c2, int32_t c3, int32_t c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

// orders this thread's global accesses of the generic proxy (plain loads and stores) with
// those of the async proxy (TMA copies), in both directions
MOK_DEV void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// 1D bulk copy global -> shared (16-byte aligned, size a multiple of 16), counted on `bar`
MOK_DEV void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"((uint64_t)gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 1D bulk copy shared -> global (16-byte aligned, size a multiple of 16) in this thread's
// current bulk group; commit_group closes the group, wait_group_read<N> waits until the
// shared-memory sources of all but the N most recent groups have been read, wait_group<N>
// until their writes are complete
MOK_DEV void bulk_store(void *gdst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     (uint64_t)gdst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}
MOK_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
MOK_DEV void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
MOK_DEV void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- Cluster Launch Control
// Ask the hardware to cancel the launch of a CTA (a cluster of one) that has not started;
// a 16-byte response lands in shared memory and completes 16 transaction bytes on `bar`.
MOK_DEV void clc_try_cancel(void *resp16, uint64_t *bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
        " [%0], [%1];" ::"r"(smem_u32(resp16)),
        "r"(smem_u32(bar))
        : "memory");
}
// Decode a response: true and the cancelled CTA's x index if a launch was cancelled, false
// when no CTA was left to cancel.
MOK_DEV bool clc_query(const void *resp16, uint32_t *ctaid_x) {
    uint32_t ok, x = 0;
    asm volatile(
        "{\n.reg .pred p;\n.reg .b128 r;\nld.shared.b128 r, [%2];\n"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid.v4.b32.b128 {%1, _, _, _}, r;\n"
        "}\n"
        : "=r"(ok), "+r"(x)
        : "r"(smem_u32(resp16))
        : "memory");
    *ctaid_x = x;
    return ok != 0;
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation by one full warp; the base address is written to shared memory.
MOK_DEV void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
MOK_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOK_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}
MOK_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOK_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit inputs, fp32 accumulation; one thread issues.
MOK_DEV void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                     uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= (A * scale_A)[smem] * (B * scale_B)[smem]^T for E4M3 operands with one E8M0
// scale per 32 K-elements taken from TMEM (kind::mxf8f6f4, K = 32 per instruction).
MOK_DEV void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copies a 32-row x 16-byte block of shared memory into TMEM: row i goes to lane i of each
// of the four 32-lane quadrants, 4 consecutive 32-bit columns.
MOK_DEV void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread is done.
MOK_DEV void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane (base + i).
MOK_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
MOK_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- pairs of SMs
// A cluster of two CTAs on two SMs shares one MMA (cta_group::2): the CTA of rank 0 issues
// it, each CTA supplies half of each operand from its own shared memory and receives its
// half of the accumulator in its own TMEM. Every tcgen05 instruction of such a kernel
// names cta_group::2; allocation, relinquish and deallocation are issued by one warp of
// each CTA of the pair.
MOK_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
MOK_DEV uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
MOK_DEV uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// the shared::cluster address of this CTA's shared variable `p` in the CTA of rank `rank`
MOK_DEV uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// arrive on an mbarrier given by its shared::cluster address (this CTA's or another's)
MOK_DEV void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     bar_cluster)
                 : "memory");
}
MOK_DEV bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], "
        "%2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// wait_bounded for a barrier that other CTAs of the cluster arrive on
MOK_DEV bool wait_bounded_cluster(uint64_t *bar, uint32_t parity, int *status,
                                  volatile int *abort, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (!mbar_try_wait_cluster(bar, parity)) {
        if ((++n & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                raise_status(status, MOK_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}
// every thread of both CTAs (non-aligned forms: threads may arrive from diverged paths)
MOK_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}
// 2D tile load into this CTA's shared memory whose transaction bytes complete on an
// mbarrier of either CTA of the pair (its shared::cluster address)
MOK_DEV void tma_load_2d_pair(void *smem_dst, const CUtensorMap *m, uint32_t bar_cluster,
                              int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}
// 5D tile load (coordinates innermost first), likewise completing on either CTA's mbarrier
MOK_DEV void tma_load_5d_pair(void *smem_dst, const CUtensorMap *m, uint32_t bar_cluster,
                              int32_t c0, int32_t c1, int32_t c2, int32_t c3, int32_t c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}
MOK_DEV void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
MOK_DEV void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOK_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}
// D (+)= A B^T over the pair: M = 256 (rows 0-127 from rank 0's A, 128-255 from rank 1's),
// N columns (the first N/2 from rank 0's B, the rest from rank 1's); each CTA's TMEM gets
// its 128 rows x N. Issued by one thread of rank 0; descriptors name this CTA's tiles, the
// peer's sit at the same shared-memory offsets.
MOK_DEV void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                          uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on the mbarrier at `bar`'s offset in each CTA of `cta_mask` when every
// tcgen05 operation issued so far by this thread is done
MOK_DEV void mma_commit_pair(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose 8-row groups
// of 128-byte rows are `sbo` bytes apart (1024 for densely stacked rows) and whose
// 64-element column blocks along the other dimension are `lbo` bytes apart (MN-major
// operands only). Fields: start address >> 4 (bits 0-13), leading byte offset >> 4
// (16-29), stride byte offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0
// (49-51), swizzle mode 2 = 128-byte swizzle (61-63). The tile must be 1024-byte aligned.
MOK_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Shared-memory descriptor of a non-swizzled block of 8-row x 16-byte core matrices
// stacked along the rows every 128 bytes (the source of tcgen05.cp 32x128b).
MOK_DEV uint64_t sdesc_plain_rows16(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 A and B (format 0),
// fp32 D (bit 4), K-major operands, B scale-factor id (bits 4-5), N >> 3 (17-22), scale
// type UE8M0 (bit 23), M >> 4 (24-28), A scale-factor id (29-30). The ids select the byte
// of the 32-bit TMEM scale word that holds this instruction's 32-element block.
MOK_DEV uint32_t idesc_mxf8(int M, int N, uint32_t sf_id) {
    uint32_t d = 0;
    d |= (sf_id & 3u) << 4;
    d |= (uint32_t)(N >> 3) << 17;
    d |= 1u << 23;
    d |= (uint32_t)(M >> 4) << 24;
    d |= (sf_id & 3u) << 29;
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, M x N:
// D format f32 (bits 4-5 = 1), A type bf16 (7-9 = 1), B type bf16 (10-12 = 1),
// A major (15: 0 K-major, 1 MN-major), B major (16), N >> 3 (17-22), M >> 4 (24-28).
MOK_DEV uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    uint32_t d = 0;
    d |= 1u << 4;
    d |= 1u << 7;
    d |= 1u << 10;
    d |= (a_mn_major ? 1u : 0u) << 15;
    d |= (b_mn_major ? 1u : 0u) << 16;
    d |= (uint32_t)(N >> 3) << 17;
    d |= (uint32_t)(M >> 4) << 24;
    return d;
}

}  // namespace tc
}  // namespace mok
