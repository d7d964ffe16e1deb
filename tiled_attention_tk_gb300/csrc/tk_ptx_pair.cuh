// tk_ptx_pair.cuh -- PTX wrappers for kernels that run on pairs of CTAs
// (a cluster of two sharing each tcgen05 product, cta_group::2).  Kept apart
// from tk_ptx.cuh: only the GEMM's pair kernel uses them.
#pragma once

#include <cstdint>

namespace tk {

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
// Two CTAs of a cluster share each MMA: the leader (rank 0) issues it over
// both CTAs' shared-memory operands and TMEM.  Every tcgen05 instruction of
// such a kernel names cta_group::2.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of `addr` (a shared::cta address of this CTA's
// layout) in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One arrival on an mbarrier of any CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

// try_wait with cluster-scope acquire, for barriers that other CTAs arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// 3-D tiled load into this CTA's shared memory whose completion (transaction
// bytes) is signalled on `cbar`, an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void *tmap, uint32_t cbar, int c0, int c1,
                                                 int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(cbar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// TMEM allocation of a pair: one warp of each CTA executes each of these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Four pair MMAs (leader only), as umma_ss_x4.
__device__ __forceinline__ void umma_ss_x4_pair(uint32_t d_tmem, const uint32_t *a, uint32_t a_hi, const uint32_t *b,
                                                uint32_t b_hi, uint32_t idesc, uint32_t acc_first) {
    asm volatile(
        "{\n\t.reg .pred pt, pa;\n\t.reg .b64 ad0, ad1, ad2, ad3, bd0, bd1, bd2, bd3;\n\t"
        "setp.eq.u32 pt, 1, 1;\n\tsetp.ne.u32 pa, %12, 0;\n\t"
        "mov.b64 ad0, {%1, %9};\n\tmov.b64 bd0, {%5, %10};\n\t"
        "mov.b64 ad1, {%2, %9};\n\tmov.b64 bd1, {%6, %10};\n\t"
        "mov.b64 ad2, {%3, %9};\n\tmov.b64 bd2, {%7, %10};\n\t"
        "mov.b64 ad3, {%4, %9};\n\tmov.b64 bd3, {%8, %10};\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], ad0, bd0, %11, pa;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], ad1, bd1, %11, pt;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], ad2, bd2, %11, pt;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], ad3, bd3, %11, pt;\n\t}" ::"r"(d_tmem),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(a_hi),
        "r"(b_hi), "r"(idesc), "r"(acc_first)
        : "memory");
}

// Arrive once on `cbar` (an mbarrier of either CTA of the pair, shared::cluster
// address) when every pair MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t cbar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(cbar)
                 : "memory");
}

}  // namespace tk
