// zq_cluster.cuh -- inline-PTX wrappers for kernels that run as a pair of
// CTAs (a thread-block cluster of two) driving the tensor cores of both SMs
// with one MMA instruction (tcgen05 .cta_group::2): cluster rank and barrier,
// addresses in the peer CTA's shared memory, remote mbarrier arrivals, the
// pair's TMA loads, MMAs, commits and tensor-memory allocation, and register
// reallocation between warpgroups.  Every wait built on these is bounded by
// the global timer, like the single-CTA kernels'.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "zq_async.cuh"

namespace zq {

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs arrives; returns once all have (shared-memory
// writes before it are visible to the peer after it).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster's shared window, of the variable at local
// shared-memory address `local` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Arrive (release, cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr) : "memory");
}

// Asynchronous 4-byte store into a CTA of the cluster whose completion is
// counted (4 bytes) on an mbarrier of that CTA, with release semantics at
// cluster scope.  Measured in the pair GEMM: ~125 cycles of the issuing
// thread, against ~1200 for a release-arrive at cluster scope.
__device__ __forceinline__ void st_async_signal(uint32_t cl_dst, uint32_t cl_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cl_dst), "r"(0u),
                 "r"(cl_bar)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cl_addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cl_addr), "r"(v) : "memory");
}

// Phase test of a barrier whose arrivals may come from the peer CTA (its
// converter and epilogue warps' st.async bytes, its TMA bytes, the pair's MMA
// commits).  Default (CTA-scope acquire) semantics: the peer's signals are
// releases at cluster scope, and the data they publish is read by the tensor
// cores after tcgen05 fences, not by this thread.  (An acquire at cluster
// scope made each probe cost ~300 cycles.)
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t *bar, uint32_t parity)
{
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

__device__ __forceinline__ bool mbar_try_wait_cl_sleep(uint64_t *bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// 2-D tiled TMA load into this CTA's shared memory whose completion (bytes)
// is counted on `cl_bar`, an mbarrier of either CTA of the pair (cluster
// address).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, int x, int y, uint32_t cl_bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cl_bar)
        : "memory");
}

// ---- tensor memory and MMAs of a CTA pair --------------------------------
// Allocation and release are performed by one warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (M = 256 rows: 128 in each CTA's tensor memory) (+)= A * B^T, A's rows
// 0..127 from this CTA's shared memory and 128..255 from the peer's (same
// descriptor), B's rows likewise split in halves.  Issued by one thread of
// the even CTA.
__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same, with A in tensor memory: rows 0..127 from this CTA's tensor memory at
// column address a_tmem (K along the columns, two binary16 per column), rows
// 128..255 from the peer's at the same address.
__device__ __forceinline__ void mma_f16_pair_ta(uint32_t tmem_d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at local offset `bar` in every CTA of `cta_mask`
// once all MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Same, arriving on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---- register reallocation between warpgroups ----------------------------
// Executed by all threads of a warpgroup; the counts of all warpgroups must
// add up to no more than the registers the block was launched with.
template <uint32_t N>
__device__ __forceinline__ void regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

template <uint32_t N>
__device__ __forceinline__ void regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

}  // namespace zq
