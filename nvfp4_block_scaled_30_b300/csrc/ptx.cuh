// Inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk[.tensor]),
// tcgen05 (TMEM alloc, MMA, copy, load, commit, fences) and the FP8/FP4
// conversions.  Every wait here is bounded by a deadline on %globaltimer.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "bounds.cuh"

namespace nv4 {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id()
{
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

// ---- mbarrier ----------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
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

// Waits for the phase with the given parity to complete.  Returns false when
// timeout_ns (measured on %globaltimer) passes or *abort (if not null)
// becomes non-zero first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t deadline = globaltimer_ns() + timeout_ns;
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((spin & 63u) == 63u) {
            if (abort != nullptr && *abort)
                return false;
            if (globaltimer_ns() > deadline)
                return false;
        }
    }
}

// 16-byte asynchronous copy global -> shared; bytes beyond src_bytes (0..16)
// are filled with zeros.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, uint32_t src_bytes)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), 16) && aligned_to(NV4_SITE(1), smem_u32(dst), 16) &&
          in_bounds(NV4_SITE(1), src_bytes, 17)))
        return;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

// L2 eviction-priority policies for the cache-hint forms below: data read
// once (a weight stream) and data read again soon (gathered activations).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// cp_async_16 with an L2 cache policy.
__device__ __forceinline__ void cp_async_16_hint(void *dst, const void *src, uint32_t src_bytes, uint64_t policy)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), 16) && aligned_to(NV4_SITE(1), smem_u32(dst), 16) &&
          in_bounds(NV4_SITE(1), src_bytes, 17)))
        return;
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes), "l"(policy)
                 : "memory");
}

// 4-byte cp.async (src_bytes 0 or 4; 0 zero-fills the destination).
__device__ __forceinline__ void cp_async_4(void *dst, const void *src, uint32_t src_bytes)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), 4) && aligned_to(NV4_SITE(1), smem_u32(dst), 4) &&
          in_bounds(NV4_SITE(1), src_bytes, 5)))
        return;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Arrive on *bar (without raising its expected count) once every cp.async
// this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- TMA / bulk copies ----------------------------------------------------------

// 2-D tiled copy of the box at (x, y) of a byte-element tensor map; box_bytes
// is the box's size in shared memory (checked in the bounds-checked build,
// with x a multiple of 16 and dst 128-byte aligned).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar, uint32_t box_bytes)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), box_bytes) && aligned_to(NV4_SITE(1), smem_u32(dst), 128) &&
          aligned_to(NV4_SITE(1), (uint32_t)x, 16)))
        return;
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 4-D tiled TMA load (coordinates innermost first); x must be a multiple of
// 16 bytes.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint64_t *bar, uint32_t box_bytes)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), box_bytes) && aligned_to(NV4_SITE(1), smem_u32(dst), 128) &&
          aligned_to(NV4_SITE(1), (uint32_t)x, 16)))
        return;
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 uint64_t *bar, uint32_t box_bytes, uint64_t policy)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), box_bytes) && aligned_to(NV4_SITE(1), smem_u32(dst), 128) &&
          aligned_to(NV4_SITE(1), (uint32_t)x, 16)))
        return;
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch.  pdl_wait blocks until the grids this one
// depends on have completed and their memory is visible (no-op when the
// launch carried no programmatic dependency); pdl_trigger lets the next
// grid in the stream start launching.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block cluster: this CTA's rank, a full cluster barrier (every
// thread of every CTA; release/acquire on shared::cluster), and a 32-bit
// load from the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_dsmem_u32(void *local, uint32_t rank, uint32_t v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// Split cluster barrier: arrive without ordering (e.g. "this CTA is
// running") and, later, wait for every CTA's arrival.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(const void *local, uint32_t rank)
{
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// Fetch a tensor map (kernel parameter) into the descriptor cache.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 prefetch of one tile of a 2-D tensor map (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int32_t x, int32_t y)
{
    if (!aligned_to(NV4_SITE(1), (uint32_t)x, 16))
        return;
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// L2 prefetch of a contiguous range; address 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    if (!(aligned_to(NV4_SITE(1), reinterpret_cast<uint64_t>(src), 16) && aligned_to(NV4_SITE(1), bytes, 16)))
        return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    if (!(in_dyn_smem(NV4_SITE(1), smem_u32(dst), bytes) && aligned_to(NV4_SITE(1), smem_u32(dst), 16) &&
          aligned_to(NV4_SITE(1), reinterpret_cast<uint64_t>(src), 16) && aligned_to(NV4_SITE(1), bytes, 16)))
        return;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 ----------------------------------------------------------------------

// Whole warp.  Writes the TMEM base address to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Bounds-checked build: the TMEM columns [col, col + n) of taddr lie within
// the 512 columns, and the operand tiles that the descriptors address (128
// rows of A, N rows of B, 128 bytes each, from the 1024-byte aligned tile
// base) lie in dynamic shared memory.
__device__ __forceinline__ bool tmem_cols_ok(uint32_t site, uint32_t taddr, uint32_t n)
{
    return in_bounds(site, (taddr & 0xFFFFu) + n - 1, 512) && in_bounds(site, taddr >> 16, 128);
}

__device__ __forceinline__ bool mma_operands_ok(uint32_t site, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc)
{
    if (!kCheckBounds)
        return true;
    const uint32_t n = ((idesc >> 17) & 0x3Fu) << 3;
    const uint32_t a0 = ((uint32_t)(adesc & 0x3FFFu) << 4) & ~1023u;
    const uint32_t b0 = ((uint32_t)(bdesc & 0x3FFFu) << 4) & ~1023u;
    return tmem_cols_ok(site, d_tmem, n) && in_dyn_smem(site, a0, 128 * 128) && in_dyn_smem(site, b0, n * 128);
}

// Single thread: D(tmem) (+)= A(smem) x B(smem)^T, block-scaled E2M1 x E2M1
// with UE4M3 scales per 16 elements of K (K = 64 per instruction).
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    if (!(mma_operands_ok(NV4_SITE(1), d_tmem, adesc, bdesc, idesc) && tmem_cols_ok(NV4_SITE(1), sfa_tmem, 1) &&
          tmem_cols_ok(NV4_SITE(1), sfb_tmem, 1)))
        return;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Single thread: D(tmem) (+)= A(smem) x B(smem)^T, kind::f16 (FP16 or BF16
// operands of the same type, as the instruction descriptor says), K = 16.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    if (!mma_operands_ok(NV4_SITE(1), d_tmem, adesc, bdesc, idesc))
        return;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Single thread: D(tmem) (+)= A(tmem) x B(smem)^T, kind::f16 with the A
// operand in TMEM (M = 128 rows in lanes 0..127, each 32-bit column holding
// two consecutive K elements, K = 16 per instruction: 8 columns from a_tmem).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    if (kCheckBounds) {
        const uint32_t n = ((idesc >> 17) & 0x3Fu) << 3;
        const uint32_t b0 = ((uint32_t)(bdesc & 0x3FFFu) << 4) & ~1023u;
        if (!(tmem_cols_ok(NV4_SITE(1), d_tmem, n) && tmem_cols_ok(NV4_SITE(1), a_tmem, 8) &&
              aligned_to(NV4_SITE(1), a_tmem & 0xFFFFu, 8) && in_dyn_smem(NV4_SITE(1), b0, n * 128)))
            return;
    }
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Whole warp: 16 consecutive 32-bit columns into this warp's 32 TMEM lanes
// (one row of 16 words per lane); taddr's column a multiple of 16.
__device__ __forceinline__ void tc_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16])
{
    if (!(tmem_cols_ok(NV4_SITE(1), taddr, 16) && aligned_to(NV4_SITE(1), taddr & 0xFFFFu, 16)))
        return; // taddr is the same in every lane
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15, %16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

// Whole warp: every tcgen05.st of this thread has completed.
__device__ __forceinline__ void tc_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Single thread: copy 32 rows x 16 bytes from shared memory into TMEM lanes
// 0..31 of 4 consecutive columns, replicated into all four lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc)
{
    if (!(tmem_cols_ok(NV4_SITE(1), taddr, 4) &&
          in_dyn_smem(NV4_SITE(1), (uint32_t)(sdesc & 0x3FFFu) << 4, 512)))
        return;
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Single thread: arrive once on *bar when all earlier tcgen05 operations of
// this thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Whole warp: 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    if (!tmem_cols_ok(NV4_SITE(1), taddr, 32)) { // taddr is the same in every lane
        for (int c = 0; c < 32; ++c)
            r[c] = 0u;
        return;
    }
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Whole warp: 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    if (!tmem_cols_ok(NV4_SITE(1), taddr, 16)) {
        for (int c = 0; c < 16; ++c)
            r[c] = 0u;
        return;
    }
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format).  K-major operand tile with
// 128-byte rows and the 128-byte swizzle: 8-row atoms of 1024 bytes, stride
// (SBO) 1024 between atoms; the tile must start 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);           // start address
    d |= (uint64_t)(16u >> 4) << 16;                     // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;                   // stride byte offset
    d |= (uint64_t)1u << 46;                             // descriptor version for sm_100+
    d |= (uint64_t)2u << 61;                             // 128-byte swizzle
    return d;
}

// Descriptor of 32 rows x 16 bytes stored contiguously (no swizzle): 8-row
// core matrices of 128 bytes, 128 bytes apart.  Source of tcgen05.cp 32x128b.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// Instruction descriptor: kind::mxf4nvf4, A and B E2M1, K-major, UE4M3 scales,
// scale-factor ids 0, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(uint32_t n)
{
    return (1u << 7)              // A format E2M1
           | (1u << 10)           // B format E2M1
           | ((n >> 3) << 17)     // N / 8
           | (0u << 23)           // scale format UE4M3
           | ((128u >> 4) << 24); // M / 16
}

// Instruction descriptor: kind::f16, FP16 x FP16 -> FP32, K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t n)
{
    return (1u << 4)              // D format FP32
           | (0u << 7)            // A format FP16
           | (0u << 10)           // B format FP16
           | ((n >> 3) << 17)
           | ((128u >> 4) << 24);
}

// ---- conversions ----------------------------------------------------------------------

// E2M1 codes of (lo, hi) packed in one byte: lo in bits 0..3, hi in bits 4..7.
// cvt.rn.satfinite rounds to nearest even and saturates at +-6; measured on
// B300 over every non-NaN binary32 input, in both operand positions, it
// keeps the sign of results that round to zero (code 0x8), as the format
// reading requires, so no sign fix-up follows it.  The exhaustive GPU test of
// the conversions against the oracle checks this on every run.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t b;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(b)
        : "f"(hi), "f"(lo));
    return b;
}

// Eight values' E2M1 codes packed into one word: byte i holds the codes of
// q[2i] (low nibble) and q[2i+1] (high nibble), each byte as e2m1x2 forms it;
// the four bytes are joined by one vector move instead of per-byte widening,
// shifts and ORs.
__device__ __forceinline__ uint32_t e2m1x8(float q0, float q1, float q2, float q3, float q4, float q5, float q6,
                                           float q7)
{
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
    return w;
}

// E4M3 code of v (round to nearest even, saturating at +-448).
__device__ __forceinline__ uint32_t e4m3(float v)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
    return h & 0xFFu;
}

// Exact value of a non-negative E4M3 code 0x00..0x7E.
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    uint32_t ex = (c >> 3) & 15u, m = c & 7u;
    if (ex == 0u)
        return __uint_as_float(0x3B000000u) * (float)m; // m * 2^-9 (exact)
    return __uint_as_float(((ex + 120u) << 23) | (m << 20));
}

// NVFP4 block encode arithmetic shared by the quantisers and the GEMM
// epilogue that quantises its output (binary32, explicit round-to-nearest):
// the E4M3 scale code of a block whose absolute maximum is amax_b under the
// second-level scale s, and the reciprocal of a dequantisation step (0 for
// 0, at most the largest float).
__device__ __forceinline__ uint32_t block_scale_code(float amax_b, float s)
{
    if (s == 0.0f)
        return 0u;
    const float t = __fdiv_rn(amax_b, 6.0f);
    const float u = __fdiv_rn(t, s);
    return e4m3(u);
}

__device__ __forceinline__ float recip_step(float d)
{
    return d == 0.0f ? 0.0f : fminf(__frcp_rn(d), 3.402823466e+38f);
}

// Two IEEE round-to-nearest products at once (bit-identical to two
// __fmul_rn).
__device__ __forceinline__ void mul2_rn(float a0, float a1, float r, float &p0, float &p1)
{
    uint64_t a = (uint64_t)__float_as_uint(a0) | ((uint64_t)__float_as_uint(a1) << 32);
    const uint64_t rr = (uint64_t)__float_as_uint(r) | ((uint64_t)__float_as_uint(r) << 32);
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(rr));
    p0 = __uint_as_float((uint32_t)d);
    p1 = __uint_as_float((uint32_t)(d >> 32));
}

// One 16-element block of BF16 values (8 words, element 2i in the low half
// of word i) encoded under the tensor scale s by the quantisers' rule: the
// block maximum from the magnitude bits (exact, equal to the float maximum
// of finite values), the E4M3 scale code, the reciprocal step, and the 16
// E2M1 codes packed into two words (element 2j in the low nibble of byte j).
// Returns the scale code.
__device__ __forceinline__ uint32_t encode_bf16_block(const uint32_t (&w)[8], float s, uint32_t (&pk)[2])
{
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m2 = __vmaxu2(m2, w[i] & 0x7FFF7FFFu);
    const float amb = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
    const uint32_t e = block_scale_code(amb, s);
    const float r = recip_step(__fmul_rn(e4m3_value(e), s));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float q[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t ww = w[4 * h + i];
            mul2_rn(__uint_as_float(ww << 16), __uint_as_float(ww & 0xFFFF0000u), r, q[2 * i], q[2 * i + 1]);
        }
        pk[h] = e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
    }
    return e;
}

} // namespace nv4

