// Device helpers for sm_103a: mbarriers, TMA bulk copies, tcgen05 (TMEM allocation,
// block-scaled MMA, scale-factor copies, TMEM loads), NVFP4 element conversions.
// Everything here is inline PTX written from the PTX ISA's descriptions of these
// instructions; no library code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4moe.h"

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kRowAlign = 128;        // padded groups start on multiples of this
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded pipeline waits: 2 s

// ------------------------------------------------------------------ small utilities

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits)
{
    if (status) atomicOr(status, bits);
}

// Adds v to *p with release semantics at GPU scope: writes this thread has made, or has
// observed (through a block barrier it passed), are visible to a thread that sees the sum.
__device__ __forceinline__ void red_release_gpu(int32_t* p, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A 32-bit load with acquire semantics at GPU scope: reads that follow it in this thread see
// the writes released (a fence, then an atomic) by the thread whose value it observed.
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Programmatic dependent launch.  The forward's kernels are launched so that each may start
// while its predecessor finishes.  pdl_wait() blocks the calling thread until the preceding
// kernel has completed and its writes are visible (a no-op without the launch attribute);
// pdl_trigger() lets the next kernel be scheduled.  Every kernel calls pdl_wait() before
// pdl_trigger(), so when a kernel starts, all kernels before its predecessor are complete:
// it may read their outputs (and constant data) before its own pdl_wait().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
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

// As mbar_try_wait, but the thread may stay suspended up to kSuspendHintNs while the phase
// is incomplete (it resumes as soon as the phase completes), so a waiting warp takes no
// issue slots from the warps doing the work.
constexpr uint32_t kSuspendHintNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if the wait ran
// longer than limit_ns or if *abort became nonzero (another warp gave up).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// mbar_wait for a waiter off the critical path (a producer far ahead, an epilogue waiting
// for a whole tile): between polls the thread sleeps sleep_ns, leaving the issue slots to
// the warps doing the work.
__device__ __forceinline__ bool mbar_wait_lazy(uint64_t* bar, uint32_t parity,
                                               volatile int* abort, uint32_t sleep_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// As mbar_wait, with cluster-scope acquire: for a barrier that threads of the peer CTA of a
// cluster arrive on (their writes before the arrival become visible to the waiter).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// ------------------------------------------------------------------ CTA pairs (clusters of 2)

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs of the cluster arrives and waits (release / acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on the mbarrier at the same shared-memory offset in CTA `rank` of the cluster.  The
// callers' data is complete before they arrive (TMA transfers their barrier has counted, TMEM
// stores waited for with tcgen05.wait::st), so the arrive carries only the default release:
// a cluster-scope release would wait for every outstanding memory operation of the thread
// and put a cross-SM round trip into every pipeline stage.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank)
{
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
        "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar)),
        "r"(rank)
        : "memory");
}

// TMEM allocation for a CTA pair: one warp of each CTA executes it; both CTAs receive the
// same columns.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem of both CTAs] (+)= A[smem, M = 256: 128 rows in each CTA] . B[smem, N rows: N / 2 in
// each CTA]^T, block-scaled NVFP4 (K = 64); the scale factors at the same TMEM addresses in
// both CTAs (each CTA: its own A rows' scales, and all N B rows' scales).  Leader CTA only.
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d_taddr, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t sfa_taddr,
                                                 uint32_t sfb_taddr, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X "
        "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_taddr),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_taddr), "r"(sfb_taddr), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at bar's offset in every CTA of cta_mask when the pair MMAs
// issued so far by this thread are done.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------------------------------ TMA / bulk copies

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled tensor load into shared memory, completion counted on bar (bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// 2-D tiled tensor store shared -> global (bulk-group completion).
// The tensor stores are the down GEMMs' y rows: stored with the L2 evict-first policy, so that
// a large y (a prefill chunk's 0.6 GB) is written back while the GEMM runs rather than under
// the combine's reads (prefill forward 1.357 -> 1.344 ms; decode and the expert shard, whose
// y stays in L2 either way, unchanged; evict-last: 1.357 -> 1.353 ms).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, const void* src, int32_t x,
                                             int32_t y)
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(m)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most one committed bulk store still reads its shared-memory source.
__device__ __forceinline__ void bulk_wait_read1()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Wait until no committed bulk store still reads its shared-memory source.
__device__ __forceinline__ void bulk_wait_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store has completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on bar when every tcgen05 async op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle: rows of 128
// bytes, 8-row groups (1024 B) one after another.  The tile base must be 1024-aligned;
// the start address may be advanced by k-step offsets inside the 128-byte row.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;             // leading byte offset (ignored for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;   // stride byte offset: next 8-row group
    d |= (uint64_t)1u << 46;             // descriptor version for tcgen05
    d |= (uint64_t)2u << 61;             // 128-byte swizzle
    return d;
}

// Descriptor of a 32-row x 16-byte scale-factor block (no swizzle): 8-row core matrices of
// 128 contiguous bytes, the four of them 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// Copy one 512-byte scale atom (32 rows x 16 bytes) into TMEM, replicated to the four
// 32-lane quarters: lane l, column c then holds the 4 scales of row 32c + l.  (The GEMMs
// write the same layout with tcgen05.st from four "scale warps" instead: a copy issued by
// the MMA thread sits in the same in-order queue as the MMAs and serialises with them.)
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Instruction descriptor: block-scaled MMA, E2M1 x E2M1 with UE4M3 scales (NVFP4),
// fp32 accumulate, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N)
{
    return (1u << 7)                              // A: E2M1
           | (1u << 10)                           // B: E2M1
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | (0u << 23)                           // scale type UE4M3
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulate, K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4)                              // D: fp32
           | (1u << 7)                            // A: bf16
           | (1u << 10)                           // B: bf16
           | ((uint32_t)(N >> 3) << 17)
           | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]^T with per-16 UE4M3 block scales from TMEM (K = 64).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_taddr, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_taddr,
                                            uint32_t sfb_taddr, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
        "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_taddr),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_taddr), "r"(sfb_taddr), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, bf16 operands (K = 16).
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_taddr, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_taddr),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, bf16 operands (K = 16).  A sits in TMEM: lane m holds
// row m, each 32-bit column two consecutive K elements (lower K index in the low half), so a
// K = 16 step spans 8 columns from a_taddr.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_taddr, uint32_t a_taddr,
                                               uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
        "r"(a_taddr), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Each thread of the warp writes 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ NVFP4 conversions

// fp32 -> E4M3 byte, round to nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float q)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(q));
    return r & 0xFFu;
}

// E4M3 byte (non-negative, not NaN) -> fp32, from the format: exponent bias 7,
// 3 mantissa bits, exponent 0 subnormal (m * 2^-9).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b)
{
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    return e == 0 ? (float)m * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight fp32 values -> eight E2M1 codes (round to nearest even, saturating at +-6),
// packed little-endian: value 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t f32x8_to_e2m1(const float* v)
{
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
          "f"(v[7]));
    return out;
}

// Quantise 16 fp32 values with global encode scale gs (the NVFP4 block step):
//   m = max|x|;  sf = E4M3(m*gs/6);  sf == 0 -> all codes +0;
//   r = gs / E4M3value(sf);  code_i = E2M1(x_i * r)
// Every operation is an IEEE round-to-nearest fp32 operation (no contraction).
// Writes 8 code bytes to codes[0..1] (two 32-bit words) and returns the scale byte.
__device__ __forceinline__ uint32_t quant16(const float* x, float gs, uint32_t* codes)
{
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(x[i]));
    const float q = __fdiv_rn(__fmul_rn(m, gs), 6.0f);
    const uint32_t sf = f32_to_e4m3(q);
    if (sf == 0) {
        codes[0] = codes[1] = 0u;
        return 0u;
    }
    const float r = __fdiv_rn(gs, e4m3_to_f32(sf));
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(x[i], r);
    codes[0] = f32x8_to_e2m1(y);
    codes[1] = f32x8_to_e2m1(y + 8);
    return sf;
}

// Byte offset of scale (row, block) in the tiled atom layout of a K-wide matrix:
// atom (row/128, block/4) of 512 bytes; inside it row m at (m%32)*16 + (m/32)*4.
__host__ __device__ __forceinline__ size_t sf_atom_offset(int64_t row, int block, int K)
{
    const int64_t rb = row >> 7;
    const int m = (int)(row & 127);
    const int s = block >> 2, kk = block & 3;
    return (size_t)((rb * (K / 64) + s) * 512 + (m & 31) * 16 + (m >> 5) * 4 + kk);
}

__host__ __device__ __forceinline__ int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Row pitch (bytes) of tiled NVFP4 codes of a K-wide matrix.
__host__ __device__ __forceinline__ int codes_pitch(int K) { return round_up(K / 2, 128); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

}  // namespace moe
