// sm103_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100a family,
// here sm_103a) asynchronous machinery the fp16 kernel is built from:
// mbarriers with transaction counts, TMA tensor loads, and the tcgen05
// tensor-core instructions with their Tensor Memory (TMEM) accumulators.
//
// The pages describe this machinery in prose only ("异步拷贝与 Hopper/Blackwell
// 新特性", sections "TMA：张量内存加速器 sm_90+" and "Blackwell 概览 sm_100";
// "第 6 章 · Shared Memory & Tile", section "6.10.4 Blackwell TMEM GEMM —
// TCGEN05"); the encodings below follow the PTX ISA's definitions of
// tcgen05.mma, its instruction descriptor and its shared-memory matrix
// descriptor.
#pragma once

#include <cstdint>

namespace gb300 {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the barrier's expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Longest time a waiting thread stays suspended inside one try_wait before it
// re-checks (it wakes at once when the phase completes).  Suspending instead of
// re-polling frees issue slots and power; measured faster under the power cap.
constexpr uint32_t kWaitSuspendNs = 20000;

// True once the phase with parity `parity` has completed.  A fresh barrier is
// in phase 0, so waiting for parity 1 returns at once (the "previous" phase).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    return ok != 0;
}

// Bounded wait: spins on try_wait; gives up (returns false) when `*abort` is
// set by another role or when `budget_ns` of wall time has passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t budget_ns,
                                          const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > budget_ns) return false;
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tile mode, completion counted on an mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const void *desc) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// Ask L2 for the box at coordinates (c0 innermost, c1): a hint that fills L2
// and writes nothing else, so values read later are never affected by it.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void *desc, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(desc)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// Load the box at coordinates (c0 innermost, c1) into shared memory `dst`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *desc, uint32_t bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, TMEM -> register loads
// ---------------------------------------------------------------------------

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the TMEM
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_alloc_permit() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T for kind::f16 (fp16/bf16 in, fp32 accumulate).
// `accumulate` == 0 overwrites D.  Issued by a single thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 async operation this thread issued
// before (MMAs, with their shared-memory reads) has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Warp-wide: this warp's 32 TMEM lanes (lane base from the address), 32
// consecutive 32-bit columns per lane -> 32 registers per thread.  The load
// and its completion wait are one asm statement so that no use of the
// registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// ---------------------------------------------------------------------------
// Clusters and CTA pairs (tcgen05 .cta_group::2)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Four fp32 values at a shared::cluster address (another CTA's shared memory).
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

// All threads of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same barrier, ordering execution only: the arrive releases nothing, so
// whatever another CTA must see has to be released before it (barrier
// initialisation by fence.mbarrier_init.release.cluster) or be carried by an
// mbarrier that CTA has already waited on.  Measured ~0.5 us cheaper than the
// releasing form at kernel start and ~0.4 us at kernel end.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile(
        "barrier.cluster.arrive.relaxed.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// try_wait with cluster-scope acquire: for barriers that threads or the
// tensor core of the peer CTA arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t budget_ns,
                                                  const volatile int *abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > budget_ns) return false;
    }
}

// Arrive on a barrier given by its shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on a
// barrier that may live in the peer CTA of the pair (`bar_cluster` is a
// shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *desc, uint32_t bar_cluster,
                                                 int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

// The same, multicast: the box lands at offset `dst` in every CTA of
// `cta_mask`, and each receiving CTA's bytes are counted on the barrier at
// the offset of `bar_cluster` in the even CTA of that CTA's pair.
__device__ __forceinline__ void tma_load_2d_pair_multicast(uint32_t dst, const void *desc,
                                                           uint32_t bar_cluster, int c0, int c1,
                                                           uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".multicast::cluster.cta_group::2 [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar_cluster), "r"(c0), "r"(c1), "h"(cta_mask)
        : "memory");
}

// One warp in each CTA of the pair allocates the same TMEM columns in both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_alloc_permit_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Pair MMA, issued by one thread of the even CTA: A rows come half from each
// CTA's shared memory, B columns half from each, and each CTA's TMEM receives
// its own 128 rows of D.
__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at offset `bar` in every CTA of `cta_mask` when
// all earlier tcgen05 operations of this thread have completed.
__device__ __forceinline__ void mma_commit_pair_multicast(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------

// Let the next kernel of the stream (if launched with programmatic stream
// serialisation) begin its launch once every CTA of this grid has called this
// or exited.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Block until the grids this one depends on have completed and their memory
// operations are visible.  A no-op when launched without the dependency.
__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA stores (shared -> global), bulk-group completion
// ---------------------------------------------------------------------------

// Store the box at (c0 innermost, c1) from shared memory `src`; elements
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void *desc, uint32_t src, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(desc)),
        "r"(src), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Global flags between CTAs of one grid (all co-resident)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *flag == value; false when `budget_ns` passed or *abort was set.
__device__ __forceinline__ bool wait_flag_equal(const uint32_t *flag, uint32_t value,
                                                uint64_t budget_ns, const volatile int *abort) {
    if (ld_acquire_gpu(flag) == value) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire_gpu(flag) == value) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > budget_ns) return false;
    }
}

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 64 halves (128 B), 8-row swizzle atoms of
// 1024 B stacked along M/N.  Fields: start address >> 4 in [0,14), leading
// byte offset >> 4 in [16,30) (not used by swizzled K-major layouts; 1), stride
// byte offset >> 4 in [32,46) (1024 B between 8-row atoms), the fixed value
// 0b001 in [46,49), base offset 0 in [49,52) (atoms are 1024-byte aligned),
// and the swizzle mode in [61,64) (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits [4,6) = 1),
// A and B fp16 (bits [7,10) and [10,13) = 0), both K-major (bits 15, 16 = 0),
// N >> 3 in [17,23), M >> 4 in [24,29).
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Block-scaled FP8 (kind::mxf8f6f4): scale factors, bulk copies, the MMA
// ---------------------------------------------------------------------------

// Contiguous global -> shared copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Shared-memory descriptor of an unswizzled K-major block: rows of 16 bytes,
// 8-row core matrices `sbo` bytes apart along M/N (`lbo` along K).
__device__ __forceinline__ uint64_t plain_kmajor_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version of sm_100+; layout 0 = no swizzle
    return d;
}

// Shared -> TMEM: 32 rows of 128 bits (16 bytes) into TMEM lanes 0..31,
// repeated in each of the four 32-lane quarters, 4 columns from `taddr`.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D (fp32, TMEM) (+)= (A * 2^SA) (B * 2^SB)^T for FP8 A, B in shared memory
// and UE8M0 scale factors in TMEM (one per row per 32 K, the byte chosen by
// the descriptor's scale-factor IDs).
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// The CTA-pair forms (issued by the even CTA for both): the copy moves the
// chunk at the same shared-memory offset of each CTA into that CTA's TMEM;
// the MMA takes A's rows and half of B's from each CTA.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void mma_mxf8_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// D (fp32) (+)= (A * SA) (B * SB)^T for packed FP4 (E2M1) A, B and 8-bit
// scales, one per row per 16 elements of K: each MMA (K = 64) takes all four
// scale bytes of the row's TMEM word.
__device__ __forceinline__ void mma_nvf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Block-scaled descriptor for FP4 E2M1 operands (format 1 in [7,10) and
// [10,13)) with UE4M3 scales (bit 23 = 0), K = 64 (bit 31 = 0), scale IDs 0.
__host__ __device__ constexpr uint32_t idesc_nvf4_e2m1(int m, int n) {
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor of the block-scaled kinds: B scale-factor ID in
// [4,6), A and B formats in [7,10) and [10,13) (E4M3 = 0), K-major (bits 15,
// 16 = 0), N >> 3 in [17,23), scale format UE8M0 (bit 23 = 1), M >> 4 in
// [24,29), A scale-factor ID in [29,31); D is fp32.
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int m, int n, int sf_id) {
    return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(m >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

}  // namespace gb300
