// tma.cuh -- inline-PTX helpers for the Tensor Memory Accelerator and shared
// memory barriers (sm_90+ PTX ISA: mbarrier.*, cp.async.bulk.tensor.*), plus the
// host-side lookup of cuTensorMapEncodeTiled through the runtime.
//
// Every wait is bounded: wait_parity_bounded waits for at most kWaitLimitNs of
// %globaltimer time; on expiry it sets FNO_DEVERR_TIMEOUT in the error word and
// returns false so the kernel can leave without hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fno {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA) before use.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may be suspended for up to `hint_ns` while
// the phase is incomplete; it resumes as soon as the phase completes.  A
// suspended warp takes no issue slots, where a polling loop would spend them
// on the timer reads, compares and branches of every retry.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

constexpr uint32_t kSleepHintNs = 100000;  // per retry; the total stays bounded below

// Wait for phase `parity` of the barrier to complete, for at most kWaitLimitNs.
// `err` points at the plan's two device words: err[0] collects error bits,
// err[1] holds debug flags.  With bit 0 of err[1] set (the forced-timeout test
// hook) every such wait gives up at once, as if its time had run out.  The flag
// is written by the host between launches only, so the read-only cache may hold
// it (one L2 read per SM, L1 hits after).  Waits that drain copies or MMAs still
// in flight pass err = nullptr: they are bounded but never cut short, so that
// no kernel leaves while an asynchronous operation can still write its shared
// or tensor memory.
__device__ __forceinline__ bool wait_parity_bounded(uint64_t* bar, uint32_t parity,
                                                    unsigned* err) {
    if (err && (__ldg(err + 1) & 1u)) {
        atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < kWaitLimitNs)
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (err) atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
    return false;
}

// 3D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Bulk copy of `bytes` contiguous bytes from global memory into shared memory,
// completing on `bar` (complete_tx).  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Ask the TMA unit to pull [p, p + bytes) into L2 (no completion to wait for).
// p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace fno

// Host: the driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (no link-time dependency on libcuda).  Returns nullptr if unavailable.
typedef CUresult (*fno_encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                        const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                        const cuuint32_t*, CUtensorMapInterleave,
                                        CUtensorMapSwizzle, CUtensorMapL2promotion,
                                        CUtensorMapFloatOOBfill);
fno_encode_tiled_fn fno_get_encode_tiled();

namespace fno {

// 3D tiled TMA store of one box from shared memory (bulk-group completion:
// commit with bulk_commit(), wait with bulk_wait_read0() before the shared
// memory is reused or the CTA exits).  Elements of the box outside the
// tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int c0,
                                             int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk group of this thread has finished reading
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

}  // namespace fno
