// tcgen05.cuh -- inline-PTX wrappers for the fifth-generation tensor cores
// (sm_100 family, here sm_103a), one CTA per MMA (cta_group::1): tensor
// memory allocation, the MMA with both operands in shared memory and the
// accumulator in tensor memory, its completion on an mbarrier, tensor-memory
// loads, and the cluster operations the split-K reduction uses.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mbglu {

// Allocates ncols (a power of two, 32..512) tensor-memory columns; the
// address (lane in bits 31:16, column in 15:0) is written to *slot.  Whole
// warp, converged.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
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

// Orders tcgen05 operations around a thread synchronisation.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// d (+)= A * B^T with A (M x 16) and B (N x 16) K-major bf16 tiles in shared
// memory, fp32 accumulator in tensor memory; accumulate = false overwrites.
// One thread issues.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// One arrival on bar once every tcgen05 operation this thread issued before
// has completed (shared memory read, accumulator written).
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of one tensor-memory lane per thread: thread t
// of the warp reads lane (taddr's lane + t).  A warp may touch only the
// 32-lane quarter (warp index % 4) of tensor memory.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major bf16 tile in the layout a
// tensor copy with 128-byte swizzling writes: rows of 64 elements (128 bytes),
// groups of 8 rows 1024 bytes apart, the tile 1024-byte aligned.  Fields:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (not used by swizzled
//               K-major layouts; 1)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 bytes: 8-row groups)
//   bits 46-47  descriptor version, 1 on the sm_100 family
//   bits 49-51  base offset (0: 1024-byte aligned tiles)
//   bits 61-63  swizzle: 2 = 128-byte
// Advancing K by 16 elements (32 bytes) inside the swizzled row adds 2 to the
// start-address field.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void *tile)
{
    const uint64_t addr = smem_addr(tile);
    return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, an M x N tile.
//   bits  4-5   D format (1: f32)       bits  7-9   A format (1: bf16)
//   bits 10-12  B format (1: bf16)      bits 15, 16 A, B major (0: K-major)
//   bits 17-22  N >> 3                  bits 24-28  M >> 4
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int m, int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// ---- clusters ----------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders the barrier
// initialisations before any remote access.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address of this shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 16 bytes (addr 16-byte aligned) into another CTA's shared memory
__device__ __forceinline__ void st_cluster_v4_f32(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Arrival on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}

// Bounded wait that acquires at cluster scope (arrivals from other CTAs).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t phase)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t phase, uint64_t limit_ns)
{
    if (mbar_try_wait_cluster(bar, phase)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_cluster(bar, phase)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

}  // namespace mbglu
