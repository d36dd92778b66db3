// glu_tc.cuh -- the batched GEMV on the fifth-generation tensor cores
// (tcgen05), batches of 17..64 rows in one pass over the weights.
//
// With the weights as the MMA's M side ("swap AB"), a CTA owns a tile of 128
// weight rows and one of ksplit ranges of K.  Per 64-wide K chunk it receives
// by tensor copy, in the 128-byte swizzled layout:
//   gate_w[tile rows][chunk], up_w[tile rows][chunk]   16 KB each
//   h[batch rows][chunk], rows M..Np-1 zero-filled     Np * 128 bytes
// and one thread issues, per 16-wide K step, two MMAs (128 x Np x 16):
//   g^T += gate_w_tile * h^T  in tensor-memory columns [0, Np)
//   u^T += up_w_tile * h^T    in columns [C/2, C/2 + Np), C = the columns allocated
// Tensor-memory lane i holds weight row i of the tile, column m the batch
// row.  Every SM takes in the weight bytes of its tile once, plus the
// (L2-resident) h chunks: no per-batch-block re-reads.
//
// Roles (192 threads): warp 0 lane 0 copies, warp 1 lane 0 issues MMAs and
// warp 1 owns the tensor memory, warps 2-5 read the accumulators (warp w may
// read lanes 32 * (w % 4) .. +31).  With ksplit = 2..4 the CTAs of a tile
// form a cluster: rank 0 frees its stage memory once its MMAs are done,
// ranks 1.. write their partial sums there (slot r - 1, [128 rows][2 Np + 4]
// fp32, 16-byte stores) through distributed shared memory, and rank 0 adds them (own, then ranks 1, 2, ... in order)
// before the epilogue.  Every wait is bounded; every thread reaches the final
// cluster barrier, so no CTA leaves while another may still touch its memory.
#pragma once

#include "glu_kernels.cuh"
#include "tcgen05.cuh"

namespace mbglu {

constexpr int kTcRows = 128;                              // weight rows per tile: the MMA's M
constexpr int kTcBox = 64;                                // K per tensor copy: one 128-byte swizzled row
constexpr int kTcBoxes = 2;                               // copies per matrix and stage, adjacent in K
constexpr int kTcChunk = kTcBox * kTcBoxes;               // K per stage: 128 (256 bytes of each row)
constexpr int kTcMaxStages = 8;
constexpr uint32_t kTcWBox = kTcRows * kTcBox * 2;        // one matrix's box: 16 KB
constexpr uint32_t kTcWBytes = kTcWBox * kTcBoxes;        // one matrix's stage: 32 KB
constexpr int kTcThreads = 192;
constexpr uint32_t kTcHeader = 1024;                      // barriers, tensor-memory address
constexpr uint32_t kTcSmemSlack = 1024;                   // room to align the stages to 1024 bytes
constexpr int kTcMaxSplit = 4;                            // CTAs per tile at most (K split over a cluster)

// Row pitch (fp32) of a rank's partial sums in rank 0's shared memory: a
// weight row's Np g values then Np u values, 4 floats of padding so that the
// 16-byte accesses of consecutive rows fall in different banks.
__host__ __device__ constexpr int tc_part_pitch(int Np) { return 2 * Np + 4; }

struct TcParams {
    uint16_t *out;
    int64_t ldo;
    int M, N, K, mode;
    int Np;          // batch rows padded to a multiple of 16: the MMA's N
    int nchunk;      // kTcChunk-wide K chunks
    int ksplit;      // CTAs per tile (the cluster size), 1..kTcMaxSplit
    int stages;
    int prefetch;    // weight stages requested before the dependency wait
};

struct TcMaps {
    TensorMap gate, up;   // [N][K] bf16, box 64 x 128, 128-byte swizzle
    TensorMap h;          // [M][K] bf16, box 64 x Np, 128-byte swizzle
};

__global__ void __launch_bounds__(kTcThreads, 1) glu_tc_kernel(const TcParams p, const __grid_constant__ TcMaps maps)
{
    extern __shared__ unsigned char tc_smem[];
    unsigned char *base = tc_smem + ((1024u - (smem_addr(tc_smem) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(base);      // [stage]: the chunk has landed
    uint64_t *empty = full + kTcMaxStages;                     // [stage]: its MMAs have read it
    uint64_t *acc_bar = empty + kTcMaxStages;                  // every MMA of the CTA is done
    uint64_t *go_bar = acc_bar + 1;                            // ranks 1..: rank 0's stage memory is free
    uint64_t *red_bar = go_bar + 1;                            // rank 0: the other ranks' partial sums have landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red_bar + 1);
    unsigned char *stages = base + kTcHeader;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages, Np = p.Np, ks = p.ksplit;
    const uint32_t hbox = static_cast<uint32_t>(Np) * 128u;   // one h box: Np rows of 64 columns
    const uint32_t sbytes = 2 * kTcWBytes + hbox * kTcBoxes;
    const uint32_t rank = ks > 1 ? cluster_ctarank() : 0u;
    const int tile = static_cast<int>(blockIdx.x) / ks;
    const int c0 = p.nchunk * static_cast<int>(rank) / ks;
    const int nch = p.nchunk * (static_cast<int>(rank) + 1) / ks - c0;
    const uint32_t ncols = 2 * Np <= 64 ? 64u : 128u;          // a power of two >= 2 Np
    const uint32_t ucol = ncols / 2;                            // u's accumulator columns start here (>= Np)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_bar, 1);
        mbar_init(go_bar, 1);
        mbar_init(red_bar, (ks > 1 ? ks - 1 : 1) * kTcRows);   // the other ranks' 128 epilogue threads each
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    tc_fence_after();
    if (ks > 1) cluster_sync();   // both CTAs' barriers exist before any remote arrival
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_h = l2_policy_evict_last();   // every tile reads h
            const int row0 = tile * kTcRows;
            const int pre = p.prefetch ? min(S, nch) : 0;
            // a stage: gate boxes, up boxes, h boxes; the boxes of one matrix
            // adjacent in K and issued back to back (longer runs of each row)
            auto load_w = [&](int s, int k) {
                unsigned char *st = stages + s * sbytes;
#pragma unroll
                for (int b = 0; b < kTcBoxes; ++b)
                    tma_load_2d(st + b * kTcWBox, &maps.gate, k + b * kTcBox, row0, &full[s], pol_w);
#pragma unroll
                for (int b = 0; b < kTcBoxes; ++b)
                    tma_load_2d(st + kTcWBytes + b * kTcWBox, &maps.up, k + b * kTcBox, row0, &full[s], pol_w);
            };
            auto load_h = [&](int s, int k) {
                unsigned char *st = stages + s * sbytes + 2 * kTcWBytes;
#pragma unroll
                for (int b = 0; b < kTcBoxes; ++b) tma_load_2d(st + b * hbox, &maps.h, k + b * kTcBox, 0, &full[s], pol_h);
            };
            for (int i = 0; i < pre; ++i) {   // weights only: nothing before the wait may depend on the predecessor
                mbar_arrive_expect_tx(&full[i], sbytes);
                load_w(i, (c0 + i) * kTcChunk);
            }
            grid_dependency_wait();
            for (int i = 0; i < pre; ++i) load_h(i, (c0 + i) * kTcChunk);
            int issued = pre;
            for (int i = pre; i < nch; ++i) {
                const int s = i % S;
                if (i >= S && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((i / S - 1) & 1), kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const int k = (c0 + i) * kTcChunk;
                mbar_arrive_expect_tx(&full[s], sbytes);
                load_w(s, k);
                load_h(s, k);
                issued = i + 1;
            }
            // none of this CTA's copies may still be in flight when it leaves:
            // wait for the last chunk issued into each stage
            for (int i = max(0, issued - S); i < issued; ++i)
                if (!mbar_wait_bounded(&full[i % S], static_cast<uint32_t>((i / S) & 1), kWaitLimitNs)) ok = false;
        } else {
            grid_dependency_wait();
        }
    } else {
        grid_dependency_wait();
    }
    grid_launch_dependents();

    if (warp == 1 && lane == 0) {
        const uint32_t idesc = tc_idesc_bf16(kTcRows, Np);
        for (int i = 0; i < nch; ++i) {
            const int s = i % S;
            if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((i / S) & 1), kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            unsigned char *st = stages + s * sbytes;
#pragma unroll
            for (int b = 0; b < kTcBoxes; ++b) {
                const uint64_t ag = smem_desc_sw128(st + b * kTcWBox);
                const uint64_t au = smem_desc_sw128(st + kTcWBytes + b * kTcWBox);
                const uint64_t bh = smem_desc_sw128(st + 2 * kTcWBytes + b * hbox);
#pragma unroll
                for (int kk = 0; kk < kTcBox / 16; ++kk) {
                    const bool acc = i > 0 || b > 0 || kk > 0;
                    tc_mma_bf16(tmem, ag + 2 * kk, bh + 2 * kk, idesc, acc);
                    tc_mma_bf16(tmem + ucol, au + 2 * kk, bh + 2 * kk, idesc, acc);
                }
            }
            tc_commit(&empty[s]);   // the stage is free once these MMAs have read it
        }
        tc_commit(acc_bar);   // after a timeout too: it fires once the MMAs issued so far are done
    }

    if (warp >= 2) {
        const int q = warp & 3;                     // the tensor-memory lane quarter this warp may read
        const int row = q * 32 + lane;              // weight row within the tile
        const int n = tile * kTcRows + row;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const bool ready = __all_sync(0xffffffffu, mbar_wait_bounded(acc_bar, 0, kWaitLimitNs));
        tc_fence_after();
        if (!ready) ok = false;
        if (ks == 1 || rank == 0) {
            bool have_partial = false;
            if (ks > 1) {
                // rank 0's stages are free: every MMA (and so every copy) is done
                if (threadIdx.x == 64) {
                    fence_proxy_async_smem();   // the copies' writes and the MMAs' reads before the others' stores
                    for (int r = 1; r < ks; ++r) mbar_arrive_remote(map_to_rank(go_bar, static_cast<uint32_t>(r)));
                }
                have_partial = __all_sync(0xffffffffu, mbar_wait_cluster_bounded(red_bar, 0, kWaitLimitNs));
                if (!have_partial) ok = false;
            }
            // [rank - 1][128 rows][2 Np + 4] fp32: a row's g then u partials
            const float *part = reinterpret_cast<const float *>(stages);
            const int pitch = tc_part_pitch(Np), slot = kTcRows * pitch;
            for (int c = 0; c < Np; c += 16) {
                float g[16], u[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c), g);
                tmem_ld16(taddr + ucol + static_cast<uint32_t>(c), u);
                if (have_partial) {
                    for (int r = 1; r < ks; ++r) {
                        const float4 *pg = reinterpret_cast<const float4 *>(part + (r - 1) * slot + row * pitch + c);
                        const float4 *pu = reinterpret_cast<const float4 *>(part + (r - 1) * slot + row * pitch + Np + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 a = pg[j], b = pu[j];
                            g[4 * j] += a.x;
                            g[4 * j + 1] += a.y;
                            g[4 * j + 2] += a.z;
                            g[4 * j + 3] += a.w;
                            u[4 * j] += b.x;
                            u[4 * j + 1] += b.y;
                            u[4 * j + 2] += b.z;
                            u[4 * j + 3] += b.w;
                        }
                    }
                }
                if (ready && n < p.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c + j < p.M) p.out[static_cast<int64_t>(c + j) * p.ldo + n] = glu_epilogue(g[j], u[j], p.mode);
                }
            }
        } else {
            // ranks 1..: the partial sums into slot rank - 1 of rank 0's stage
            // memory once rank 0 frees it
            const bool go = __all_sync(0xffffffffu, mbar_wait_cluster_bounded(go_bar, 0, kWaitLimitNs));
            if (!go) ok = false;
            const int pitch = tc_part_pitch(Np);
            const uint32_t dst = map_to_rank(stages, 0) +
                                 static_cast<uint32_t>(((rank - 1) * kTcRows + row) * pitch * 4);
            for (int c = 0; c < 2 * Np; c += 16) {   // g's columns 0..Np-1, then u's
                float v[16];
                tmem_ld16(taddr + (c < Np ? static_cast<uint32_t>(c) : ucol + static_cast<uint32_t>(c - Np)), v);
                if (go) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_cluster_v4_f32(dst + static_cast<uint32_t>((c + 4 * j) * 4), v[4 * j], v[4 * j + 1],
                                          v[4 * j + 2], v[4 * j + 3]);
                }
            }
            mbar_arrive_remote(map_to_rank(red_bar, 0));   // also after a timeout, so rank 0 is not kept waiting
        }
    }

    if (!ok) atomicExch(&g_device_error, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    __syncwarp();   // the warp-collective operations below need converged warps
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
    if (ks > 1) cluster_sync();   // neither CTA leaves while the other may still access its shared memory
}

}  // namespace mbglu
