// glu_slice.cuh -- the dual-weight GLU GEMV at batch 1..16 on the tensor
// cores, with h held in registers.
//
// DeepSpeed PR #8602, comment "Plan B: Dual-Weight GEMV", section "Plan B
// Design": one pass over h reads gate_w and up_w in place and applies
// SiLU(g) * u in the epilogue; PR #9057's A100 commit runs decode at batch 8
// and above, and batch 1 is the comment's own case.  g[m][n] = sum_k h[m][k] Wg[n][k],
// u likewise, then the mode's epilogue (glu_epilogue) or the backward's dG, dU
// (glu_store).
//
// Layout of the work.  A CTA owns a balanced share [r0, r1) of the N rows,
// in groups of 8 (the MMA's n); the last group may run past r1 (its extra
// rows belong to the next CTA or lie past N, where the copy reads zeros) and
// only rows < r1 are stored.  Compute warp w owns the K columns [x0, x0 +
// 256 SPW), x0 = 256 SPW w, as SPW segments of 256 columns: it holds h's MMA
// fragments for those columns in registers for the whole kernel (32 SPW per
// lane) and streams, for each of the CTA's groups in order, the group's 8
// rows of both matrices over its segments through a private ring of S stages.
// A stage is one segment: four 64-column x 8-row boxes per matrix (8 KB),
// 128-byte swizzled (16-byte chunk j of row r at r * 128 + ((j ^ r) << 4)),
// so each ldmatrix of 8 rows meets no bank conflict.  No h in shared memory,
// so nearly all of it is ring: 160 KB of weights in flight per SM at K = 2560
// (10 warps x 2 stages), 192 KB at K = 4096 (8 warps x 3 stages).
//
// Arithmetic: A (16 x 16) = h's rows 0..15 at the k-step (rows >= M read as
// zero; at MB = 8, for M <= 8, rows 8..15 are the zero registers a1 and a3),
// B (16 x 8) = 8 weight rows, D = g (or u) for the batch rows x 8 features.  Per segment one MMA chain per
// matrix over its 16 k-steps, started from zero (the tensor core's adds are
// not specified to round to nearest; a chain stays 16 MMAs long); the chains
// are added to the warp's fp32 partial in segment order (round to nearest).
// The warps' partials of a group go through a ring of slots (4 at MB = 8, 2
// at MB = 16) to the epilogue warp (warp W), which adds them in warp order
// (round to nearest) and stores.  Every sum runs in a fixed order: results
// are bitwise deterministic and do not depend on the timing of the warps.
//
// MB = 16 (batch 9..16) holds h's rows 8..15 too (64 registers per lane at
// one segment per warp, so up to 10 warps: K up to 2560).
//
// NORM (add_rmsnorm_glu, [9057/Changes] zero-centred RMSNorm): the block
// first forms h in shared memory with the norm prologue of the other kernels
// (residual rows copied in, s = bf16(x + residual) when fused, the
// double-float statistic and the correctly rounded h = bf16(s inv (1 + w)),
// all threads taking part), at a row pitch of K + 8 so that the warps' loads
// of their fragments meet no bank conflict (K % 16 == 0; two rows share a
// bank at K % 16 == 8); a barrier then hands the region
// to the slots.  When fused, the epilogue warp writes this CTA's slice of the
// residual at the end, once every CTA has read it (fused_residual_helper).
//
// Shared memory (dynamic, from a 1024-byte aligned base):
//   [0, 512)        mbarriers [warp][stage] (W S <= 64)
//   [512, 576)      slot barriers: full[slots] (count 32 W), empty[slots] (count 32)
//   [784, 792)      NORM: the prologue copies' mbarrier (kProBarOffset)
//   [1024, ...)     slots [slots][W][NP][32] fp32: lane l's g(m, n), g(m, n+1)[, g(m+8, n),
//                   g(m+8, n+1)], then u likewise, m = l / 4, n = 2 (l % 4); NORM: first h_s[M][K + 8]
//   [off_s, ...)    NORM: norm_w [K] bf16, then the statistic's partials (2 floats per thread)
//   [off_ring, ...) ring [W][S][matrix][4][8][64] bf16
#pragma once

#include "glu_kernels.cuh"

namespace mbglu {

constexpr int kSliceBoxes = 4;                                  // 64-column boxes per segment
constexpr int kSliceSeg = 64 * kSliceBoxes;                     // 256 columns
constexpr uint32_t kSliceBox = 8u * 128u;                       // one 64 x 8 box, bytes
constexpr uint32_t kSliceStage = 2u * kSliceBoxes * kSliceBox;  // both matrices, 8 KB
// the most compute warps (plus the epilogue warp) at SPW segments per warp:
// what the registers a thread needs (h's 32 SPW fragments and the rest)
// leave on each of the SM's four register files
__host__ __device__ constexpr int slice_max_warps(int spw, int mb = 8)
{
    return mb > 8 ? 10 : spw <= 1 ? 12 : spw == 2 ? 8 : 6;
}
// group slots between the compute warps and the epilogue warp (MB = 16
// carries twice the partial sums per slot)
__host__ __device__ constexpr int slice_slots(int mb) { return mb > 8 ? 2 : 4; }

// one warp's partials of one group: 4 (MB = 8) or 8 (MB = 16) floats per lane
__host__ __device__ constexpr uint32_t slice_slot_bytes(int mb) { return (mb > 8 ? 8u : 4u) * 32u * 4u; }

struct SliceMaps {
    TensorMap gate, up;   // [N][K] bf16, box 64 x 8, 128-byte swizzle
};

template <int SPW, bool NORM, int MB>
__global__ void __launch_bounds__(32 * (slice_max_warps(SPW, MB) + 1), 1)
    glu_slice_kernel(const GluParams p, const __grid_constant__ SliceMaps maps)
{
    static_assert(MB == 8 || MB == 16, "batch tile of 8 or 16 rows");
    static_assert(!(NORM && MB > 8), "the norm variant takes batch 1..8");
    constexpr int NP = MB > 8 ? 8 : 4;         // partial sums per lane and group
    constexpr int NA = MB > 8 ? 4 : 2;         // A registers per k-step
    constexpr int NSLOT = slice_slots(MB);
    extern __shared__ __align__(128) unsigned char sl_raw[];
    __shared__ float inv_s[2 * 8];   // NORM: (inv_hi, inv_lo) per row
    unsigned char *sm = sl_raw + ((1024u - (smem_addr(sl_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = static_cast<int>(blockDim.x >> 5) - 1;   // compute warps; warp W runs the epilogue
    const int S = p.stages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm);      // [W][S]
    uint64_t *full = bars + 64;
    uint64_t *empty = full + NSLOT;
    float *slots = reinterpret_cast<float *>(sm + 1024);
    const int r0 = static_cast<int>((static_cast<int64_t>(p.N) * blockIdx.x) / gridDim.x);
    const int r1 = static_cast<int>((static_cast<int64_t>(p.N) * (blockIdx.x + 1)) / gridDim.x);
    const int ngroups = (r1 - r0 + 7) >> 3;
    const int x0 = warp * (SPW * kSliceSeg);
    // this warp's segments: those that start before K
    const int nseg = warp < W ? max(0, min(SPW, (p.K - x0 + kSliceSeg - 1) / kSliceSeg)) : 0;
    const int nunits = ngroups * nseg;   // (group, segment), group-major
    unsigned char *ring = sm + p.off_ring + static_cast<uint32_t>(warp) * S * kSliceStage;
    // the backward's next step reads the weights again: keep them in L2 in that mode
    const uint64_t policy = p.mode == kModeBwd ? l2_policy_evict_last() : l2_policy_evict_first();

    uint64_t *pro_bar = reinterpret_cast<uint64_t *>(sm + kProBarOffset);
    uint16_t *h_s = reinterpret_cast<uint16_t *>(sm + 1024);   // NORM: [M][K + 8], before the slots
    uint16_t *nw_s = reinterpret_cast<uint16_t *>(sm + p.off_s);
    const int HS = p.K + 8;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&full[s], 32u * static_cast<uint32_t>(W));
            mbar_init(&empty[s], 32u);
        }
        if constexpr (NORM) mbar_init(pro_bar, 2);   // the norm_w copy and the residual copy
    }
    if (warp < W && lane == 0)
        for (int st = 0; st < S; ++st) mbar_init(&bars[warp * S + st], 1);
    fence_mbar_init();
    __syncthreads();

    // lane 0: unit u (group u / nseg, segment u % nseg) into stage u % S
    auto fill = [&](int u) {
        const int g = u / nseg, s = u - g * nseg;
        const int st = u % S;
        unsigned char *dst = ring + st * kSliceStage;
        uint64_t *bar = &bars[warp * S + st];
        const int y = r0 + 8 * g, x = x0 + s * kSliceSeg;
        mbar_arrive_expect_tx(bar, kSliceStage);
#pragma unroll
        for (int i = 0; i < kSliceBoxes; ++i) {
            tma_load_2d(dst + i * kSliceBox, &maps.gate, x + 64 * i, y, bar, policy);
            tma_load_2d(dst + (kSliceBoxes + i) * kSliceBox, &maps.up, x + 64 * i, y, bar, policy);
        }
    };
    // bounded waits for this warp's copies in flight, units u..u+S-1 (before an early return)
    auto drain = [&](int u) {
        if (lane == 0)
            for (int v = u; v < min(u + S, nunits); ++v)
                mbar_wait_bounded(&bars[warp * S + v % S], static_cast<uint32_t>((v / S) & 1), kWaitLimitNs);
        __syncwarp();
    };

    auto copy_norm_w = [&]() {
        if constexpr (NORM) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(p.K) * 2u);
                bulk_g2s_plain(nw_s, p.norm_w, static_cast<uint32_t>(p.K) * 2u, pro_bar);
            }
        }
    };
    if (p.prefetch) {   // weights only: before the dependency wait
        copy_norm_w();
        if (lane == 0)
            for (int u = 0; u < min(S, nunits); ++u) fill(u);
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (!p.prefetch) {
        copy_norm_w();
        if (lane == 0)
            for (int u = 0; u < min(S, nunits); ++u) fill(u);
    }
    __syncwarp();

    if constexpr (NORM) {   // h = the normed rows, in h_s (every thread of the block)
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(p.M) * static_cast<uint32_t>(p.K) * 2u);
            copy_rows_async(h_s, HS, p.s, p.K, p.M, p.K, pro_bar);   // the residual rows, padded
        }
        const RowMap rm = row_map(p.M, p.K);
        XRowsN<kXRowsSmall> xr;
        if (p.fused) x_prefetch_rows(p, rm, xr);
        prologue_wait(pro_bar);
        float2 ss;
        if (p.fused) {
            if (threadIdx.x == 0) fused_arrive(p);
            ss = add_rows_in_place(p, rm, h_s, HS, xr);
        } else {
            ss = square_rows(rm, h_s, HS);
        }
        norm_rows_in_place(p, rm, ss, h_s, HS, nw_s, norm_partials(sm, p), inv_s, p.M);   // ends with a barrier
    }

    // the epilogue warp: each group's partials, added in warp order
    auto epilogue = [&]() {
        const int m = lane >> 2, n = 2 * (lane & 3);
        for (int g = 0; g < ngroups; ++g) {
            const int sl = g % NSLOT;
            if (!mbar_wait_bounded(&full[sl], static_cast<uint32_t>((g / NSLOT) & 1), kWaitLimitNs)) {
                if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
                return;
            }
            const float *src = slots + static_cast<int64_t>(sl) * W * NP * 32;
            float acc[NP];
#pragma unroll
            for (int e = 0; e < NP; ++e) acc[e] = src[e * 32 + lane];
            for (int w = 1; w < W; ++w)
#pragma unroll
                for (int e = 0; e < NP; ++e) acc[e] = __fadd_rn(acc[e], src[(w * NP + e) * 32 + lane]);
            mbar_arrive(&empty[sl]);   // every lane, after its reads
            const int row = r0 + 8 * g + n;
            // acc: g at (m, n), (m, n + 1)[, (m + 8, n), (m + 8, n + 1)], then u likewise
#pragma unroll
            for (int hh = 0; hh < MB / 8; ++hh) {
                const int mm = m + 8 * hh;
                if (mm < p.M) {
                    if (row < r1) glu_store(p, mm, row, acc[2 * hh], acc[NP / 2 + 2 * hh]);
                    if (row + 1 < r1) glu_store(p, mm, row + 1, acc[2 * hh + 1], acc[NP / 2 + 2 * hh + 1]);
                }
            }
        }
        if constexpr (NORM) {
            if (p.fused) fused_residual_helper(p);   // this CTA's slice of residual = bf16(x + residual)
        }
    };

    // a compute warp: its K-slice of every group of the share
    auto compute = [&]() {
        // h's A fragments: ha[NA j + ...] = (h[row][k], h[row][k + 1]) at k = x0 + 16 j + 8 e + 2 c for
        // row = g (and g + 8 at MB = 16), in the order a0 (g, e 0), [a1 (g + 8, e 0),] a2 (g, e 1),
        // [a3 (g + 8, e 1)]; zero past K and for batch rows >= M
        const int g4 = lane >> 2, c4 = lane & 3;
        uint32_t ha[NA * 16 * SPW];
#pragma unroll
        for (int j = 0; j < 16 * SPW; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int rr = 0; rr < MB / 8; ++rr) {
                    const int k = x0 + 16 * j + 8 * e + 2 * c4, row = g4 + 8 * rr;
                    uint32_t v = 0;
                    if (row < p.M && k < p.K) {
                        if constexpr (NORM) {
                            v = *reinterpret_cast<const uint32_t *>(h_s + row * HS + k);
                        } else {
                            const uint16_t *src = p.h + static_cast<int64_t>(row) * p.ldh + k;
                            v = p.vec_in ? *reinterpret_cast<const uint32_t *>(src)
                                         : static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[1]) << 16);
                        }
                    }
                    ha[NA * j + (MB / 8) * e + rr] = v;
                }

        if constexpr (NORM) bar_sync_named(1, 32 * W);   // every compute warp holds h: the slots may reuse h_s
        const int mi = lane >> 3, ri = lane & 7;
        int u = 0;
        for (int g = 0; g < ngroups; ++g) {
            float part[NP];
#pragma unroll
            for (int e = 0; e < NP; ++e) part[e] = 0.0f;
#pragma unroll
            for (int s = 0; s < SPW; ++s) {
                if (s >= nseg) break;
                const int st = u % S;
                if (!mbar_wait_bounded(&bars[warp * S + st], static_cast<uint32_t>((u / S) & 1), kWaitLimitNs)) {
                    if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
                    drain(u);
                    return;
                }
                const uint32_t sb = smem_addr(ring + st * kSliceStage);
                float dg[4], du[4];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    // matrices: gate k 0-7, gate k 8-15, up k 0-7, up k 8-15 of this k-step
                    const int ch = 2 * j + (mi & 1);
                    uint32_t b[4];
                    ldsm_x4(b, sb + static_cast<uint32_t>((mi >> 1) * kSliceBoxes * kSliceBox + (ch >> 3) * kSliceBox +
                                                          ri * 128 + (((ch & 7) ^ ri) << 4)));
                    const int q = 16 * s + j;
                    uint32_t a[4];
                    if constexpr (MB > 8) {
                        a[0] = ha[4 * q];
                        a[1] = ha[4 * q + 1];
                        a[2] = ha[4 * q + 2];
                        a[3] = ha[4 * q + 3];
                    } else {
                        a[0] = ha[2 * q];
                        a[1] = 0u;
                        a[2] = ha[2 * q + 1];
                        a[3] = 0u;
                    }
                    if (j == 0) {
                        mma16_bf16_z(dg, a, b[0], b[1]);
                        mma16_bf16_z(du, a, b[2], b[3]);
                    } else {
                        mma16_bf16(dg, a, b[0], b[1]);
                        mma16_bf16(du, a, b[2], b[3]);
                    }
                }
#pragma unroll
                for (int e = 0; e < NP / 2; ++e) {
                    part[e] = __fadd_rn(part[e], dg[e]);
                    part[NP / 2 + e] = __fadd_rn(part[NP / 2 + e], du[e]);
                }
                __syncwarp();
                if (lane == 0 && u + S < nunits) {
                    fence_proxy_async_smem();
                    fill(u + S);   // the unit S ahead, into the stage just read
                }
                ++u;
            }
            // the group's partials to the epilogue warp
            const int sl = g % NSLOT;
            if (g >= NSLOT &&
                !mbar_wait_bounded(&empty[sl], static_cast<uint32_t>((g / NSLOT - 1) & 1), kWaitLimitNs)) {
                if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
                drain(u);
                return;
            }
            float *dst = slots + (static_cast<int64_t>(sl) * W + warp) * NP * 32;
#pragma unroll
            for (int e = 0; e < NP; ++e) dst[e * 32 + lane] = part[e];
            mbar_arrive(&full[sl]);   // every lane: releases its own stores
        }
    };

    if (warp == W)
        epilogue();
    else
        compute();
}

}  // namespace mbglu
