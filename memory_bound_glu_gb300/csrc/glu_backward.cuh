// glu_backward.cuh -- the backward of the dual-weight GLU GEMV.
//
// DeepSpeed PR #8602, comment "Plan B: Dual-Weight GEMV -- Investigation
// Results & Implementation", section "Plan B Design: kernel adapts to the
// weights": the autograd wrapper works on the model's own weight tensors, so
// their gradients land on those tensors; "Verification Results" checks them
// against the composite.  For out = SiLU(g) * u with g = h Wg^T and
// u = h Wu^T, and an upstream gradient dout:
//
//   dG = dout * u * SiLU'(g)        dU = dout * SiLU(g)            [M][N]
//   grad_h    = dG Wg + dU Wu                                      [M][K]
//   grad_gate = dG^T h,  grad_up = dU^T h                          [N][K]
//
// The path for aligned operands, two passes over the weights:
//   1. the forward kernels with the backward epilogue (glu_store with
//      kModeBwd) recompute g and u and write dG, dU in fp32;
//   2. one pass that reads each weight block once for grad_h's partials and
//      writes both weight gradients: glu_bwd_mma_kernel on the tensor cores
//      (M = 3..16; dG and dU enter as three exact bf16 terms) or
//      glu_bwd_hw_kernel on the CUDA cores (M <= 2); glu_bwd_h_reduce8_kernel
//      then adds the partials in order and rounds grad_h once.
// Batches above 16 rows and unaligned operands take three steps instead:
// step 1 per 16-row block; grad_h by glu_bwd_rows_kernel (passes of 8 rows)
// or glu_bwd_h_kernel with glu_bwd_h_reduce_kernel; the weight gradients by
// glu_bwd_w_rows_kernel or glu_bwd_w_kernel.
// Every sum runs in a fixed order: results are bitwise deterministic.
#pragma once

#include "glu_kernels.cuh"

namespace mbglu {

struct BwdParams {
    const uint16_t *h;
    int64_t ldh;
    const uint16_t *gate;
    int64_t ld_gate;
    const uint16_t *up;
    int64_t ld_up;
    const float *dG, *dU;   // [M][N], row stride N
    float *part;            // grad_h partials [nsplit][M][K]
    uint16_t *grad_h;
    int64_t ldgh;
    uint16_t *grad_gate;
    int64_t ldgg;
    uint16_t *grad_up;
    int64_t ldgu;
    int M, N, K;
    int ldm;                // row stride of dG, dU (N; the rows kernel's block offset applies to the pointers)
    int R, S;               // glu_bwd_rows_kernel: rows per stage, stages in the ring
    uint32_t off_ring;      // glu_bwd_rows_kernel: ring offset in dynamic shared memory
    int rows_cta;           // glu_bwd_rows_kernel, glu_bwd_hw_kernel: largest row share of a CTA
    int col_groups;         // glu_bwd_hw_kernel, glu_bwd_mma_kernel: CTAs sharing a row share (each a group of column slices)
    int rows_pad;           // glu_bwd_mma_kernel: rows_cta rounded up to a multiple of 16
    uint32_t off_nm;           // glu_bwd_mma_kernel: staged dG, dU
    int vec_w;              // gate, up rows 8-byte aligned: 4-element loads
    int vec_out;            // grad_gate, grad_up rows and h 16-byte aligned, K % 8 == 0: 8-element access
    int h_smem;             // glu_bwd_w_kernel: h staged in shared memory
};

constexpr int kBwdCols = 512;        // glu_bwd_h_kernel: columns per CTA, 4 per thread
constexpr int kBwdRowChunk = 256;    // glu_bwd_h_kernel: rows of dG, dU staged at a time
constexpr int kBwdMaxSplits = 48;    // glu_bwd_h_kernel: row splits of N (partials in the workspace)

// 4 consecutive bf16 of a weight row as fp32 (zeros past the row's end)
__device__ __forceinline__ void load4_bf16(const uint16_t *ptr, bool vec, int left, float (&v)[4])
{
    if (vec) {
        const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(ptr));
        v[0] = bf16_lo(w.x);
        v[1] = bf16_hi(w.x);
        v[2] = bf16_lo(w.y);
        v[3] = bf16_hi(w.y);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = i < left ? bf16_to_f32(ptr[i]) : 0.0f;
    }
}

// grad_h partials.  blockIdx.x: 512 columns, 4 per thread (threads 0..127
// take rows n0, n0+2, ..., threads 128..255 rows n0+1, n0+3, ...);
// blockIdx.y: rows [n0, n1) of N.  part[y][m][k] = the two halves' sums of
// dG[m][n] Wg[n][k] + dU[m][n] Wu[n][k], added half 0 + half 1.
template <int MB>
__global__ void __launch_bounds__(256) glu_bwd_h_kernel(const BwdParams q)
{
    extern __shared__ __align__(16) float bwd_s[];   // [2][M][kBwdRowChunk]; then [MB * 4][128]
    const int nb = blockIdx.y, nsplit = gridDim.y;
    const int n0 = static_cast<int>((static_cast<int64_t>(q.N) * nb) / nsplit);
    const int n1 = static_cast<int>((static_cast<int64_t>(q.N) * (nb + 1)) / nsplit);
    const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
    const int k = blockIdx.x * kBwdCols + 4 * c;
    const bool vec = q.vec_w && k + 4 <= q.K;
    float *dg_s = bwd_s, *du_s = bwd_s + q.M * kBwdRowChunk;

    float acc[MB][4];
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.0f;

    for (int c0 = n0; c0 < n1; c0 += kBwdRowChunk) {
        const int rows = min(kBwdRowChunk, n1 - c0);
        __syncthreads();   // the previous chunk's reads are done
        for (int m = 0; m < q.M; ++m)
            for (int j = threadIdx.x; j < rows; j += blockDim.x) {
                dg_s[m * kBwdRowChunk + j] = q.dG[static_cast<int64_t>(m) * q.N + c0 + j];
                du_s[m * kBwdRowChunk + j] = q.dU[static_cast<int64_t>(m) * q.N + c0 + j];
            }
        __syncthreads();
        if (k < q.K) {
#pragma unroll 4
            for (int j = half; j < rows; j += 2) {
                const int64_t n = c0 + j;
                float wg[4], wu[4];
                load4_bf16(q.gate + n * q.ld_gate + k, vec, q.K - k, wg);
                load4_bf16(q.up + n * q.ld_up + k, vec, q.K - k, wu);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    if (m < q.M) {
                        const float a = dg_s[m * kBwdRowChunk + j], b = du_s[m * kBwdRowChunk + j];
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[m][i] = fmaf(b, wu[i], fmaf(a, wg[i], acc[m][i]));
                    }
                }
            }
        }
    }
    __syncthreads();   // dG, dU no longer read: the same shared memory combines the halves
    float *red = bwd_s;
    if (half == 1) {
#pragma unroll
        for (int m = 0; m < MB; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[(m * 4 + i) * 128 + c] = acc[m][i];
    }
    __syncthreads();
    if (half == 0 && k < q.K) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            if (m < q.M) {
                float *dst = q.part + (static_cast<int64_t>(nb) * q.M + m) * q.K + k;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (k + i < q.K) dst[i] = acc[m][i] + red[(m * 4 + i) * 128 + c];
            }
        }
    }
}

// grad_h partials by whole rows: the main path (operands 16-byte aligned,
// K % 8 == 0).  CTA b owns a balanced share [n0, n1) of the N rows of both
// weights and every column; thread t owns the 8-column chunks t, t + T, ...
// (CPT of them, T = blockDim.x <= 512).  The share streams through a ring of
// S stages of R rows each (gate rows, then up rows; one bulk copy per matrix
// and stage when the rows are contiguous), LAST rows first: the first step
// read this share in rising order and left its tail in L2 (evict-last), so
// much of it is read back from there.  For each row n (descending), thread t
// adds dG[m][n] Wg[n][k] + dU[m][n] Wu[n][k] into its fp32 accumulators,
// m < M <= MB.  part[b][m][k] receives the CTA's sums;
// glu_bwd_h_reduce_kernel adds the CTAs in order.  The share's dG and dU are
// staged in shared memory after the dependency wait; the first S stages of
// weights are requested before it.
// Dynamic shared memory: [0, 256) stage barriers, [256, off_ring) dG and dU
// of the share ([2][MB][rows_cta] fp32), [off_ring, ...) the ring.
constexpr int kBwdRowsThreads = 512;   // glu_bwd_rows_kernel: most threads per CTA

template <int MB, int CPT>
__global__ void __launch_bounds__(kBwdRowsThreads, 1) glu_bwd_rows_kernel(const BwdParams q)
{
    extern __shared__ __align__(128) unsigned char bwd_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(bwd_smem);
    float *dg_s = reinterpret_cast<float *>(bwd_smem + 256);
    float *du_s = dg_s + MB * q.rows_cta;
    uint16_t *ring = reinterpret_cast<uint16_t *>(bwd_smem + q.off_ring);
    const int b = blockIdx.x, G = gridDim.x, K = q.K, R = q.R, S = q.S;
    const int n0 = static_cast<int>((static_cast<int64_t>(q.N) * b) / G);
    const int n1 = static_cast<int>((static_cast<int64_t>(q.N) * (b + 1)) / G);
    const int rows = n1 - n0, nblk = (rows + R - 1) / R;
    const int64_t stage_elems = static_cast<int64_t>(2) * R * K;
    const bool contig = q.ld_gate == K && q.ld_up == K;
    const uint64_t policy = l2_policy_evict_first();

    // block j: rows [lo, hi) with hi = n1 - j R
    auto fill = [&](int j) {
        const int hi = n1 - j * R, lo = max(n0, hi - R), nr = hi - lo;
        const int st = j % S;
        uint16_t *dst = ring + st * stage_elems;
        const uint32_t bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(K) * 2u;
        mbar_arrive_expect_tx(&full[st], 2u * bytes);
        if (contig) {
            bulk_g2s(dst, q.gate + static_cast<int64_t>(lo) * K, bytes, &full[st], policy);
            bulk_g2s(dst + static_cast<int64_t>(R) * K, q.up + static_cast<int64_t>(lo) * K, bytes, &full[st], policy);
        } else {
            for (int i = 0; i < nr; ++i) {
                bulk_g2s(dst + static_cast<int64_t>(i) * K, q.gate + (lo + i) * q.ld_gate, K * 2u, &full[st], policy);
                bulk_g2s(dst + static_cast<int64_t>(R + i) * K, q.up + (lo + i) * q.ld_up, K * 2u, &full[st],
                         policy);
            }
        }
    };

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int j = 0; j < min(S, nblk); ++j) fill(j);   // weights only: before the dependency wait
    grid_dependency_wait();                                 // dG, dU of the first step
    for (int i = threadIdx.x; i < q.M * rows; i += blockDim.x) {
        const int m = i / rows, r = i - m * rows;
        dg_s[m * q.rows_cta + r] = q.dG[static_cast<int64_t>(m) * q.ldm + n0 + r];
        du_s[m * q.rows_cta + r] = q.dU[static_cast<int64_t>(m) * q.ldm + n0 + r];
    }
    __syncthreads();

    float2 acc[CPT][MB][4];
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc)
#pragma unroll
        for (int m = 0; m < MB; ++m)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[cc][m][k] = make_float2(0.0f, 0.0f);

    for (int j = 0; j < nblk; ++j) {
        const int st = j % S;
        const uint32_t phase = static_cast<uint32_t>(j / S) & 1u;
        if (!mbar_wait_bounded(&full[st], phase, kWaitLimitNs)) {
            atomicExch(&g_device_error, kErrTimeout);
            mbar_wait_bounded(&full[st], phase, kWaitLimitNs);
        }
        const int hi = n1 - j * R, lo = max(n0, hi - R);
        const uint16_t *gs = ring + st * stage_elems;
        const uint16_t *us = gs + static_cast<int64_t>(R) * K;
        for (int i = hi - lo - 1; i >= 0; --i) {   // descending rows
            const int r = lo - n0 + i;
            float2 a2[MB], b2[MB];
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                const float a = m < q.M ? dg_s[m * q.rows_cta + r] : 0.0f;
                const float bb = m < q.M ? du_s[m * q.rows_cta + r] : 0.0f;
                a2[m] = make_float2(a, a);
                b2[m] = make_float2(bb, bb);
            }
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                const int col = 8 * (threadIdx.x + cc * blockDim.x);
                if (col < K) {
                    const uint4 g4 = *reinterpret_cast<const uint4 *>(gs + static_cast<int64_t>(i) * K + col);
                    const uint4 u4 = *reinterpret_cast<const uint4 *>(us + static_cast<int64_t>(i) * K + col);
                    const float2 gv[4] = {make_float2(bf16_lo(g4.x), bf16_hi(g4.x)),
                                          make_float2(bf16_lo(g4.y), bf16_hi(g4.y)),
                                          make_float2(bf16_lo(g4.z), bf16_hi(g4.z)),
                                          make_float2(bf16_lo(g4.w), bf16_hi(g4.w))};
                    const float2 uv[4] = {make_float2(bf16_lo(u4.x), bf16_hi(u4.x)),
                                          make_float2(bf16_lo(u4.y), bf16_hi(u4.y)),
                                          make_float2(bf16_lo(u4.z), bf16_hi(u4.z)),
                                          make_float2(bf16_lo(u4.w), bf16_hi(u4.w))};
#pragma unroll
                    for (int m = 0; m < MB; ++m)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            acc[cc][m][k] = __ffma2_rn(b2[m], uv[k], __ffma2_rn(a2[m], gv[k], acc[cc][m][k]));
                }
            }
        }
        __syncthreads();   // every thread is done with stage st
        if (threadIdx.x == 0 && j + S < nblk) {
            fence_proxy_async_smem();
            fill(j + S);
        }
    }
    grid_launch_dependents();
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
        const int col = 8 * (threadIdx.x + cc * blockDim.x);
        if (col >= K) continue;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            if (m < q.M) {
                float4 *dst = reinterpret_cast<float4 *>(q.part + (static_cast<int64_t>(b) * q.M + m) * K + col);
                dst[0] = make_float4(acc[cc][m][0].x, acc[cc][m][0].y, acc[cc][m][1].x, acc[cc][m][1].y);
                dst[1] = make_float4(acc[cc][m][2].x, acc[cc][m][2].y, acc[cc][m][3].x, acc[cc][m][3].y);
            }
        }
    }
}

// Steps 2 and 3 of the backward in one pass over the rows (M <= MB <= 8,
// operands 16-byte aligned with row strides of whole chunks, K % 8 == 0):
// CTA (s, c) owns a balanced share [n0, n1) of the N rows and a group of
// Wc 256-column slices; warp w of the CTA owns one slice and lane l its
// 8 columns k.  Each warp streams the share's rows of both weights for its
// slice through its own ring of S stages (one TMA box of R rows x 256
// columns per matrix and stage), LAST rows first -- the first step read the
// share in rising order and left its tail in L2 -- with no CTA-wide barrier
// in the loop.  For each row n, lane l
//   * adds dG[m][n] Wg[n][k] + dU[m][n] Wu[n][k] into its fp32 grad_h
//     partials (m < M), and
//   * writes grad_gate[n][k] = bf16(sum_m dG[m][n] h[m][k]) and grad_up
//     likewise (m in order), 16-byte streaming stores, h kept unpacked in
//     registers.
// So the weights are read once here and every gradient element is written
// once.  part[s][m][k] receives the share's grad_h sums;
// glu_bwd_h_reduce8_kernel adds the shares in order.  The share's dG and dU
// are staged in shared memory after the dependency wait; the first stages of
// weights are requested before it.
// Dynamic shared memory: [0, 256) barriers [warp][stage], [256, off_ring)
// dG and dU ([2][MB][rows_cta] fp32), [off_ring, ...) ring[warp][stage]
// [2][R][256] bf16.
constexpr int kBwdSlice = 256;   // columns per warp: one TMA box row (512 bytes)

struct BwdMaps {
    TensorMap gate, up;   // [N][K] bf16, box 256 x R, no swizzle
};

// the most warps (column slices) per CTA at batch tile MB: the registers of
// 32 * warps threads (~190 each at MB = 8) must fit the SM's 65536
__host__ __device__ constexpr int bwd_hw_warps(int MB) { return MB >= 8 ? 10 : MB >= 4 ? 14 : 16; }

template <int MB>
__global__ void __launch_bounds__(32 * bwd_hw_warps(MB), 1) glu_bwd_hw_kernel(const BwdParams q,
                                                                            const __grid_constant__ BwdMaps maps)
{
    extern __shared__ __align__(128) unsigned char hw_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = q.S, R = q.R;
    uint64_t *bars = reinterpret_cast<uint64_t *>(hw_smem) + warp * S;
    float *dg_s = reinterpret_cast<float *>(hw_smem + 256);
    float *du_s = dg_s + MB * q.rows_cta;
    const uint32_t stage_bytes = 2u * static_cast<uint32_t>(R) * kBwdSlice * 2u;
    unsigned char *ring = hw_smem + q.off_ring + static_cast<uint32_t>(warp) * S * stage_bytes;
    const int G = gridDim.x / q.col_groups;
    const int share = blockIdx.x / q.col_groups, cgrp = blockIdx.x - share * q.col_groups;
    const int n0 = static_cast<int>((static_cast<int64_t>(q.N) * share) / G);
    const int n1 = static_cast<int>((static_cast<int64_t>(q.N) * (share + 1)) / G);
    const int rows = n1 - n0, nblk = (rows + R - 1) / R;
    const int x0 = (cgrp * static_cast<int>(blockDim.x >> 5) + warp) * kBwdSlice;   // the warp's first column
    const int col = x0 + 8 * lane;
    const bool active = x0 < q.K && col < q.K;
    const uint64_t policy = l2_policy_evict_first();

    // block j: rows [lo, hi) with hi = n1 - j R; the box starts at lo
    auto fill = [&](int j) {
        const int hi = n1 - j * R, lo = max(n0, hi - R);
        const int st = j % S;
        unsigned char *dst = ring + st * stage_bytes;
        mbar_arrive_expect_tx(&bars[st], stage_bytes);
        tma_load_2d(dst, &maps.gate, x0, lo, &bars[st], policy);
        tma_load_2d(dst + stage_bytes / 2, &maps.up, x0, lo, &bars[st], policy);
    };

    if (lane == 0 && x0 < q.K) {
        for (int st = 0; st < S; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0 && x0 < q.K)
        for (int j = 0; j < min(S, nblk); ++j) fill(j);   // weights only: before the dependency wait
    grid_dependency_wait();                                 // dG, dU of the first step
    for (int i = threadIdx.x; i < q.M * rows; i += blockDim.x) {
        const int m = i / rows, r = i - m * rows;
        dg_s[m * q.rows_cta + r] = q.dG[static_cast<int64_t>(m) * q.ldm + n0 + r];
        du_s[m * q.rows_cta + r] = q.dU[static_cast<int64_t>(m) * q.ldm + n0 + r];
    }
    float2 hf[MB][4];   // h's 8 columns of this lane, unpacked once
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        const uint4 v = (m < q.M && active) ? *reinterpret_cast<const uint4 *>(q.h + m * q.ldh + col)
                                            : make_uint4(0, 0, 0, 0);
        hf[m][0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
        hf[m][1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
        hf[m][2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
        hf[m][3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
    }
    __syncthreads();   // dG, dU staged
    if (x0 >= q.K) return;   // a slice past K (the last column group): no rows to stream

    float2 acc[MB][4];
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[m][k] = make_float2(0.0f, 0.0f);

    for (int j = 0; j < nblk; ++j) {
        const int st = j % S;
        const uint32_t phase = static_cast<uint32_t>(j / S) & 1u;
        if (!mbar_wait_bounded(&bars[st], phase, kWaitLimitNs)) {
            if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
            mbar_wait_bounded(&bars[st], phase, kWaitLimitNs);
        }
        const int hi = n1 - j * R, lo = max(n0, hi - R);
        const uint16_t *gs = reinterpret_cast<const uint16_t *>(ring + st * stage_bytes);
        const uint16_t *us = gs + R * kBwdSlice;
        if (active) {
            for (int i = hi - lo - 1; i >= 0; --i) {   // descending rows
                const int r = lo - n0 + i;
                const int64_t n = lo + i;
                const uint4 g4 = *reinterpret_cast<const uint4 *>(gs + i * kBwdSlice + 8 * lane);
                const uint4 u4 = *reinterpret_cast<const uint4 *>(us + i * kBwdSlice + 8 * lane);
                const float2 gv[4] = {make_float2(bf16_lo(g4.x), bf16_hi(g4.x)), make_float2(bf16_lo(g4.y), bf16_hi(g4.y)),
                                      make_float2(bf16_lo(g4.z), bf16_hi(g4.z)), make_float2(bf16_lo(g4.w), bf16_hi(g4.w))};
                const float2 uv[4] = {make_float2(bf16_lo(u4.x), bf16_hi(u4.x)), make_float2(bf16_lo(u4.y), bf16_hi(u4.y)),
                                      make_float2(bf16_lo(u4.z), bf16_hi(u4.z)), make_float2(bf16_lo(u4.w), bf16_hi(u4.w))};
                float2 sg[4], su[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) sg[k] = su[k] = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    // rows m >= M of the tile are padding: their dG, dU are not staged
                    const float a = m < q.M ? dg_s[m * q.rows_cta + r] : 0.0f;
                    const float bb = m < q.M ? du_s[m * q.rows_cta + r] : 0.0f;
                    const float2 a2 = make_float2(a, a), b2 = make_float2(bb, bb);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        acc[m][k] = __ffma2_rn(b2, uv[k], __ffma2_rn(a2, gv[k], acc[m][k]));
                        sg[k] = __ffma2_rn(a2, hf[m][k], sg[k]);
                        su[k] = __ffma2_rn(b2, hf[m][k], su[k]);
                    }
                }
                __stcs(reinterpret_cast<uint4 *>(q.grad_gate + n * q.ldgg + col),
                       make_uint4(pack_bf16x2(sg[0].x, sg[0].y), pack_bf16x2(sg[1].x, sg[1].y),
                                  pack_bf16x2(sg[2].x, sg[2].y), pack_bf16x2(sg[3].x, sg[3].y)));
                __stcs(reinterpret_cast<uint4 *>(q.grad_up + n * q.ldgu + col),
                       make_uint4(pack_bf16x2(su[0].x, su[0].y), pack_bf16x2(su[1].x, su[1].y),
                                  pack_bf16x2(su[2].x, su[2].y), pack_bf16x2(su[3].x, su[3].y)));
            }
        }
        __syncwarp();
        if (lane == 0 && j + S < nblk) {
            fence_proxy_async_smem();
            fill(j + S);
        }
        __syncwarp();
    }
    grid_launch_dependents();
    if (active) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            if (m < q.M) {
                float4 *dst = reinterpret_cast<float4 *>(q.part + (static_cast<int64_t>(share) * q.M + m) * q.K + col);
                dst[0] = make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
                dst[1] = make_float4(acc[m][2].x, acc[m][2].y, acc[m][3].x, acc[m][3].y);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Steps 2 and 3 on the tensor cores (glu_bwd_mma_kernel, M = 3..16)
// ---------------------------------------------------------------------------
// The pass of glu_bwd_hw_kernel with both contractions as bf16 MMAs
// (mma.sync, fp32 accumulators):
//   grad_h^T[k][m] += sum_n W[n][k] dG[m][n]    A = W^T from the stage, B = dG
//   grad_W[n][k]    = sum_m dG[m][n] h[m][k]    A = dG^T,               B = h
// dG and dU are fp32 and the MMA multiplies bf16, so each value x enters as
// three bf16 terms: hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid)
// (each difference exact in fp32).  bf16 keeps 8 of fp32's 24 significant
// bits, so the three terms hold x exactly (unless lo falls below bf16's
// normal range), and a product of two bf16 values is exact in fp32: the MMAs
// see the same products as fp32 arithmetic would.  The batch is padded to a
// tile of MB = 8 or 16 rows with zero rows.
//   * grad_h takes one m16n8k16 per term and 8-row batch tile.
//   * grad_W lays the terms along the MMA's reduction.  At MB = 8 that is
//     [hi m0..7 | mid m0..7] against [h; h] (m16n8k16) and lo m0..7 against
//     h (m16n8k8); at MB = 16, one m16n8k16 per term over m0..15.
//
// A CTA owns a row share [n0, n1) and a group of column slices.  Its rows go
// in blocks of 16, block b = [n0 + 16 b, n0 + 16 b + 16), the LAST block
// first (the first step read the share in rising order and left its tail in
// L2).  A block's tensor copy may run past n1 into the next share, or past N
// where it reads zeros: those rows meet dG = dU = 0 (the staging is
// zero-padded) and their weight gradients are not stored.  Warp w of column
// group c owns the columns [x0, x0 + 64 NB), x0 = (c W + w) 64 NB, as NB
// boxes of 64 columns x 16 rows per matrix and stage, 128-byte swizzled:
// 16-byte chunk j of row r sits at r * 128 + ((j ^ (r & 7)) << 4), so the
// transposed matrix loads of a column pair meet no bank conflict.  The
// weight gradients need no weights, so a stage goes back to the copy engine
// as soon as grad_h has read it.  In grad_W's MMAs, column j of tile t
// (t = 4 p + t') stands for weight column 32 p + 8 (j / 2) + 2 t' + j % 2 of
// the warp's slice: over the four tiles of a group, lane (g, c) then holds
// 8 consecutive columns of rows g and g + 8, stored as one 16-byte piece
// each.  part[s][m][k] receives the share's grad_h sums;
// glu_bwd_h_reduce8_kernel adds the shares in order.
//
// dG and dU are staged once, as [matrix][rows_pad][PITCH] bf16: row n holds
// hi for m = 0..MB-1, then mid, then lo (PITCH = 24 at MB = 8, 48 + 8 of
// padding at MB = 16, so that 8 rows of a matrix load fall in 8 different
// bank groups).  grad_W reads it as its A operand (ldmatrix); grad_h reads it
// transposed (ldmatrix.trans) as its B operand.
//
// Shared memory (dynamic, from a 1024-byte aligned base):
//   [0, 512)                   mbarriers [warp][stage]
//   [off_nm, + 4 PITCH rp)     dG, dU as above (rp = rows_pad)
//   [off_ring, ...)            ring [warp][stage][matrix][NB][16][64] bf16
// at most 12 warps at MB = 8 (160 registers a thread leave room for 3 warps
// on each of the SM's four register files), 8 at MB = 16 (twice the grad_h
// accumulators and h fragments)
__host__ __device__ constexpr int bwd_mma_warps(int NB, int MB = 8) { return MB > 8 ? 8 : NB >= 4 ? 8 : 12; }
__host__ __device__ constexpr int bwd_mma_pitch(int MB) { return MB > 8 ? 56 : 24; }
constexpr uint32_t kBwdMmaBox = 16u * 128u;   // one 64-column x 16-row box, bytes

// x = hi + mid + lo, each bf16 (exact for normal x down to 2^-110 or so);
// mid = lo = 0 when hi is not finite
__device__ __forceinline__ void split3_bf16(float x, uint16_t (&t)[3])
{
    t[0] = f32_to_bf16(x);
    const float h = bf16_to_f32(t[0]);
    if (!isfinite(h)) {
        t[1] = t[2] = 0;
        return;
    }
    const float r = x - h;
    t[1] = f32_to_bf16(r);
    t[2] = f32_to_bf16(r - bf16_to_f32(t[1]));
}

// One 16-row x 64-column piece of a weight gradient (two groups of four
// tiles), rounded to bf16 and stored.  MB = 8: D = [hi | mid]^T [h; h] + lo^T h
// (a, a8); MB = 16: D = hi^T h + mid^T h + lo^T h (aw[0..2]).  hb: the B
// fragments (h[2c][k], h[2c+1][k][, h[8+2c][k], h[8+2c+1][k]]) of the tiles'
// permuted columns from tile t0; dst: row g of the piece's first column; nr
// valid rows, kleft columns left in the row.
template <int MB, int NH>
__device__ __forceinline__ void bwd_mma_w_tile(const uint32_t (&aw)[3][4], const uint32_t (&hb)[NH][2], int t0,
                                               uint16_t *dst, int64_t ld, int nr, int kleft, int lane)
{
    float d[8][4];
    if constexpr (MB > 8) {
#pragma unroll
        for (int t = 0; t < 8; ++t) mma16_bf16_z(d[t], aw[0], hb[t0 + t][0], hb[t0 + t][1]);
#pragma unroll
        for (int t = 0; t < 8; ++t) mma16_bf16(d[t], aw[1], hb[t0 + t][0], hb[t0 + t][1]);
#pragma unroll
        for (int t = 0; t < 8; ++t) mma16_bf16(d[t], aw[2], hb[t0 + t][0], hb[t0 + t][1]);
    } else {
        const uint32_t a8[2] = {aw[2][0], aw[2][1]};
#pragma unroll
        for (int t = 0; t < 8; ++t) mma16_bf16_z(d[t], aw[0], hb[t0 + t][0], hb[t0 + t][0]);
#pragma unroll
        for (int t = 0; t < 8; ++t) mma8_bf16(d[t], a8, hb[t0 + t][0]);
    }
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int col = 32 * p + 8 * c;
        if (col >= kleft) continue;
        const int t = 4 * p;
        if (g < nr)
            __stcs(reinterpret_cast<uint4 *>(dst + col),
                   make_uint4(pack_bf16x2(d[t][0], d[t][1]), pack_bf16x2(d[t + 1][0], d[t + 1][1]),
                              pack_bf16x2(d[t + 2][0], d[t + 2][1]), pack_bf16x2(d[t + 3][0], d[t + 3][1])));
        if (g + 8 < nr)
            __stcs(reinterpret_cast<uint4 *>(dst + 8 * ld + col),
                   make_uint4(pack_bf16x2(d[t][2], d[t][3]), pack_bf16x2(d[t + 1][2], d[t + 1][3]),
                              pack_bf16x2(d[t + 2][2], d[t + 2][3]), pack_bf16x2(d[t + 3][2], d[t + 3][3])));
    }
}

template <int NB, int MB>
__global__ void __launch_bounds__(32 * bwd_mma_warps(NB, MB), 1) glu_bwd_mma_kernel(const BwdParams q,
                                                                                  const __grid_constant__ BwdMaps maps)
{
    static_assert(MB == 8 || MB == 16, "batch tile of 8 or 16 rows");
    constexpr int NT = MB / 8;                    // 8-row batch tiles (grad_h's n8 tiles)
    constexpr int PITCH = bwd_mma_pitch(MB);      // staged row, elements
    constexpr int NC = 3 * NT;                    // (term, batch tile) chunks of a staged row
    extern __shared__ __align__(128) unsigned char bm_raw[];
    unsigned char *sm = bm_raw + ((1024u - (smem_addr(bm_raw) & 1023u)) & 1023u);
    constexpr uint32_t kMat = NB * kBwdMmaBox;   // one matrix's part of a stage
    constexpr uint32_t kStage = 2 * kMat;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = static_cast<int>(blockDim.x >> 5), S = q.S;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm) + warp * S;
    unsigned char *ring = sm + q.off_ring + static_cast<uint32_t>(warp) * S * kStage;
    const uint32_t ring_a = smem_addr(ring);
    const uint32_t nm = smem_addr(sm + q.off_nm);
    const int rp = q.rows_pad;
    const uint32_t mat_bytes = static_cast<uint32_t>(rp) * PITCH * 2u;   // one matrix's staged rows
    const int G = gridDim.x / q.col_groups;
    const int share = blockIdx.x / q.col_groups, cgrp = blockIdx.x - share * q.col_groups;
    const int n0 = static_cast<int>((static_cast<int64_t>(q.N) * share) / G);
    const int n1 = static_cast<int>((static_cast<int64_t>(q.N) * (share + 1)) / G);
    const int rows = n1 - n0, nblk = (rows + 15) >> 4;
    const int x0 = (cgrp * W + warp) * (64 * NB);   // the warp's first column
    const bool live = x0 < q.K;
    const uint64_t policy = l2_policy_evict_first();

    // the j-th block in order, block nblk - 1 - j, into stage j % S
    auto fill = [&](int j) {
        const int y = n0 + 16 * (nblk - 1 - j);
        const int st = j % S;
        unsigned char *dst = ring + st * kStage;
        mbar_arrive_expect_tx(&bars[st], kStage);
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            tma_load_2d(dst + i * kBwdMmaBox, &maps.gate, x0 + 64 * i, y, &bars[st], policy);
            tma_load_2d(dst + kMat + i * kBwdMmaBox, &maps.up, x0 + 64 * i, y, &bars[st], policy);
        }
    };

    if (lane == 0 && live) {
        for (int st = 0; st < S; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0 && live)
        for (int j = 0; j < min(S, nblk); ++j) fill(j);   // weights only: before the dependency wait
    grid_dependency_wait();                                 // dG, dU of the first step

    {   // dG, dU of the share as three bf16 terms, zero past the share and past M
        uint16_t *nmp = reinterpret_cast<uint16_t *>(sm + q.off_nm);
        for (int i = threadIdx.x; i < MB * rp; i += blockDim.x) {
            const int m = i / rp, r = i - m * rp;
            float x[2] = {0.0f, 0.0f};
            if (m < q.M && r < rows) {
                x[0] = q.dG[static_cast<int64_t>(m) * q.ldm + n0 + r];
                x[1] = q.dU[static_cast<int64_t>(m) * q.ldm + n0 + r];
            }
#pragma unroll
            for (int mat = 0; mat < 2; ++mat) {
                uint16_t t[3];
                split3_bf16(x[mat], t);
#pragma unroll
                for (int e = 0; e < 3; ++e) nmp[(mat * rp + r) * PITCH + e * MB + m] = t[e];
            }
        }
    }
    // B fragments of grad_W: hb[t] = (h[2c][k], h[2c+1][k]) [and (h[8+2c][k], h[8+2c+1][k])] with k the
    // weight column of MMA column g in tile t = 4 p + t'
    const int g4 = lane >> 2, c4 = lane & 3;
    uint32_t hb[8 * NB][2];
#pragma unroll
    for (int t = 0; t < 8 * NB; ++t) {
        const int k = x0 + 32 * (t >> 2) + 8 * (g4 >> 1) + 2 * (t & 3) + (g4 & 1);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t lo = 0, hi = 0;
            const int m = 2 * c4 + 8 * half;
            if (half < NT && k < q.K) {
                if (m < q.M) lo = q.h[static_cast<int64_t>(m) * q.ldh + k];
                if (m + 1 < q.M) hi = q.h[static_cast<int64_t>(m + 1) * q.ldh + k];
            }
            hb[t][half] = lo | (hi << 16);
        }
    }
    __syncthreads();   // dG, dU staged
    if (!live) return;   // a slice past K (the last column group): no rows to stream

    float acc[NT][4 * NB][4];
#pragma unroll
    for (int mt = 0; mt < NT; ++mt)
#pragma unroll
        for (int i = 0; i < 4 * NB; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][i][e] = 0.0f;

    const int mi = lane >> 3, ri = lane & 7;
    for (int j = 0; j < nblk; ++j) {
        const int st = j % S;
        const uint32_t phase = static_cast<uint32_t>(j / S) & 1u;
        if (!mbar_wait_bounded(&bars[st], phase, kWaitLimitNs)) {
            if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
            mbar_wait_bounded(&bars[st], phase, kWaitLimitNs);
        }
        const int nb0 = 16 * (nblk - 1 - j);   // the block's first row in the share
        const int nr = min(16, rows - nb0);
        const uint32_t sg = ring_a + st * kStage, su = sg + kMat;
        {   // grad_h: the stage's weights, as W^T by transposed matrix loads.  B:
            // dG, dU at the block's rows, per (term, batch tile) chunk: rows n 0-7
            // then 8-15 of the staged layout, transposed
            uint32_t bh[2][NC][2];
#pragma unroll
            for (int mat = 0; mat < 2; ++mat) {
#pragma unroll
                for (int c0 = 0; c0 < NC; c0 += 2) {
                    const int ch = min(c0 + (mi >> 1), NC - 1);   // the x4 past the last chunk repeats it
                    const uint32_t addr = nm + mat * mat_bytes +
                                          static_cast<uint32_t>((nb0 + 8 * (mi & 1) + ri) * PITCH * 2 + ch * 16);
                    uint32_t r[4];
                    ldsm_x4_trans(r, addr);
                    bh[mat][c0][0] = r[0];
                    bh[mat][c0][1] = r[1];
                    if (c0 + 1 < NC) {
                        bh[mat][c0 + 1][0] = r[2];
                        bh[mat][c0 + 1][1] = r[3];
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                // the box's four 16-column groups, their MMAs interleaved chunk by chunk
#pragma unroll
                for (int mat = 0; mat < 2; ++mat) {
                    uint32_t a[4][4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int n = ri + 8 * (mi >> 1), chunk = 2 * q4 + (mi & 1);
                        ldsm_x4_trans(a[q4], (mat ? su : sg) +
                                                 static_cast<uint32_t>(i * kBwdMmaBox + n * 128 + ((chunk ^ ri) << 4)));
                    }
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            mma16_bf16(acc[c % NT][4 * i + q4], a[q4], bh[mat][c][0], bh[mat][c][1]);
                }
            }
        }
        // the weight gradients need no weights: the stage goes back to the
        // copy engine now, and its next block streams in meanwhile
        __syncwarp();
        if (lane == 0 && j + S < nblk) {
            fence_proxy_async_smem();
            fill(j + S);
        }
        {   // grad_W's A: rows nb0 .. nb0 + 15, per term (MB = 16) or [hi | mid], lo (MB = 8)
            uint32_t ag[3][4], au[3][4];
            const int n = nb0 + ri + 8 * (mi & 1);
#pragma unroll
            for (int mat = 0; mat < 2; ++mat) {
                uint32_t(&aw)[3][4] = mat ? au : ag;
                const uint32_t row = nm + mat * mat_bytes + static_cast<uint32_t>(n * PITCH * 2);
                if constexpr (MB > 8) {
#pragma unroll
                    for (int e = 0; e < 3; ++e) ldsm_x4(aw[e], row + static_cast<uint32_t>((2 * e + (mi >> 1)) << 4));
                } else {
                    uint32_t a8[2];
                    ldsm_x4(aw[0], row + static_cast<uint32_t>((mi >> 1) << 4));
                    ldsm_x2(a8, row + 32u);
                    aw[2][0] = a8[0];
                    aw[2][1] = a8[1];
                }
            }
            const int64_t nrow = static_cast<int64_t>(n0) + nb0 + g4;   // row g of the block
#pragma unroll
            for (int i = 0; i < NB; ++i) {   // grad_gate, grad_up: the box's 16 x 64 pieces
                const int col = x0 + 64 * i;
                bwd_mma_w_tile<MB>(ag, hb, 8 * i, q.grad_gate + nrow * q.ldgg + col, q.ldgg, nr, q.K - col, lane);
                bwd_mma_w_tile<MB>(au, hb, 8 * i, q.grad_up + nrow * q.ldgu + col, q.ldgu, nr, q.K - col, lane);
            }
        }
    }
    grid_launch_dependents();
    // acc[mt][gq]: D[k][m] with k = x0 + 16 gq + g (+8), m = 8 mt + 2c (+1)
#pragma unroll
    for (int mt = 0; mt < NT; ++mt)
#pragma unroll
        for (int gq = 0; gq < 4 * NB; ++gq) {
            const int k = x0 + 16 * gq + g4;
            const int m = 8 * mt + 2 * c4;
            float *p0 = q.part + (static_cast<int64_t>(share) * q.M + m) * q.K;
            if (m < q.M) {
                if (k < q.K) p0[k] = acc[mt][gq][0];
                if (k + 8 < q.K) p0[k + 8] = acc[mt][gq][2];
            }
            if (m + 1 < q.M) {
                if (k < q.K) p0[q.K + k] = acc[mt][gq][1];
                if (k + 8 < q.K) p0[q.K + k + 8] = acc[mt][gq][3];
            }
        }
}

// grad_h[m][k] = bf16( part[0][m][k] + part[1][m][k] + ... ), splits in order
__global__ void __launch_bounds__(256) glu_bwd_h_reduce_kernel(const BwdParams q, int nsplit)
{
    const int64_t total = static_cast<int64_t>(q.M) * q.K;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / q.K, k = i - m * q.K;
        float s = q.part[i];
        for (int b = 1; b < nsplit; ++b) s += q.part[static_cast<int64_t>(b) * total + i];
        q.grad_h[m * q.ldgh + k] = f32_to_bf16(s);
    }
}

// grad_h[m][8c .. 8c+7] = bf16( the sum of the nsplit partials ), the main
// path (K % 8 == 0): one warp per (row m, 8-column chunk c); lane l adds
// partials l, l + 32, ... in order, then a fixed butterfly adds the lanes.
__global__ void __launch_bounds__(256) glu_bwd_h_reduce8_kernel(const BwdParams q, int nsplit, int vec_store)
{
    const int lane = threadIdx.x & 31;
    const int chunks = q.K >> 3;
    const int64_t nwarp = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t total = static_cast<int64_t>(q.M) * chunks;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
         w += nwarp) {
        const int m = static_cast<int>(w / chunks), c = static_cast<int>(w - static_cast<int64_t>(m) * chunks);
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int64_t pstride = static_cast<int64_t>(q.M) * q.K;   // between consecutive partials
        const float *base = q.part + static_cast<int64_t>(m) * q.K + 8 * c;
        for (int b0 = lane; b0 < nsplit; b0 += 32 * 4) {
            // up to four partials of this lane in flight at once, added in order
            float4 x[4], y[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int b = b0 + 32 * t;
                if (b < nsplit) {
                    const float4 *src = reinterpret_cast<const float4 *>(base + b * pstride);
                    x[t] = src[0];
                    y[t] = src[1];
                } else {
                    x[t] = y[t] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                v[0] += x[t].x;
                v[1] += x[t].y;
                v[2] += x[t].z;
                v[3] += x[t].w;
                v[4] += y[t].x;
                v[5] += y[t].y;
                v[6] += y[t].z;
                v[7] += y[t].w;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], off);
        if (lane == 0) {
            uint16_t *dst = q.grad_h + static_cast<int64_t>(m) * q.ldgh + 8 * c;
            if (vec_store) {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                             pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = f32_to_bf16(v[i]);
            }
        }
    }
}

// grad_gate[n][k] = bf16( sum_m dG[m][n] h[m][k] ), grad_up likewise with dU,
// the m-sum in order m = 0, 1, ...: the main path at M <= MB <= 8 (K % 8 ==
// 0, gradients and h 16-byte aligned with row strides of whole chunks).  CTA
// b owns a balanced share [n0, n1) of the rows; thread t owns the 8-column
// chunks t, t + T, ... (CPT of them) and keeps h's columns there in
// registers; the share's dG and dU are staged in shared memory.  Each row's
// two gradient rows are written once, with streaming stores.
template <int MB, int CPT>
__global__ void __launch_bounds__(kBwdRowsThreads, 1) glu_bwd_w_rows_kernel(const BwdParams q)
{
    extern __shared__ __align__(16) float wdg_s[];   // [2][MB][rows_cta]
    float *du_s = wdg_s + MB * q.rows_cta;
    const int b = blockIdx.x, G = gridDim.x, K = q.K;
    const int n0 = static_cast<int>((static_cast<int64_t>(q.N) * b) / G);
    const int n1 = static_cast<int>((static_cast<int64_t>(q.N) * (b + 1)) / G);
    const int rows = n1 - n0;
    grid_dependency_wait();
    for (int i = threadIdx.x; i < q.M * rows; i += blockDim.x) {
        const int m = i / rows, r = i - m * rows;
        wdg_s[m * q.rows_cta + r] = q.dG[static_cast<int64_t>(m) * q.ldm + n0 + r];
        du_s[m * q.rows_cta + r] = q.dU[static_cast<int64_t>(m) * q.ldm + n0 + r];
    }
    float2 hf[CPT][MB][4];   // h's columns of this thread, unpacked once
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
        const int col = 8 * (threadIdx.x + cc * blockDim.x);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const uint4 v = (m < q.M && col < K) ? *reinterpret_cast<const uint4 *>(q.h + m * q.ldh + col)
                                                 : make_uint4(0, 0, 0, 0);
            hf[cc][m][0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
            hf[cc][m][1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
            hf[cc][m][2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
            hf[cc][m][3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
        }
    }
    __syncthreads();
    grid_launch_dependents();
    for (int r = 0; r < rows; ++r) {
        const int64_t n = n0 + r;
        float a[MB], bb[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            a[m] = m < q.M ? wdg_s[m * q.rows_cta + r] : 0.0f;
            bb[m] = m < q.M ? du_s[m * q.rows_cta + r] : 0.0f;
        }
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) {
            const int col = 8 * (threadIdx.x + cc * blockDim.x);
            if (col >= K) continue;
            float2 sg[4], su[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) sg[j] = su[j] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                const float2 a2 = make_float2(a[m], a[m]), b2 = make_float2(bb[m], bb[m]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sg[j] = __ffma2_rn(a2, hf[cc][m][j], sg[j]);
                    su[j] = __ffma2_rn(b2, hf[cc][m][j], su[j]);
                }
            }
            __stcs(reinterpret_cast<uint4 *>(q.grad_gate + n * q.ldgg + col),
                   make_uint4(pack_bf16x2(sg[0].x, sg[0].y), pack_bf16x2(sg[1].x, sg[1].y),
                              pack_bf16x2(sg[2].x, sg[2].y), pack_bf16x2(sg[3].x, sg[3].y)));
            __stcs(reinterpret_cast<uint4 *>(q.grad_up + n * q.ldgu + col),
                   make_uint4(pack_bf16x2(su[0].x, su[0].y), pack_bf16x2(su[1].x, su[1].y),
                              pack_bf16x2(su[2].x, su[2].y), pack_bf16x2(su[3].x, su[3].y)));
        }
    }
}

// 8 consecutive bf16 as fp32 (zeros past `left`)
__device__ __forceinline__ void load8_bf16(const uint16_t *ptr, bool vec, int left, float (&v)[8])
{
    if (vec) {
        const uint4 w = *reinterpret_cast<const uint4 *>(ptr);
        v[0] = bf16_lo(w.x);
        v[1] = bf16_hi(w.x);
        v[2] = bf16_lo(w.y);
        v[3] = bf16_hi(w.y);
        v[4] = bf16_lo(w.z);
        v[5] = bf16_hi(w.z);
        v[6] = bf16_lo(w.w);
        v[7] = bf16_hi(w.w);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = i < left ? bf16_to_f32(ptr[i]) : 0.0f;
    }
}

__device__ __forceinline__ void store8_bf16(uint16_t *ptr, bool vec, int left, const float (&v)[8])
{
    if (vec) {
        __stcs(reinterpret_cast<uint4 *>(ptr), make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                          pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7])));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < left) ptr[i] = f32_to_bf16(v[i]);
    }
}

// grad_gate[n][k] = bf16( sum_m dG[m][n] h[m][k] ), grad_up likewise with dU;
// the m-sum in order m = 0, 1, ... .  Rows n are dealt over the CTAs, 8
// columns per thread.
template <int MB>
__global__ void __launch_bounds__(256) glu_bwd_w_kernel(const BwdParams q)
{
    extern __shared__ __align__(16) uint16_t hw_s[];   // h [M][K], row stride K (h_smem)
    const uint16_t *hb = q.h;
    int64_t hld = q.ldh;
    if (q.h_smem) {
        for (int m = 0; m < q.M; ++m)
            for (int k = threadIdx.x; k < q.K; k += blockDim.x)
                hw_s[static_cast<int64_t>(m) * q.K + k] = q.h[m * q.ldh + k];
        __syncthreads();
        hb = hw_s;
        hld = q.K;
    }
    for (int64_t n = blockIdx.x; n < q.N; n += gridDim.x) {
        float a[MB], b[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            a[m] = m < q.M ? q.dG[static_cast<int64_t>(m) * q.N + n] : 0.0f;
            b[m] = m < q.M ? q.dU[static_cast<int64_t>(m) * q.N + n] : 0.0f;
        }
        for (int k = 8 * threadIdx.x; k < q.K; k += 8 * blockDim.x) {
            const bool vec = q.vec_out && k + 8 <= q.K;
            float sg[8], su[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) sg[i] = su[i] = 0.0f;
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                if (m < q.M) {
                    float hv[8];
                    load8_bf16(hb + m * hld + k, vec, q.K - k, hv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        sg[i] = fmaf(a[m], hv[i], sg[i]);
                        su[i] = fmaf(b[m], hv[i], su[i]);
                    }
                }
            }
            store8_bf16(q.grad_gate + n * q.ldgg + k, vec, q.K - k, sg);
            store8_bf16(q.grad_up + n * q.ldgu + k, vec, q.K - k, su);
        }
    }
}

}  // namespace mbglu
