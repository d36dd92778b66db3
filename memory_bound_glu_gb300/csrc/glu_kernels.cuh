// glu_kernels.cuh -- sm_103a kernels of the dual-weight GLU GEMV.
//
//   out[m,n] = SiLU(g[m,n]) * u[m,n],  g = h . W_gate[n],  u = h . W_up[n]
//
// DeepSpeed PR #8602, comment "Plan B: Dual-Weight GEMV", section "Plan B
// Design: kernel adapts to the weights": both nn.Linear weights are read in
// place, fp32 accumulation, SiLU(gate) * up with one round-to-nearest-even at
// the end.  Section "Why cuBLAS-level performance is achievable at b=1": each
// weight element takes part in exactly one product, so the op is bound by the
// bytes it streams, and the design target is the HBM roofline.
//
// GB300 design (the pages' warp-per-row Ada kernel with scalar loads is prior
// art only):
//   * one persistent CTA per SM, a balanced contiguous range of rows each;
//   * every warp owns a private ring of shared-memory stages filled with
//     asynchronous copies (mbarrier completion, L2 evict-first hint): one
//     stage holds a group of rows of BOTH matrices;
//   * with programmatic dependent launch the first stages are requested
//     before waiting on the preceding kernel, so consecutive calls overlap
//     one call's tail with the next call's ramp;
//   * every wait is bounded (globaltimer); a timeout records an error word and
//     returns instead of hanging or trapping.
// The K-slice tensor-core kernel, which takes batch 1-16 where its plan fits
// (the headline shape among them), is in glu_slice.cuh.  Kernels in this file:
//   glu_stream_kernel   batch 1-2 past the K-slice kernel's reach, CUDA cores:
//                       1-D bulk copies of whole rows, h in registers at
//                       batch 1, packed fp32x2 FMAs and a warp butterfly;
//                       optional add + RMSNorm prologue;
//   glu_mma_kernel      batch 3-16 past the K-slice kernel's reach, tensor
//                       cores (mma.sync m16n8k16): one TMA box per matrix per
//                       stage, static per-warp unit ranges with exact
//                       accumulator hand-off, h staged in up to two K-phases;
//                       optional add + RMSNorm prologue;
//   glu_generic_kernel  any 2-byte-aligned operands (the correctness path);
//   residual_add_kernel, zero_fill_kernel, silu_mul_kernel,
//   gdn_gates_chunk_kernel, gdn_gates_kernel.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mbglu {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait
constexpr int kErrTimeout = 8;                    // == MBGLU_ERR_TIMEOUT
constexpr int kMaxWarps = 16;        // any kernel's block, for the norm reduction
constexpr int kMaxStreamWarps = 8;   // the streaming kernels' block, a helper warp included
constexpr int kMaxM = 16;

// Error word of the device (read and cleared by mbglu_read_device_error).
__device__ int g_device_error;

struct GluParams {
    const uint16_t *h;
    int64_t ldh;
    const uint16_t *gate;
    int64_t ld_gate;
    const uint16_t *up;
    int64_t ld_up;
    uint16_t *out;
    int64_t ldo;
    const uint16_t *s;       // norm prologue: updated residual rows [M][K], contiguous
    const uint16_t *norm_w;  // norm prologue: [K]
    float eps;
    int M, N, K, mode;
    int KS, nseg, stages;    // streaming kernel: segment length, #segments, ring depth
    uint32_t off_h, off_ring;
    uint32_t off_piece;      // tensor-core kernel: handed-off accumulators, [warp][16][32] fp32
    uint32_t off_carry;      // tensor-core kernel, nphase > 1: accumulators between phases, [group][16][32] fp32
    int nphase, nsp;         // tensor-core kernel: K staged through h_s in nphase phases of nsp segments
    int tma;                 // tensor-core kernel: whole 8-row groups arrive as one tensor copy per matrix
    int vec_in;              // 1: h (or s, norm_w) may be read with 16-byte loads
    int prefetch;            // 1: first weight stages requested before the dependency wait
    int interleave;          // 1: this CTA's row groups are blockIdx.x, +gridDim.x, ... of all groups
    // single-kernel add_rmsnorm_glu (fused != 0): s = bf16(x + residual) is formed in
    // shared memory at off_s, and the last CTA to arrive on *ws writes it to residual
    int fused;
    const uint16_t *x;
    uint16_t *residual;
    int *ws;                 // arrival counters, 0 between calls
    uint32_t off_s;
    int helper_warp;         // single-kernel path: the extra warp that writes the residual slice (-1: none)
    // backward (mode == kModeBwd): the epilogue reads dout and writes the
    // fp32 gradients of g and u, [M][N] with row stride N, instead of out
    const uint16_t *dout;
    int64_t ldd;
    float *dG, *dU;
};

constexpr int kModeBwd = 2;   // internal mode of the forward kernels: the backward's dG, dU epilogue

// ---------------------------------------------------------------------------
// scalar helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float round_to_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
// two floats rounded to nearest-even bf16 in one paired conversion
// (cvt.rn.bf16x2.f32), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// SiLU(x) = x / (1 + e^-x) = x * e^x / (1 + e^x), evaluated with t = e^-|x| so
// that nothing overflows: for x < -88.7 the first form's e^-x is +inf in fp32
// and would flush SiLU to -0, although x * e^x is still a normal bf16 value
// down to x ~ -92 (bf16 keeps fp32's exponent range).  Precise expf and IEEE
// division (no fast math).
__device__ __forceinline__ float silu_f32(float x)
{
    const float t = expf(-fabsf(x));
    return (x >= 0.0f ? x : x * t) / (1.0f + t);
}

// mode 0 (FUSED): one rounding.  mode 1 (HF): the bf16 composite's roundings:
// g, u, SiLU(g) and the product each round to bf16 (PR #9057, section
// "Changes").  sb * ub is exact in fp32.
__device__ __forceinline__ uint16_t glu_epilogue(float g, float u, int mode)
{
    if (mode == 0) return f32_to_bf16(silu_f32(g) * u);
    const float gb = round_to_bf16(g);
    const float ub = round_to_bf16(u);
    const float sb = round_to_bf16(silu_f32(gb));
    return f32_to_bf16(sb * ub);
}

// SiLU(x) and SiLU'(x) = sigma(x) * (1 + x * (1 - sigma(x))), from t = e^-|x|
// so that nothing overflows: sigma = 1/(1+t), 1 - sigma = t/(1+t) for x >= 0,
// and the two swapped below.  Precise expf and IEEE division.
__device__ __forceinline__ void silu_and_derivative(float x, float &silu, float &dsilu)
{
    const float t = expf(-fabsf(x));
    const float sig = (x >= 0.0f ? 1.0f : t) / (1.0f + t);
    const float rest = (x >= 0.0f ? t : 1.0f) / (1.0f + t);   // 1 - sigma
    silu = x * sig;
    dsilu = sig * (1.0f + x * rest);
}

// The store of one output of the GEMV kernels.  Forward modes: out = the GLU
// epilogue.  kModeBwd ([8602/PlanB] autograd wrapper: the gradients of
// SiLU(g) * u): dG = dout * u * SiLU'(g), dU = dout * SiLU(g), in fp32.
__device__ __forceinline__ void glu_store(const GluParams &p, int m, int64_t n, float g, float u)
{
    if (p.mode == kModeBwd) {
        const float d = bf16_to_f32(p.dout[m * p.ldd + n]);
        float sl, ds;
        silu_and_derivative(g, sl, ds);
        p.dG[static_cast<int64_t>(m) * p.N + n] = (d * u) * ds;
        p.dU[static_cast<int64_t>(m) * p.N + n] = d * sl;
    } else {
        p.out[m * p.ldo + n] = glu_epilogue(g, u, p.mode);
    }
}

__device__ __forceinline__ float warp_allsum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// The normed row, correctly rounded: h = bf16( s * (mean_k s^2 + eps)^-1/2 *
// (1 + w) ) is the bf16 value nearest to the exact real number.  A plain
// fp32 chain (sum, sqrt, two products: a few fp32 ulps in all) rounds h to
// the other bf16 neighbour wherever the exact value lies that close to a
// midpoint -- about 3e-5 of the elements -- and in HF mode one such element
// of a row shifts g and u of every output of that row enough to re-round a
// few percent of them.  So:
//   * the statistic is summed in double-float (a pair of fp32 words whose sum
//     carries the value), each s^2 (exact in fp32) added with Knuth's
//     error-free TwoSum, the thread partials combined the same way;
//   * (var + eps)^-1/2 starts from rsqrtf and takes one Newton step,
//     y (1 + e/2) with e = 1 - v y^2 formed with exact products (FMA), to
//     about 2^-44 relative, kept as inv_hi + inv_lo;
//   * each element is formed in fp32 first; if it lies within 8 fp32 ulps
//     of a bf16 midpoint (the fp32 chain's error is at most 5) it is formed
//     again in double-float (Dekker's exact products) and rounded from that.
// The statistic is exact up to ~2^-46 and the element up to ~2^-44, so h is
// the correctly rounded value except where the exact value lies within
// ~2^-44 relative of a midpoint.  Every path computes the same h.
// ---------------------------------------------------------------------------

// s = fl(a + b), e = (a + b) - s exactly (TwoSum; the _rn intrinsics keep
// the compiler from contracting or reordering it)
__device__ __forceinline__ float two_sum(float a, float b, float &e)
{
    const float s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
    return s;
}

__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }

// A thread's sum of squares as two packed double-float accumulators (the
// even and the odd elements of its chunks).
struct SumSq {
    float2 hi, lo;
};

__device__ __forceinline__ SumSq sumsq_zero()
{
    SumSq a;
    a.hi = a.lo = make_float2(0.0f, 0.0f);
    return a;
}

// acc += x (x exact), TwoSum on both packed lanes
__device__ __forceinline__ void sumsq_add(SumSq &acc, float2 x)
{
    const float2 t = __fadd2_rn(acc.hi, x);
    const float2 bp = __fadd2_rn(t, neg2(acc.hi));
    const float2 e = __fadd2_rn(__fadd2_rn(acc.hi, neg2(__fadd2_rn(t, neg2(bp)))), __fadd2_rn(x, neg2(bp)));
    acc.lo = __fadd2_rn(acc.lo, e);
    acc.hi = t;
}

// the squares of 8 bf16 (exact in fp32) into four independent accumulators
// (one per 32-bit word: four short dependency chains instead of one long)
__device__ __forceinline__ void sumsq_bf16x8(uint4 v, SumSq (&acc)[4])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 a = make_float2(bf16_lo(w[j]), bf16_hi(w[j]));
        sumsq_add(acc[j], __fmul2_rn(a, a));
    }
}

// (hi, lo) of a thread's accumulators: hi the fp32 sum of the high words
// (TwoSum, errors kept), lo every remaining part (small against hi)
__device__ __forceinline__ float2 sumsq_total(const SumSq (&a)[4])
{
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float e;
        hi = two_sum(hi, a[j].hi.x, e);
        lo = __fadd_rn(lo, __fadd_rn(e, a[j].lo.x));
        hi = two_sum(hi, a[j].hi.y, e);
        lo = __fadd_rn(lo, __fadd_rn(e, a[j].lo.y));
    }
    return make_float2(hi, lo);
}

// (hi, lo) += (bhi, blo), renormalised so that |lo| <= ulp(hi) / 2 (for
// non-negative sums, where the error of hi + bhi is far below the sum)
__device__ __forceinline__ void df_add(float &hi, float &lo, float bhi, float blo)
{
    float e;
    const float t = two_sum(hi, bhi, e);
    e = __fadd_rn(e, __fadd_rn(lo, blo));
    hi = __fadd_rn(t, e);
    lo = __fsub_rn(e, __fsub_rn(hi, t));
}

// the butterfly of a double-float over the warp: every lane gets the same sum
__device__ __forceinline__ void df_warp_allsum(float &hi, float &lo)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, off);
        const float ol = __shfl_xor_sync(0xffffffffu, lo, off);
        df_add(hi, lo, oh, ol);
    }
}

// (inv_hi, inv_lo) = (S / K + eps)^-1/2 for the row's sum of squares S = hi + lo
__device__ __forceinline__ float2 norm_inv(float hi, float lo, int K, float eps)
{
    const float kf = static_cast<float>(K);
    const float q = __fdiv_rn(hi, kf);
    const float rem = __fmaf_rn(-q, kf, hi);                  // hi - q K, exact
    float vh = q, vl = __fdiv_rn(__fadd_rn(rem, lo), kf);
    df_add(vh, vl, eps, 0.0f);
    const float y = rsqrtf(vh);
    const float y2 = __fmul_rn(y, y);
    const float y2l = __fmaf_rn(y, y, -y2);                   // y^2 = y2 + y2l exactly
    const float t = __fmul_rn(vh, y2);
    const float tl = __fmaf_rn(vl, y2, __fmaf_rn(vh, y2l, __fmaf_rn(vh, y2, -t)));
    const float e = __fsub_rn(__fsub_rn(1.0f, t), tl);       // 1 - v y^2; 1 - t is exact (t near 1)
    const float c = __fmul_rn(__fmul_rn(0.5f, y), e);
    const float ih = __fadd_rn(y, c);
    return make_float2(ih, __fsub_rn(c, __fsub_rn(ih, y)));
}

// one element of h from s, w and the row's (inv_hi, inv_lo), in double-float
__device__ __forceinline__ uint16_t norm_elem_df(float sv, float w, float ih, float il)
{
    float al;
    const float ah = two_sum(1.0f, w, al);                    // 1 + w = ah + al exactly
    const float ph = __fmul_rn(sv, ih);
    const float pl = __fmaf_rn(sv, il, __fmaf_rn(sv, ih, -ph));
    const float qh = __fmul_rn(ph, ah);
    const float ql = __fmaf_rn(ph, al, __fmaf_rn(pl, ah, __fmaf_rn(ph, ah, -qh)));
    const float t = __fadd_rn(qh, ql);
    const float l = __fsub_rn(ql, __fsub_rn(t, qh));
    const uint32_t b = __float_as_uint(t);
    if ((b & 0xffffu) == 0x8000u && l != 0.0f) {
        // t sits on a bf16 midpoint and the exact value lies past it on l's side
        const bool away = (l > 0.0f) == (t > 0.0f);
        return static_cast<uint16_t>((b >> 16) + (away ? 1u : 0u));
    }
    return f32_to_bf16(t);
}

// the element in fp32: (s * inv_hi) * (1 + w)
__device__ __forceinline__ float norm_elem_f32(float sv, float w, float ih)
{
    return __fmul_rn(__fmul_rn(sv, ih), __fadd_rn(1.0f, w));
}

// true if the fp32 element lies within 8 fp32 ulps of a bf16 midpoint (the
// fp32 chain is off by at most 5): only then can its rounding be wrong
__device__ __forceinline__ bool near_midpoint(float v) { return ((__float_as_uint(v) + 8u) & 0xfff0u) == 0x8000u; }

__device__ __forceinline__ uint16_t norm_elem(float sv, float w, float ih, float il)
{
    const float v = norm_elem_f32(sv, w, ih);
    return near_midpoint(v) ? norm_elem_df(sv, w, ih, il) : f32_to_bf16(v);
}

// 8 elements of h from 8 of s and of w (bf16 pairs) in fp32; `near` is set
// if any of them needs the double-float evaluation (norm_fix_rows)
__device__ __forceinline__ uint4 norm_chunk_f32(uint4 v, uint4 w, float ih, bool &near)
{
    const uint32_t sv[4] = {v.x, v.y, v.z, v.w};
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = norm_elem_f32(bf16_lo(sv[j]), bf16_lo(ww[j]), ih);
        const float hi = norm_elem_f32(bf16_hi(sv[j]), bf16_hi(ww[j]), ih);
        near |= near_midpoint(lo) | near_midpoint(hi);
        o[j] = pack_bf16x2(lo, hi);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// The rare second pass of a thread one of whose chunks holds an element near
// a bf16 midpoint: the chunks c0 + i P with bit i of `mask` set still hold s
// (the fast pass left them alone) and are formed again element by element.
// Out of line, so that the hot loop stays small: every CTA fetches that code
// once per launch, and instruction-cache misses set the prologue's pace.
__device__ __noinline__ void norm_fix_chunks(uint4 *row, const uint4 *w_row, int c0, int P, uint64_t mask, float ih,
                                             float il)
{
    while (mask) {
        const int i = __ffsll(static_cast<long long>(mask)) - 1;
        mask &= mask - 1;
        const int c = c0 + i * P;
        const uint4 v = row[c], w = w_row[c];
        const uint32_t sv[4] = {v.x, v.y, v.z, v.w};
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
        for (int j = 0; j < 4; ++j)
            o[j] = static_cast<uint32_t>(norm_elem(bf16_lo(sv[j]), bf16_lo(ww[j]), ih, il)) |
                   (static_cast<uint32_t>(norm_elem(bf16_hi(sv[j]), bf16_hi(ww[j]), ih, il)) << 16);
        row[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------------------------------
// prologues: h into shared memory
// ---------------------------------------------------------------------------

// Copies h[M][K] (row stride ldh) to h_s[MB][K]; rows M..MB-1 become zero.
template <int MB>
__device__ __forceinline__ void load_h_to_smem(const GluParams &p, uint16_t *h_s)
{
    const int K = p.K;
    if (p.vec_in) {
        const int nch = K >> 3;
        for (int i = threadIdx.x; i < MB * nch; i += blockDim.x) {
            const int m = i / nch, c = i - m * nch;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m < p.M) v = *reinterpret_cast<const uint4 *>(p.h + m * p.ldh + c * 8);
            *reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(m) * K + c * 8) = v;
        }
    } else {
        for (int i = threadIdx.x; i < MB * K; i += blockDim.x) {
            const int m = i / K, k = i - m * K;
            h_s[i] = (m < p.M) ? p.h[m * p.ldh + k] : static_cast<uint16_t>(0);
        }
    }
}

// Zero-centred RMSNorm of the updated residual rows for the generic kernel
// (PR #9057 "Changes"): var = mean_k s^2, inv = (var + eps)^-1/2,
// h = bf16( s * inv * (1 + w) ), correctly rounded (see norm_elem); 2-byte
// accesses, any alignment.  Every CTA runs the same code on the same data, so
// every CTA gets the same h -- the same h as the streaming kernels' prologue.
// red: [kMaxWarps][MB] shared double-floats; inv_s: [2 MB].  Writes
// rows_out rows of h_s (rows M..rows_out-1 zero, row stride K); M <= MB.
// s: the residual rows in global memory (p.s, row stride K).
template <int MB>
__device__ __forceinline__ void norm_prologue(const GluParams &p, uint16_t *h_s, float2 (*red)[MB],
                                              float *inv_s, int rows_out)
{
    const uint16_t *sp = p.s;
    const uint16_t *wp = p.norm_w;
    const int K = p.K, tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    float hi[MB], lo[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) hi[m] = lo[m] = 0.0f;
    for (int k = tid; k < K; k += nthr) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            if (m < p.M) {
                const float a = bf16_to_f32(sp[static_cast<int64_t>(m) * K + k]);
                float e;
                hi[m] = two_sum(hi[m], __fmul_rn(a, a), e);
                lo[m] = __fadd_rn(lo[m], e);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        df_warp_allsum(hi[m], lo[m]);
        if (lane == 0) red[warp][m] = make_float2(hi[m], lo[m]);
    }
    __syncthreads();
    if (tid < p.M) {
        float th = 0.0f, tl = 0.0f;
        for (int w = 0; w < nw; ++w) df_add(th, tl, red[w][tid].x, red[w][tid].y);
        const float2 inv = norm_inv(th, tl, K, p.eps);
        inv_s[2 * tid] = inv.x;
        inv_s[2 * tid + 1] = inv.y;
    }
    __syncthreads();
    for (int i = tid; i < rows_out * K; i += nthr) {
        const int m = i / K, k = i - m * K;
        uint16_t o = 0;
        if (m < p.M)
            o = norm_elem(bf16_to_f32(sp[static_cast<int64_t>(m) * K + k]), bf16_to_f32(wp[k]), inv_s[2 * m],
                          inv_s[2 * m + 1]);
        h_s[static_cast<int64_t>(m) * K + k] = o;
    }
}

// Prologue operands (h; residual; x) arrive by bulk copies on their own
// mbarrier (kProBarOffset), issued by thread 0 after the dependency wait:
// one copy when the rows are contiguous on both sides, else one per row.
constexpr uint32_t kProBarOffset = 784;

__device__ __forceinline__ void copy_rows_async(uint16_t *dst, int dstride, const uint16_t *src, int64_t ld,
                                                int rows, int K, uint64_t *bar)
{
    if (ld == K && dstride == K) {
        bulk_g2s_plain(dst, src, static_cast<uint32_t>(rows) * static_cast<uint32_t>(K) * 2u, bar);
    } else {
        for (int r = 0; r < rows; ++r)
            bulk_g2s_plain(dst + static_cast<int64_t>(r) * dstride, src + r * ld, static_cast<uint32_t>(K) * 2u, bar);
    }
}

// All threads: bounded wait for the prologue copies (phase 0).  A timeout is
// recorded; the kernel then waits once more (bounded) so that no copy is
// still writing shared memory when it goes on.
__device__ __forceinline__ void prologue_wait(uint64_t *bar)
{
    if (!mbar_wait_bounded(bar, 0u, kWaitLimitNs)) {
        atomicExch(&g_device_error, kErrTimeout);
        mbar_wait_bounded(bar, 0u, kWaitLimitNs);
    }
}

// Row-owned prologue of the streaming kernels (operands 16-byte aligned, the
// residual rows already copied into shared memory h_s).  The block's threads
// are split evenly over the M rows: thread t owns row m = t / P (P = blockDim
// / M threads per row) and its 16-byte chunks c = t % P + j * P.  A thread's
// row never changes, so its sum of squares is one register and no chunk
// needs a division; consecutive threads touch consecutive chunks of a row,
// so shared accesses are conflict-free for any row pitch and global loads of
// x are coalesced.  Measured on GB300 at M = 8, K = 2560: the earlier
// chunk-major loops (a division and 16 unrolled row slots per chunk) took
// 4.4 us for the statistic and the scale alone.
struct RowMap {
    int m, c0, P, nch;
    bool active;
};

__device__ __forceinline__ RowMap row_map(int M, int K)
{
    RowMap r;
    r.P = static_cast<int>(blockDim.x) / M;
    r.m = static_cast<int>(threadIdx.x) / r.P;
    r.c0 = static_cast<int>(threadIdx.x) - r.m * r.P;
    r.active = r.m < M;
    r.nch = K >> 3;
    return r;
}

__device__ __forceinline__ uint4 add_bf16x8(uint4 a, uint4 b)
{
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = pack_bf16x2(bf16_lo(aw[j]) + bf16_lo(bw[j]), bf16_hi(aw[j]) + bf16_hi(bw[j]));
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Single-kernel add_rmsnorm_glu: x is read straight from global memory, the
// first NX chunks of each thread before the residual copy is awaited (one
// round trip for M*K <= NX * blockDim * 8), the rest in batches of NX
// independent loads.  The prologue runs once per launch, so its code is
// fetched once per launch by each of the SM's schedulers: the kernels whose
// shares fit take the smaller batch, whose unrolled loop is half the code.
constexpr int kXRows = 16;
constexpr int kXRowsSmall = 8;

template <int NX>
struct XRowsN {
    uint4 v[NX];
};
using XRows = XRowsN<kXRows>;

template <int NX>
__device__ __forceinline__ void x_prefetch_rows(const GluParams &p, const RowMap &r, XRowsN<NX> &x, int j0 = 0)
{
    const uint4 *xrow = reinterpret_cast<const uint4 *>(p.x) + static_cast<int64_t>(r.m) * r.nch;
#pragma unroll
    for (int j = 0; j < NX; ++j) {
        const int c = r.c0 + (j0 + j) * r.P;
        x.v[j] = (r.active && c < r.nch) ? xrow[c] : make_uint4(0, 0, 0, 0);
    }
}

// s = bf16(x + residual) formed in place in h_s (the fp32 sum of two bf16
// values rounds to the same bf16 as the exact sum); returns this thread's sum
// of s^2 over its chunks as a double-float.  The statistic rides in the same
// loop, where it hides under the latency of the x loads.  The chunks are
// taken in the same order for every NX, so the sum does not depend on it.
template <int NX>
__device__ __forceinline__ float2 add_rows_in_place(const GluParams &p, const RowMap &r, uint16_t *h_s, int hstride,
                                                    XRowsN<NX> &x)
{
    SumSq ss[4] = {sumsq_zero(), sumsq_zero(), sumsq_zero(), sumsq_zero()};
    uint4 *row = reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(r.m) * hstride);
    for (int j0 = 0;; j0 += NX) {
        if (j0 > 0) x_prefetch_rows(p, r, x, j0);
#pragma unroll
        for (int j = 0; j < NX; ++j) {
            const int c = r.c0 + (j0 + j) * r.P;
            if (r.active && c < r.nch) {
                const uint4 sv = add_bf16x8(x.v[j], row[c]);
                row[c] = sv;
                sumsq_bf16x8(sv, ss);
            }
        }
        if (!r.active || r.c0 + (j0 + NX) * r.P >= r.nch) break;
    }
    return sumsq_total(ss);
}

// This thread's sum of s^2 over its chunks of h_s, in chunk order, as a
// double-float (the path whose s is already in shared memory).
__device__ __forceinline__ float2 square_rows(const RowMap &r, const uint16_t *h_s, int hstride)
{
    SumSq ss[4] = {sumsq_zero(), sumsq_zero(), sumsq_zero(), sumsq_zero()};
    if (!r.active) return make_float2(0.0f, 0.0f);
    const uint4 *row = reinterpret_cast<const uint4 *>(h_s + static_cast<int64_t>(r.m) * hstride);
#pragma unroll 2
    for (int c = r.c0; c < r.nch; c += r.P) sumsq_bf16x8(row[c], ss);
    return sumsq_total(ss);
}

// The norm's per-thread partial sums (high words, then low words, one pair
// per thread of the block): in dynamic shared memory after norm_w, whose
// region the planners size as round128(2 K) + kNormPartBytes.
constexpr uint32_t kNormPartBytes = 2u * (kMaxStreamWarps + 1) * 32u * 4u;

__device__ __forceinline__ float *norm_partials(unsigned char *smem, const GluParams &p)
{
    return reinterpret_cast<float *>(smem + p.off_s + ((static_cast<uint32_t>(p.K) * 2u + 127u) & ~127u));
}

// Zero-centred RMSNorm of the rows in h_s, in place (PR #9057 "Changes"):
//   var = mean_k s^2, inv = (var + eps)^-1/2, h = bf16( s * inv * (1 + w) ),
// with (1 + w) formed exactly and h correctly rounded (see norm_elem).
// ss: this thread's double-float partial from square_rows.  Row m's
// partials are added by one warp (lane-strided, then a butterfly), high words
// in double-float, low words alongside: a fixed order, and every CTA
// computes the identical h.  part: 2 blockDim floats of shared memory; inv_s:
// 2 M floats.  Rows M..rows_out-1 of h_s become zero.  Ends with a barrier.
__device__ __forceinline__ void norm_rows_in_place(const GluParams &p, const RowMap &r, float2 ss, uint16_t *h_s,
                                                   int hstride, const uint16_t *w_s, float *part, float *inv_s,
                                                   int rows_out)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int nthr = blockDim.x;
    part[tid] = ss.x;
    part[nthr + tid] = ss.y;
    __syncthreads();
    for (int m = warp; m < p.M; m += nw) {
        float hi = 0.0f, lo = 0.0f;
        for (int i = lane; i < r.P; i += 32) {
            float e;
            hi = two_sum(hi, part[m * r.P + i], e);
            lo = __fadd_rn(lo, __fadd_rn(e, part[nthr + m * r.P + i]));
        }
        df_warp_allsum(hi, lo);
        if (lane == 0) {
            const float2 inv = norm_inv(hi, lo, p.K, p.eps);
            inv_s[2 * m] = inv.x;
            inv_s[2 * m + 1] = inv.y;
        }
    }
    __syncthreads();
    if (r.active) {
        const float ih = inv_s[2 * r.m], il = inv_s[2 * r.m + 1];
        uint4 *row = reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(r.m) * hstride);
        const uint4 *wv = reinterpret_cast<const uint4 *>(w_s);
        uint64_t mask = 0;   // this thread's chunks left as s for norm_fix_chunks (at most 40 of them)
        int i = 0;
        // not unrolled: eight independent elements per chunk already overlap, and the loop
        // stays a few instruction-cache lines (each scheduler fetches it once per launch)
#pragma unroll 1
        for (int c = r.c0; c < r.nch; c += r.P, ++i) {
            bool near = false;
            const uint4 hv = norm_chunk_f32(row[c], wv[c], ih, near);
            if (near)
                mask |= 1ull << i;
            else
                row[c] = hv;
        }
        if (mask) norm_fix_chunks(row, wv, r.c0, r.P, mask, ih, il);
    }
    for (int i = tid; i < (rows_out - p.M) * r.nch; i += blockDim.x) {
        const int m = p.M + i / r.nch, c = i - (i / r.nch) * r.nch;
        *reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(m) * hstride + c * 8) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
}

// Part 2.  Workspace: ws[0] counts CTAs that hold their residual rows (the
// bulk copy has landed: that CTA reads residual no more), ws[1] counts CTAs
// that have written their share of the result.  Thread 0 arrives on ws[0]
// right after the copy lands.  At the end, warp 0 of every CTA waits (bounded)
// until all gridDim.x CTAs have arrived -- long true by then, since every CTA
// arrives early in its life and all of them are resident at once (grid <=
// one CTA per SM, and no dependent grid launches before all have started) --
// then writes its 1/gridDim.x slice of residual = bf16(x + residual) and
// arrives on ws[1]; the CTA arriving there last returns both counters to 0.
// The next call on the stream touches the counters only after its dependency
// wait, i.e. after this grid has completed.
__device__ __forceinline__ void fused_arrive(const GluParams &p)
{
    // the residual rows are already in shared memory: nothing to order before
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(p.ws) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *ptr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Warp 0: write this CTA's slice of residual and arrive on ws[1]; the CTA
// arriving there last returns both counters to 0.
__device__ __forceinline__ void fused_residual_slice(const GluParams &p)
{
    const int lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);
    const int n = p.M * (p.K >> 3);
    const int i0 = static_cast<int>((static_cast<int64_t>(n) * blockIdx.x) / G);
    const int i1 = static_cast<int>((static_cast<int64_t>(n) * (blockIdx.x + 1)) / G);
    for (int i = i0 + lane; i < i1; i += 32) {
        uint4 *rp = reinterpret_cast<uint4 *>(p.residual) + i;
        *rp = add_bf16x8(reinterpret_cast<const uint4 *>(p.x)[i], *rp);
    }
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        if (atomicAdd(p.ws + 1, 1) == G - 1) {
            atomicExch(p.ws, 0);
            atomicExch(p.ws + 1, 0);
        }
    }
}

// The helper warp (one extra warp that never streams): wait (bounded, with
// short sleeps) until every CTA has arrived, then write this CTA's slice.  It
// keeps the counter traffic and the slice's L2 round trips off the streaming
// warps.
__device__ __forceinline__ void fused_residual_helper(const GluParams &p)
{
    const int lane = threadIdx.x & 31;
    int ok = 1;
    if (lane == 0) {
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_gpu(p.ws) < static_cast<int>(gridDim.x)) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicExch(&g_device_error, kErrTimeout);
                ok = 0;
                break;
            }
            __nanosleep(256);
        }
    }
    if (__shfl_sync(0xffffffffu, ok, 0)) fused_residual_slice(p);
}

// ---------------------------------------------------------------------------
// the streaming kernel
// ---------------------------------------------------------------------------
//
// Work: this CTA owns rows [r0, r1) (a balanced contiguous share of N), cut
// into groups of R consecutive rows.  Warps claim groups from a shared-memory
// counter whenever they have a free stage, so every warp count stays
// balanced inside the CTA.  Each warp owns a private ring of S stages: a
// stage holds its group's rows of BOTH matrices, [R][KS] of W_gate then
// [R][KS] of W_up, and remembers which group it holds (slot_grp, -1 = none).
// A unit is (group, K-segment); the u-th unit a warp consumes sits in stage
// u % S with barrier phase (u / S) & 1 -- the ring is private and consumed in
// order, so a phase is never awaited twice.  When the rows are contiguous in
// memory (ld == K == KS) a group arrives in one bulk copy per matrix
// (R*K*2 bytes); otherwise one copy per row and matrix.
//
// Shared memory (dynamic):  [0, 512)          mbarriers [warp][stage]
//                           [512, 768)        slot_grp [warp][stage]
//                           [768, 772)        group counter
//                           [off_h, off_ring) h_s[MB][K] bf16 (not with HREG)
//                           [off_ring, ...)   ring[warp][stage][2][R][KS] bf16
//
// HREG (batch 1, K <= 4096): each lane keeps its slice of h -- chunks lane,
// lane+32, ... -- in registers, loaded by the warp itself after the
// dependency wait, so no CTA barrier sits between the wait and the first FMA.
//
// Ordering with the preceding grid (programmatic dependent launch):
//   prefetch == 1: the first S units of weights are requested BEFORE
//     griddepcontrol.wait -- weights are never written by this op, and the
//     launch policy that selects this promises the preceding kernel does
//     not write them either; h / the residual rows and `out` are touched
//     only after the wait.
//   prefetch == 0: nothing global is read before the wait.
// Dot products: exact bf16 x bf16 products, fp32 FMAs on (even, odd) element
// pairs (packed fp32x2 FMA), pairs added, then a warp butterfly.  Which warp
// computes a group does not change its arithmetic: results are bitwise
// deterministic.
constexpr int kHregChunks = 16;           // K <= 32 lanes * 16 chunks * 8 = 4096
constexpr uint32_t kSlotGrpOffset = 512;  // bytes
constexpr uint32_t kCounterOffset = 768;

template <int MB, int R, bool NORM, bool HREG>
__global__ void __launch_bounds__(kMaxStreamWarps * 32, 1) glu_stream_kernel(const GluParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float inv_s[2 * MB];                // norm: (inv_hi, inv_lo) per row

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages, KS = p.KS, K = p.K, nseg = p.nseg;
    const int64_t stage_elems = static_cast<int64_t>(2) * R * KS;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem) + warp * S;
    int *slot_grp = reinterpret_cast<int *>(smem + kSlotGrpOffset) + warp * S;
    int *counter = reinterpret_cast<int *>(smem + kCounterOffset);
    uint16_t *h_s = reinterpret_cast<uint16_t *>(smem + p.off_h);
    uint16_t *ring = reinterpret_cast<uint16_t *>(smem + p.off_ring) + static_cast<int64_t>(warp) * S * stage_elems;

    // Row groups of this CTA: a contiguous block [r0, r1) cut into groups of R
    // rows, or (interleave) the groups blockIdx.x, blockIdx.x + gridDim.x, ...
    // of the whole matrix.  group_row0(g) is the first row of local group g;
    // its rows end at min(row0 + R, rend).
    const int r0 = p.interleave ? 0 : static_cast<int>((static_cast<int64_t>(p.N) * blockIdx.x) / gridDim.x);
    const int r1 = p.interleave ? p.N : static_cast<int>((static_cast<int64_t>(p.N) * (blockIdx.x + 1)) / gridDim.x);
    const int all_groups = (p.N + R - 1) / R;
    const int ngroups = p.interleave
                            ? (all_groups > static_cast<int>(blockIdx.x)
                                   ? (all_groups - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                                   : 0)
                            : (r1 - r0 + R - 1) / R;
    auto group_row0 = [&](int g) -> int {
        return p.interleave ? (g * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x)) * R : r0 + g * R;
    };
    const bool contig = (p.ld_gate == K) && (p.ld_up == K) && (KS == K);

    uint64_t *pro_bar = reinterpret_cast<uint64_t *>(smem + kProBarOffset);
    const bool helper = warp == p.helper_warp;   // single-kernel norm path only; owns no ring
    if (lane == 0 && !helper)
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    if (threadIdx.x == 0) {
        *counter = 0;
        mbar_init(pro_bar, NORM ? 2 : 1);   // norm: the norm_w copy and the residual copy
    }
    fence_mbar_init();
    __syncthreads();

    // the backward's next step reads the weights again (last rows first):
    // keep them in L2 in that mode
    const uint64_t policy = p.mode == kModeBwd ? l2_policy_evict_last() : l2_policy_evict_first();
    // lane 0: request unit (group g, segment seg) into stage st
    auto issue = [&](int st, int g, int seg) {
        const int row0 = group_row0(g);
        const int nr = min(R, r1 - row0);
        const int k0 = seg * KS;
        const int len = min(KS, K - k0);
        const uint32_t row_bytes = static_cast<uint32_t>(len) * 2u;
        uint16_t *dg = ring + st * stage_elems;
        uint16_t *du = dg + R * KS;
        mbar_arrive_expect_tx(&bars[st], 2u * static_cast<uint32_t>(nr) * row_bytes);
        if (contig) {
            bulk_g2s(dg, p.gate + static_cast<int64_t>(row0) * K, static_cast<uint32_t>(nr) * row_bytes, &bars[st],
                     policy);
            bulk_g2s(du, p.up + static_cast<int64_t>(row0) * K, static_cast<uint32_t>(nr) * row_bytes, &bars[st],
                     policy);
        } else {
            for (int r = 0; r < nr; ++r) {
                bulk_g2s(dg + r * KS, p.gate + static_cast<int64_t>(row0 + r) * p.ld_gate + k0, row_bytes, &bars[st],
                         policy);
                bulk_g2s(du + r * KS, p.up + static_cast<int64_t>(row0 + r) * p.ld_up + k0, row_bytes, &bars[st],
                         policy);
            }
        }
    };
    // lane 0: the unit that follows (g, seg) in this warp's stream, claiming
    // a new group after the last segment; returns the group (-1: none left)
    // and updates seg.
    auto next_unit = [&](int g, int &seg) -> int {
        if (g >= 0 && seg + 1 < nseg) {
            ++seg;
            return g;
        }
        seg = 0;
        const int ng = atomicAdd(counter, 1);
        return ng < ngroups ? ng : -1;
    };
    // lane 0 state: the last unit requested
    int last_g = -1, last_seg = nseg;
    auto fill = [&](int st) {
        last_g = next_unit(last_g, last_seg);
        slot_grp[st] = last_g;
        if (last_g >= 0) issue(st, last_g, last_seg);
    };

    uint16_t *nw_s = reinterpret_cast<uint16_t *>(smem + p.off_s);   // norm: norm_w, K elements
    auto copy_norm_w = [&]() {
        if constexpr (NORM) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(K) * 2u);
                bulk_g2s_plain(nw_s, p.norm_w, static_cast<uint32_t>(K) * 2u, pro_bar);
            }
        }
    };
    if (p.prefetch) {
        copy_norm_w();   // a weight, like gate_w / up_w
        if (lane == 0 && !helper)
            for (int st = 0; st < S; ++st) fill(st);
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (!p.prefetch) {
        copy_norm_w();
        if (lane == 0 && !helper)
            for (int st = 0; st < S; ++st) fill(st);
    }
    __syncwarp();

    uint4 hreg[HREG ? kHregChunks : 1];
    if constexpr (NORM) {
        // the norm path always has 16-byte aligned operands (the host checks)
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(p.M) * static_cast<uint32_t>(K) * 2u;
            mbar_arrive_expect_tx(pro_bar, bytes);
            bulk_g2s_plain(h_s, p.s, bytes, pro_bar);   // residual rows into h_s rows 0..M-1
        }
        const RowMap rm = row_map(p.M, K);
        XRowsN<kXRowsSmall> xr;
        if (p.fused) x_prefetch_rows(p, rm, xr);
        prologue_wait(pro_bar);
        float2 ss;
        if (p.fused) {
            if (threadIdx.x == 0) fused_arrive(p);
            ss = add_rows_in_place(p, rm, h_s, K, xr);
        } else {
            ss = square_rows(rm, h_s, K);
        }
        norm_rows_in_place(p, rm, ss, h_s, K, nw_s, norm_partials(smem, p), inv_s, MB);
    } else if constexpr (!HREG) {
        if (p.vec_in) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(p.M) * static_cast<uint32_t>(K) * 2u);
                copy_rows_async(h_s, K, p.h, p.ldh, p.M, K, pro_bar);
            }
            for (int i = threadIdx.x; i < (MB - p.M) * (K >> 3); i += blockDim.x)
                reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(p.M) * K)[i] = make_uint4(0, 0, 0, 0);
            prologue_wait(pro_bar);
        } else {
            load_h_to_smem<MB>(p, h_s);
        }
        __syncthreads();
    }
    if constexpr (HREG) {
        const uint16_t *hsrc = NORM ? h_s : p.h;
        const bool vec = NORM || p.vec_in;
#pragma unroll
        for (int j = 0; j < kHregChunks; ++j) {
            const int c = lane + 32 * j;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (c < (K >> 3)) {
                if (vec) {
                    v = *reinterpret_cast<const uint4 *>(hsrc + c * 8);
                } else {
                    uint32_t w[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        w[q] = static_cast<uint32_t>(hsrc[c * 8 + 2 * q]) |
                               (static_cast<uint32_t>(hsrc[c * 8 + 2 * q + 1]) << 16);
                    v = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            hreg[j] = v;
        }
    }

    if (helper) {
        fused_residual_helper(p);
        return;
    }

    float2 ag[R][MB], au[R][MB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) ag[r][m] = au[r][m] = make_float2(0.0f, 0.0f);

    int seg = nseg;   // consumer-side segment of the current group
    for (int u = 0;; ++u) {
        const int st = u % S;
        const int g = slot_grp[st];
        if (g < 0) break;
        seg = (seg + 1 < nseg) ? seg + 1 : 0;
        const bool ok = mbar_wait_bounded(&bars[st], static_cast<uint32_t>((u / S) & 1), kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) {
                atomicExch(&g_device_error, kErrTimeout);
                // let the copies this warp still has in flight land before exiting
                for (int v = u; v < u + S; ++v)
                    if (slot_grp[v % S] >= 0)
                        mbar_wait_bounded(&bars[v % S], static_cast<uint32_t>((v / S) & 1), kWaitLimitNs);
            }
            __syncwarp();
            return;
        }
        const int k0 = seg * KS;
        const int nch = min(KS, K - k0) >> 3;
        const uint16_t *wg = ring + st * stage_elems;
        const uint16_t *wu = wg + R * KS;
        if constexpr (HREG) {
#pragma unroll
            for (int j = 0; j < kHregChunks; ++j) {
                const int c = lane + 32 * j;
                if (c < nch) {
                    const uint4 h4 = hreg[j];
                    const float2 hv[4] = {make_float2(bf16_lo(h4.x), bf16_hi(h4.x)),
                                          make_float2(bf16_lo(h4.y), bf16_hi(h4.y)),
                                          make_float2(bf16_lo(h4.z), bf16_hi(h4.z)),
                                          make_float2(bf16_lo(h4.w), bf16_hi(h4.w))};
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint4 g4 = *reinterpret_cast<const uint4 *>(wg + r * KS + c * 8);
                        const uint4 u4 = *reinterpret_cast<const uint4 *>(wu + r * KS + c * 8);
                        ag[r][0] = __ffma2_rn(hv[0], make_float2(bf16_lo(g4.x), bf16_hi(g4.x)), ag[r][0]);
                        au[r][0] = __ffma2_rn(hv[0], make_float2(bf16_lo(u4.x), bf16_hi(u4.x)), au[r][0]);
                        ag[r][0] = __ffma2_rn(hv[1], make_float2(bf16_lo(g4.y), bf16_hi(g4.y)), ag[r][0]);
                        au[r][0] = __ffma2_rn(hv[1], make_float2(bf16_lo(u4.y), bf16_hi(u4.y)), au[r][0]);
                        ag[r][0] = __ffma2_rn(hv[2], make_float2(bf16_lo(g4.z), bf16_hi(g4.z)), ag[r][0]);
                        au[r][0] = __ffma2_rn(hv[2], make_float2(bf16_lo(u4.z), bf16_hi(u4.z)), au[r][0]);
                        ag[r][0] = __ffma2_rn(hv[3], make_float2(bf16_lo(g4.w), bf16_hi(g4.w)), ag[r][0]);
                        au[r][0] = __ffma2_rn(hv[3], make_float2(bf16_lo(u4.w), bf16_hi(u4.w)), au[r][0]);
                    }
                }
            }
        } else {
            const uint16_t *hk = h_s + k0;
#pragma unroll 2
            for (int c = lane; c < nch; c += 32) {
                float2 gv[R][4], uv[R][4];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint4 g4 = *reinterpret_cast<const uint4 *>(wg + r * KS + c * 8);
                    const uint4 u4 = *reinterpret_cast<const uint4 *>(wu + r * KS + c * 8);
                    gv[r][0] = make_float2(bf16_lo(g4.x), bf16_hi(g4.x));
                    gv[r][1] = make_float2(bf16_lo(g4.y), bf16_hi(g4.y));
                    gv[r][2] = make_float2(bf16_lo(g4.z), bf16_hi(g4.z));
                    gv[r][3] = make_float2(bf16_lo(g4.w), bf16_hi(g4.w));
                    uv[r][0] = make_float2(bf16_lo(u4.x), bf16_hi(u4.x));
                    uv[r][1] = make_float2(bf16_lo(u4.y), bf16_hi(u4.y));
                    uv[r][2] = make_float2(bf16_lo(u4.z), bf16_hi(u4.z));
                    uv[r][3] = make_float2(bf16_lo(u4.w), bf16_hi(u4.w));
                }
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    const uint4 h4 = *reinterpret_cast<const uint4 *>(hk + static_cast<int64_t>(m) * K + c * 8);
                    const float2 hv[4] = {make_float2(bf16_lo(h4.x), bf16_hi(h4.x)),
                                          make_float2(bf16_lo(h4.y), bf16_hi(h4.y)),
                                          make_float2(bf16_lo(h4.z), bf16_hi(h4.z)),
                                          make_float2(bf16_lo(h4.w), bf16_hi(h4.w))};
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            ag[r][m] = __ffma2_rn(hv[j], gv[r][j], ag[r][m]);
                            au[r][m] = __ffma2_rn(hv[j], uv[r][j], au[r][m]);
                        }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async_smem();
            fill(st);   // the unit S ahead of u, or -1 once the CTA's groups run out
        }
        __syncwarp();
        if (seg == nseg - 1) {
            const int row0 = group_row0(g);
            float gsel = 0.0f, usel = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    const float gs = warp_allsum(ag[r][m].x + ag[r][m].y);
                    const float us = warp_allsum(au[r][m].x + au[r][m].y);
                    if (lane == r * MB + m) { gsel = gs; usel = us; }
                    ag[r][m] = au[r][m] = make_float2(0.0f, 0.0f);
                }
            const int r = lane / MB, m = lane - (lane / MB) * MB;
            if (lane < R * MB && m < p.M && row0 + r < r1)
                glu_store(p, m, row0 + r, gsel, usel);
        }
    }
}

// ---------------------------------------------------------------------------
// the tensor-core streaming kernel (batch 3..16)
// ---------------------------------------------------------------------------
//
// For batches where CUDA-core issue, not HBM, would bound the GEMV (about
// 150 instructions per KB of weights at M = 8), the same streaming scheme
// feeds mma.sync.m16n8k16 (bf16 in, fp32 accumulate):
//   A (16 x 16) = h rows 0..15 at k..k+15 -- rows >= M read a zero row;
//   B (16 x 8)  = 8 consecutive weight rows at k..k+15 (gate, then up);
//   D (16 x 8)  = g (or u) for 16 batch rows x 8 output features.
// A group is 8 consecutive rows; a unit is (group, K-segment of KS).  A stage
// holds the unit's 8 gate rows then 8 up rows at a pitch of KS + 8 elements:
// (KS + 8) / 8 is odd, so ldmatrix's 8 row addresses fall in 8 different
// 16-byte bank groups (no conflicts).  A whole group arrives as ONE tensor
// copy per matrix: a (KS + 8) x 8 box at (k0, row0), whose 8 extra columns
// are the next segment's first elements (read again from L2 by the next
// unit) or zeros past K.  One request per matrix instead of one per row:
// measured on GB300, 16 row copies of 0.5-0.6 KB per stage cost 9-30% of the
// call.  A CTA's last, partial group is copied row by row (lanes 0..15)
// into the same layout, so no row of another CTA's share is read.
//
// Work split: the CTA's units, in (group, segment) order, are cut into one
// contiguous range per ring-owning warp, equal to within one unit.  A CTA
// holds only ~10 groups of 8 rows, so dealing out whole groups would leave
// some warps a third more work than others.  A group cut between warps keeps
// the exact arithmetic of an uncut one: the warp holding its first segments
// runs them FIRST and parks its raw MMA accumulators in shared memory; the
// next warp runs the rest of the group LAST, resuming those accumulators.
// So each warp streams: [head of its last group, if cut] [whole groups]
// [tail of its first group, if cut].  Heads never wait; a tail waits only on
// a lower warp, so the hand-offs cannot deadlock, and every output's
// arithmetic is independent of where its row falls.  Each segment's MMAs
// form one chain from zero, which is then added (round to nearest) into the
// group's fp32 totals: the tensor core's own accumulation need not round to
// nearest, and its error would otherwise grow with K.
//
// Shared memory (dynamic):  [0, 1024)            mbarriers (ring, prologue, hand-off)
//                           [off_h, off_s)       h_s[M + 1][K + 8] bf16 (row M = 0; no row M at M = 16)
//                           [off_s, off_piece)   norm: norm_w[K] bf16
//                           [off_piece, off_ring) parked[warp][16][32] fp32
//                           [off_ring, ...)      ring[warp][stage][16][KS + 8] bf16
__device__ __forceinline__ void ldmatrix_x4(uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3,
                                            const void *row)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(smem_addr(row)));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t &b0, uint32_t &b1, const void *row)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(b0), "=r"(b1)
                 : "r"(smem_addr(row)));
}

__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Matrix loads by shared-memory address and register-only MMAs (the
// backward pass and the K-slice kernel).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// MMAs as plain (non-volatile) asm: register operands only, so the compiler
// may interleave independent accumulators
__device__ __forceinline__ void mma16_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// the same with C = 0
__device__ __forceinline__ void mma16_bf16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ void mma8_bf16(float (&d)[4], const uint32_t (&a)[2], uint32_t b0)
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(b0));
}

constexpr int kMmaRows = 8;                 // weight rows per group (the MMA's n)
constexpr uint32_t kPieceBarOffset = 800;   // one mbarrier per ring-owning warp
constexpr uint32_t kPhaseBarOffset = 872;   // K-phases: every ring warp has finished the phase
constexpr uint32_t kHBarOffset = 880;       // K-phases: the next phase's h rows have landed
constexpr uint32_t kPieceBytes = 2048;      // one warp's parked accumulators: [16][32] fp32
constexpr int kMaxPhases = 2;

struct MmaMaps {
    TensorMap gate, up;   // [N][K] bf16, row stride ld; box (KS + 8) x 8 rows
};

// Up to kMaxStreamWarps ring-owning warps, plus the helper warp on the
// single-kernel norm path.
template <bool NORM>
__global__ void __launch_bounds__((kMaxStreamWarps + 1) * 32, 1)
    glu_mma_kernel(const GluParams p, const __grid_constant__ MmaMaps maps)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float inv_s[2 * kMaxM];                  // norm: (inv_hi, inv_lo) per row

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages, KS = p.KS, K = p.K, nseg = p.nseg;
    const int RS = KS + 8;                                   // padded ring row, elements
    // K-phases: h_s holds NSP segments (HW columns) of h at a time; with one
    // phase it holds all of K.
    const int P = p.nphase, NSP = p.nsp;
    const int HW = min(K, NSP * KS);
    const int HS = HW + 8;                                   // padded h row, elements
    const int64_t stage_elems = static_cast<int64_t>(2) * kMmaRows * RS;
    const bool helper = warp == p.helper_warp;   // single-kernel norm path only; owns no ring
    const int W = p.helper_warp >= 0 ? p.helper_warp : static_cast<int>(blockDim.x >> 5);   // ring owners
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem) + warp * S;
    uint64_t *piece_bar = reinterpret_cast<uint64_t *>(smem + kPieceBarOffset);
    uint16_t *h_s = reinterpret_cast<uint16_t *>(smem + p.off_h);
    uint16_t *ring = reinterpret_cast<uint16_t *>(smem + p.off_ring) + static_cast<int64_t>(warp) * S * stage_elems;

    const int R = kMmaRows;
    const int r0 = p.interleave ? 0 : static_cast<int>((static_cast<int64_t>(p.N) * blockIdx.x) / gridDim.x);
    const int r1 = p.interleave ? p.N : static_cast<int>((static_cast<int64_t>(p.N) * (blockIdx.x + 1)) / gridDim.x);
    const int all_groups = (p.N + R - 1) / R;
    const int ngroups = p.interleave
                            ? (all_groups > static_cast<int>(blockIdx.x)
                                   ? (all_groups - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                                   : 0)
                            : (r1 - r0 + R - 1) / R;
    auto group_row0 = [&](int g) -> int {
        return p.interleave ? (g * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x)) * R : r0 + g * R;
    };
    // In phase ph, warp w owns the phase's units (group, segment), in that
    // order, [ub, ue) -- an equal share -- and streams them as
    //   A = [a0, ue)      head of a group that continues in the next warp
    //   B = [c1, a0)      whole groups
    //   C = [ub, c1)      tail of a group begun by the previous warp
    // The phases follow one another; a warp streams all of its phase-0 units,
    // then its phase-1 units.
    struct Range {
        int ub, ue, c1, a0, len_a, len_ab, n, nsp;
        bool cont;
    };
    auto range_of = [&](int ph, int w) -> Range {
        Range r;
        r.nsp = min(NSP, nseg - ph * NSP);
        const int units = ngroups * r.nsp;
        r.ub = static_cast<int>((static_cast<int64_t>(units) * w) / W);
        r.ue = static_cast<int>((static_cast<int64_t>(units) * (w + 1)) / W);
        if (w >= W) r.ub = r.ue = units;   // the helper warp streams nothing
        r.cont = r.ub < r.ue && r.ub % r.nsp != 0;
        r.c1 = r.cont ? min(r.ue, (r.ub / r.nsp + 1) * r.nsp) : r.ub;
        r.a0 = (r.ue % r.nsp != 0 && r.c1 < r.ue) ? ((r.ue - 1) / r.nsp) * r.nsp : r.ue;
        r.len_a = r.ue - r.a0;
        r.len_ab = r.len_a + (r.a0 - r.c1);
        r.n = r.ue - r.ub;
        return r;
    };
    // the j-th unit of range r (phase ph) -> group g, segment seg of K
    auto unit_at = [&](const Range &r, int ph, int j, int &g, int &seg) {
        const int v = j < r.len_a ? r.a0 + j : (j < r.len_ab ? r.c1 + (j - r.len_a) : r.ub + (j - r.len_ab));
        g = v / r.nsp;
        seg = ph * NSP + (v - g * r.nsp);
    };
    // this warp's ranges, computed once (kMaxPhases == 2)
    const Range rg0 = range_of(0, warp);
    const Range rg1 = range_of(P > 1 ? 1 : 0, warp);
    const int n_total = rg0.n + (P > 1 ? rg1.n : 0);
    // the i-th unit this warp streams, counted over all phases
    auto unit_seq = [&](int i, int &g, int &seg) {
        if (P == 1 || i < rg0.n)
            unit_at(rg0, 0, i, g, seg);
        else
            unit_at(rg1, 1, i - rg0.n, g, seg);
    };

    uint64_t *pro_bar = reinterpret_cast<uint64_t *>(smem + kProBarOffset);
    if (lane == 0 && !helper)
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    if (threadIdx.x == 0) {
        mbar_init(pro_bar, NORM ? 2 : 1);   // norm: the norm_w copy and the residual copy
        for (int w = 0; w < W; ++w) mbar_init(&piece_bar[w], 32);
        if (P > 1) {
            mbar_init(reinterpret_cast<uint64_t *>(smem + kPhaseBarOffset), W);
            mbar_init(reinterpret_cast<uint64_t *>(smem + kHBarOffset), 1);
        }
    }
    fence_mbar_init();
    __syncthreads();

    // the backward's next step reads the weights again (last rows first):
    // keep them in L2 in that mode
    const uint64_t policy = p.mode == kModeBwd ? l2_policy_evict_last() : l2_policy_evict_first();
    // Tensor copies need 128-byte aligned destinations: every stage and its
    // up half sit at multiples of 128 bytes from the ring (32 * (KS + 8) and
    // 16 * (KS + 8) bytes with KS % 16 == 0), so checking the ring suffices.
    const bool use_tma = p.tma && (smem_addr(smem + p.off_ring) & 127u) == 0u;
    // whole warp: request unit (g, seg) into stage st.  Lane 0 posts the byte
    // count first; lanes 0..nr-1 copy gate rows, 8..8+nr-1 up rows.
    auto issue = [&](int st, int g, int seg) {
        const int row0 = group_row0(g);
        const int nr = min(R, r1 - row0);
        const int k0 = seg * KS;
        const int len = min(KS, K - k0);
        uint16_t *stage = ring + st * stage_elems;
        if (use_tma && nr == R) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[st], 2u * static_cast<uint32_t>(R * RS) * 2u);
                tma_load_2d(stage, &maps.gate, k0, row0, &bars[st], policy);
                tma_load_2d(stage + R * RS, &maps.up, k0, row0, &bars[st], policy);
            }
            __syncwarp();
            return;
        }
        const uint32_t row_bytes = static_cast<uint32_t>(len) * 2u;
        if (lane == 0) mbar_arrive_expect_tx(&bars[st], 2u * static_cast<uint32_t>(nr) * row_bytes);
        __syncwarp();
        const int r = lane & 7;
        if (lane < 16 && r < nr) {
            const bool up = lane >= 8;
            const uint16_t *src = up ? p.up + static_cast<int64_t>(row0 + r) * p.ld_up + k0
                                     : p.gate + static_cast<int64_t>(row0 + r) * p.ld_gate + k0;
            uint16_t *dst = stage + static_cast<int64_t>((up ? R : 0) + r) * RS;
            bulk_g2s(dst, src, row_bytes, &bars[st], policy);
        }
    };
    auto prefill = [&]() {
        for (int i = 0; i < S && i < n_total; ++i) {
            int g, seg;
            unit_seq(i, g, seg);
            issue(i, g, seg);
        }
    };

    uint16_t *nw_s = reinterpret_cast<uint16_t *>(smem + p.off_s);   // norm: norm_w, K elements
    auto copy_norm_w = [&]() {
        if constexpr (NORM) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(K) * 2u);
                bulk_g2s_plain(nw_s, p.norm_w, static_cast<uint32_t>(K) * 2u, pro_bar);
            }
        }
    };
    if (p.prefetch) {
        copy_norm_w();   // a weight, like gate_w / up_w
        prefill();
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (!p.prefetch) {
        copy_norm_w();
        prefill();
    }
    __syncwarp();

    // h rows 0..M-1, then a zero row M when M < 16 (padded stride HS)
    if constexpr (NORM) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(p.M) * static_cast<uint32_t>(K) * 2u);
            copy_rows_async(h_s, HS, p.s, K, p.M, K, pro_bar);   // residual rows, padded
        }
        const RowMap rm = row_map(p.M, K);
        XRows xr;
        if (p.fused) x_prefetch_rows(p, rm, xr);
        prologue_wait(pro_bar);
        float2 ss;
        if (p.fused) {
            if (threadIdx.x == 0) fused_arrive(p);
            ss = add_rows_in_place(p, rm, h_s, HS, xr);
        } else {
            ss = square_rows(rm, h_s, HS);
        }
        norm_rows_in_place(p, rm, ss, h_s, HS, nw_s, norm_partials(smem, p), inv_s, p.M);
    } else if (p.vec_in) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(pro_bar, static_cast<uint32_t>(p.M) * static_cast<uint32_t>(HW) * 2u);
            copy_rows_async(h_s, HS, p.h, p.ldh, p.M, HW, pro_bar);   // phase 0's columns
        }
        prologue_wait(pro_bar);
    } else {
        const int nch = HW >> 3;   // one phase here (the planner stages K only from aligned h)
        for (int i = threadIdx.x; i < p.M * nch; i += blockDim.x) {
            const int m = i / nch, c = i - m * nch;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                w[q] = static_cast<uint32_t>(p.h[m * p.ldh + c * 8 + 2 * q]) |
                       (static_cast<uint32_t>(p.h[m * p.ldh + c * 8 + 2 * q + 1]) << 16);
            *reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(m) * HS + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    if (p.M < kMaxM)   // at M = 16 every A row is a real row: no zero row is allocated or read
        for (int c = threadIdx.x; c < (HW >> 3); c += blockDim.x)
            *reinterpret_cast<uint4 *>(h_s + static_cast<int64_t>(p.M) * HS + c * 8) = make_uint4(0, 0, 0, 0);
    __syncthreads();

    // ldmatrix.x4 row addresses for A: lane l -> h row (l & 15) (zero row if
    // >= M), k offset (l >> 4) * 8.  ldmatrix.x2 for B: lane l (l < 16) -> ring
    // row (l & 7), k offset ((l >> 3) & 1) * 8.
    const int arow = (lane & 15) < p.M ? (lane & 15) : p.M;
    const uint16_t *a_base = h_s + static_cast<int64_t>(arow) * HS + (lane >> 4) * 8;
    const int b_off = (lane & 7) * RS + ((lane >> 3) & 1) * 8;

    if (helper) {
        fused_residual_helper(p);
        return;
    }

    // per matrix: *0 the unit's MMA chain, started from zero at every unit;
    // *1 the fp32 total, to which each unit's chain is added once (round to
    // nearest).  The tensor core's own accumulation is not specified to round
    // to nearest, so its chains stay at most one segment (<= 15 MMAs) long.
    float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
    float v0[4] = {0.f, 0.f, 0.f, 0.f}, v1[4] = {0.f, 0.f, 0.f, 0.f};
    float *const parked = reinterpret_cast<float *>(smem + p.off_piece);
    float *const carry = reinterpret_cast<float *>(smem + p.off_carry);
    uint64_t *phase_bar = reinterpret_cast<uint64_t *>(smem + kPhaseBarOffset);
    uint64_t *h_bar = reinterpret_cast<uint64_t *>(smem + kHBarOffset);
    auto store_acc = [&](float *slot) {   // [16][32] fp32; the accumulators restart from zero
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            slot[q * 32 + lane] = g0[q];
            slot[(4 + q) * 32 + lane] = g1[q];
            slot[(8 + q) * 32 + lane] = v0[q];
            slot[(12 + q) * 32 + lane] = v1[q];
            g0[q] = g1[q] = v0[q] = v1[q] = 0.f;
        }
    };
    auto load_acc = [&](const float *slot) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            g0[q] = slot[q * 32 + lane];
            g1[q] = slot[(4 + q) * 32 + lane];
            v0[q] = slot[(8 + q) * 32 + lane];
            v1[q] = slot[(12 + q) * 32 + lane];
        }
    };
    // bounded waits for this warp's copies in flight, units i..i+S-1
    auto drain = [&](int i) {
        if (lane == 0)
            for (int j = i; j < min(i + S, n_total); ++j)
                mbar_wait_bounded(&bars[j % S], static_cast<uint32_t>((j / S) & 1), kWaitLimitNs);
        __syncwarp();
    };
    int i = 0;   // units streamed so far, over all phases
    for (int ph = 0; ph < P; ++ph) {
        const Range &r = ph == 0 ? rg0 : rg1;
        const int k_lo = ph * NSP * KS;
        bool parked_now = false;
        if (ph > 0) {   // h_s holds this phase's columns once every warp finished the last phase
            const bool okh = mbar_wait_bounded(h_bar, static_cast<uint32_t>((ph - 1) & 1), kWaitLimitNs);
            if (!__all_sync(0xffffffffu, okh)) {
                if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
                drain(i);
                return;
            }
        }
        for (int j = 0; j < r.n; ++j, ++i) {
            int g, seg;
            unit_at(r, ph, j, g, seg);
            const int sp = seg - ph * NSP, st = i % S;
            bool ok = mbar_wait_bounded(&bars[st], static_cast<uint32_t>((i / S) & 1), kWaitLimitNs);
            if (j == r.len_ab && r.cont) {
                // resume the accumulators of the warp holding the group's earlier
                // segments of this phase: the nearest lower warp with units
                int prev = warp - 1;
                while (prev > 0 && range_of(ph, prev).n == 0) --prev;
                ok = mbar_wait_bounded(&piece_bar[prev], static_cast<uint32_t>(ph & 1), kWaitLimitNs) && ok;
                load_acc(parked + prev * (kPieceBytes / 4));
            } else if (sp == 0 && ph > 0) {
                load_acc(carry + static_cast<int64_t>(g) * (kPieceBytes / 4));   // the group's earlier phases
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) atomicExch(&g_device_error, kErrTimeout);
                drain(i);
                return;
            }
            const int k0 = seg * KS;
            const int nk = min(KS, K - k0) >> 4;                 // whole k16 steps
            const uint16_t *wg = ring + st * stage_elems + b_off;
            const uint16_t *wu = wg + R * RS;
            const uint16_t *ha = a_base + (k0 - k_lo);
#pragma unroll 2
            for (int kk = 0; kk < nk; ++kk) {
                uint32_t a0r, a1r, a2r, a3r, b0, b1, c0, c1r;
                ldmatrix_x4(a0r, a1r, a2r, a3r, ha + kk * 16);
                ldmatrix_x2(b0, b1, wg + kk * 16);
                ldmatrix_x2(c0, c1r, wu + kk * 16);
                mma_bf16_16x8x16(g0, a0r, a1r, a2r, a3r, b0, b1);
                mma_bf16_16x8x16(v0, a0r, a1r, a2r, a3r, c0, c1r);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // the unit's chain into the totals
                g1[q] = __fadd_rn(g1[q], g0[q]);
                v1[q] = __fadd_rn(v1[q], v0[q]);
                g0[q] = v0[q] = 0.f;
            }
            __syncwarp();
            if (i + S < n_total) {
                int gn, segn;
                unit_seq(i + S, gn, segn);
                if (lane == 0) fence_proxy_async_smem();
                issue(st, gn, segn);   // the unit S ahead, into the stage just read
            }
            __syncwarp();
            if (j == r.len_a - 1) {   // end of A: the group continues in the next warp
                store_acc(parked + warp * (kPieceBytes / 4));
                mbar_arrive(&piece_bar[warp]);   // every lane: releases its own stores
                parked_now = true;
                continue;
            }
            if (sp != r.nsp - 1) {
                if (j == r.n - 1) {   // C inside one group: it continues in the next warp too
                    store_acc(parked + warp * (kPieceBytes / 4));
                    mbar_arrive(&piece_bar[warp]);
                    parked_now = true;
                }
                continue;
            }
            if (ph < P - 1) {   // the group goes on in the next phase
                store_acc(carry + static_cast<int64_t>(g) * (kPieceBytes / 4));
                continue;
            }
            // the group is complete.  D layout: d[0], d[1] -> batch row lane/4,
            // features 2*(lane%4) + 0, 1; d[2], d[3] -> batch row lane/4 + 8.
            const int row0 = group_row0(g);
            const int m0 = lane >> 2, n = row0 + 2 * (lane & 3);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int m = m0 + (q >> 1) * 8, nn = n + (q & 1);
                if (m < p.M && nn < r1 && nn < row0 + R)
                    glu_store(p, m, nn, g0[q] + g1[q], v0[q] + v1[q]);
                g0[q] = g1[q] = v0[q] = v1[q] = 0.f;
            }
        }
        if (P == 1) break;
        // one arrival per warp and phase on its piece barrier keeps the phase
        // parities of all piece barriers equal to the phase index
        if (!parked_now) mbar_arrive(&piece_bar[warp]);
        if (ph < P - 1) {
            // every warp has finished reading this phase's h: thread 0 then
            // copies the next phase's columns (the rings keep streaming)
            __syncwarp();
            if (lane == 0) mbar_arrive(phase_bar);
            if (warp == 0 && lane == 0) {
                if (mbar_wait_bounded(phase_bar, static_cast<uint32_t>(ph & 1), kWaitLimitNs)) {
                    const int k_next = (ph + 1) * NSP * KS, w_next = min(HW, K - k_next);
                    fence_proxy_async_smem();   // the warps' reads of h_s (acquired above) before the copy's writes
                    mbar_arrive_expect_tx(h_bar, static_cast<uint32_t>(p.M) * static_cast<uint32_t>(w_next) * 2u);
                    copy_rows_async(h_s, HS, p.h + k_next, p.ldh, p.M, w_next, h_bar);
                } else {
                    atomicExch(&g_device_error, kErrTimeout);   // the other warps give up on h_bar
                }
            }
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------------------
// generic kernel: any 2-byte-aligned operands, same arithmetic rules
// ---------------------------------------------------------------------------
// One warp per output feature (grid-stride), lanes stride K with 2-byte loads,
// a runtime loop over the batch rows.  NORM computes the normed rows into
// dynamic shared memory h_s[M][K] first.
template <bool NORM>
__global__ void __launch_bounds__(256) glu_generic_kernel(const GluParams p)
{
    extern __shared__ __align__(16) unsigned char smem_g[];
    __shared__ float2 red[kMaxWarps][kMaxM];
    __shared__ float inv_s[2 * kMaxM];
    grid_dependency_wait();
    grid_launch_dependents();
    const uint16_t *hp = p.h;
    int64_t hld = p.ldh;
    if constexpr (NORM) {
        uint16_t *h_s = reinterpret_cast<uint16_t *>(smem_g);
        GluParams q = p;
        q.vec_in = 0;
        norm_prologue<kMaxM>(q, h_s, red, inv_s, p.M);
        __syncthreads();
        hp = h_s;
        hld = p.K;
    }
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < p.N;
         row += nwarps) {
        const uint16_t *grow = p.gate + row * p.ld_gate;
        const uint16_t *urow = p.up + row * p.ld_up;
        for (int m = 0; m < p.M; ++m) {
            const uint16_t *hrow = hp + m * hld;
            float g = 0.0f, u = 0.0f;
            for (int k = lane; k < p.K; k += 32) {
                const float a = bf16_to_f32(hrow[k]);
                g = fmaf(a, bf16_to_f32(grow[k]), g);
                u = fmaf(a, bf16_to_f32(urow[k]), u);
            }
            g = warp_allsum(g);
            u = warp_allsum(u);
            if (lane == 0) glu_store(p, m, row, g, u);
        }
    }
}

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------

// s = bf16(x + residual), written back into residual (one rounding: the fp32
// sum of two bf16 values rounds to the same bf16 as the exact sum).  Releases
// the dependent GEMV launch at once (that grid touches nothing but weights
// until this grid has completed), then waits for its own predecessor before
// reading x and residual.
__global__ void __launch_bounds__(256) residual_add_kernel(const uint16_t *x, uint16_t *res, int64_t count,
                                                           int vec)
{
    grid_launch_dependents();
    grid_dependency_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec) {
        for (; i < count / 8; i += stride) {
            const uint4 a = reinterpret_cast<const uint4 *>(x)[i];
            const uint4 b = reinterpret_cast<const uint4 *>(res)[i];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
            uint32_t r[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                r[j] = pack_bf16x2(bf16_lo(aw[j]) + bf16_lo(bw[j]), bf16_hi(aw[j]) + bf16_hi(bw[j]));
            reinterpret_cast<uint4 *>(res)[i] = make_uint4(r[0], r[1], r[2], r[3]);
        }
    } else {
        for (; i < count; i += stride) res[i] = f32_to_bf16(bf16_to_f32(x[i]) + bf16_to_f32(res[i]));
    }
}

// K == 0: empty dot products, SiLU(0) * 0 = +0 in both modes.
__global__ void __launch_bounds__(256) zero_fill_kernel(uint16_t *out, int64_t ldo, int M, int N)
{
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t total = static_cast<int64_t>(M) * N;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        out[m * ldo + n] = 0;
    }
}

// ---------------------------------------------------------------------------
// silu_mul: the GLU epilogue on projections computed elsewhere
// ---------------------------------------------------------------------------
// Halves layout (PR #8602, "fused_glu" commit): row m of x holds the gate
// projection in columns [0, N) and the up projection in [N, 2N); out[m, n] =
// epilogue(x[m, n], x[m, N + n]).  g and u are bf16 already, so the HF
// roundings of g and u are identities.  Per element the work is one SiLU, so
// unlike the GEMVs the epilogue's instruction count sets the pace: SiLU here
// takes a correctly rounded reciprocal and a product instead of an IEEE
// division (three roundings in all, a few fp32 ulps, far below a bf16 ulp).
__device__ __forceinline__ float silu_rcp_f32(float x)
{
    const float t = expf(-fabsf(x));
    return (x >= 0.0f ? x : x * t) * __frcp_rn(1.0f + t);
}

// SiLU by table.  g is a bf16 value, so SiLU(g) -- and in HF mode its bf16
// rounding -- is a function of g's 16 bits.  Each CTA tabulates it, from the
// same silu_rcp_f32, for the gates |g| in [2^-8, 2^7) (15 binades x 128
// mantissas x 2 signs, 15 KB of fp32; a N(0, 1) gate lies there 99.7% of the
// time) before its dependency wait; other gates take the direct path.  Then
// FUSED: out = bf16(SiLU(g) u), one rounding; HF: out = bf16(bf16(SiLU(g)) u)
// (the bf16 product is exact in fp32).  The results are bit for bit those of
// evaluating SiLU at every output.
constexpr int kSiluLutExp0 = 127 - 8;   // biased exponent of the table's first binade
constexpr int kSiluLutBinades = 15;
constexpr int kSiluLutSize = 2 * kSiluLutBinades * 128;

__device__ __forceinline__ void silu_lut_build(float *lut, int mode)
{
    for (int i = threadIdx.x; i < kSiluLutSize; i += blockDim.x) {
        const int sign = i / (kSiluLutBinades * 128), rem = i - sign * (kSiluLutBinades * 128);
        const uint32_t bits = (static_cast<uint32_t>(sign) << 15) |
                              (static_cast<uint32_t>(kSiluLutExp0 + (rem >> 7)) << 7) | static_cast<uint32_t>(rem & 127);
        const float sl = silu_rcp_f32(bf16_to_f32(static_cast<uint16_t>(bits)));
        lut[i] = mode == 0 ? sl : round_to_bf16(sl);
    }
}

// out = epilogue(g, u) for one pair, g and u as bf16 bits
__device__ __forceinline__ float silu_mul_lut_one(const float *lut, uint32_t gbits, uint32_t ubits, int mode)
{
    const int e = static_cast<int>((gbits >> 7) & 0xffu) - kSiluLutExp0;
    float sl;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(kSiluLutBinades)) {
        sl = lut[((gbits >> 15) * kSiluLutBinades + static_cast<uint32_t>(e)) * 128u + (gbits & 127u)];
    } else {
        sl = silu_rcp_f32(bf16_to_f32(static_cast<uint16_t>(gbits)));
        if (mode != 0) sl = round_to_bf16(sl);
    }
    return sl * bf16_to_f32(static_cast<uint16_t>(ubits));
}

__device__ __forceinline__ uint4 silu_mul_chunk(const float *lut, uint4 gv, uint4 uv, int mode)
{
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        o[j] = pack_bf16x2(silu_mul_lut_one(lut, gw[j] & 0xffffu, uw[j] & 0xffffu, mode),
                           silu_mul_lut_one(lut, gw[j] >> 16, uw[j] >> 16, mode));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// HBM traffic: 4 bytes read and 2 written per output.  vec: one thread per 8
// outputs, two chunks per iteration so that four 16-byte streaming loads are
// in flight per thread; else one thread per output.  Waits for the preceding
// grid, which produces x.
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint16_t *x, int64_t ldx, uint16_t *out, int64_t ldo,
                                                       int M, int N, int mode, int vec)
{
    __shared__ float lut[kSiluLutSize];
    silu_lut_build(lut, mode);   // no global input: before the dependency wait
    __syncthreads();
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (vec) {
        // chunk i = m * nch + c, visited i, i + stride, ...: (m, c) advance by
        // (stride / nch, stride % nch) with a carry, one division per thread
        const int nch = N >> 3;
        const int64_t total = static_cast<int64_t>(M) * nch;
        int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        const int64_t dm = stride / nch, dc = stride - dm * nch;
        int64_t m0 = i / nch, c0 = i - m0 * nch;
        auto step = [&](int64_t &m, int64_t &c) {
            m += dm;
            c += dc;
            if (c >= nch) {
                c -= nch;
                ++m;
            }
        };
        for (; i + stride < total; i += 2 * stride) {
            int64_t m1 = m0, c1 = c0;
            step(m1, c1);
            const uint16_t *r0 = x + m0 * ldx + c0 * 8, *r1 = x + m1 * ldx + c1 * 8;
            const uint4 g0 = __ldcs(reinterpret_cast<const uint4 *>(r0));
            const uint4 u0 = __ldcs(reinterpret_cast<const uint4 *>(r0 + N));
            const uint4 g1 = __ldcs(reinterpret_cast<const uint4 *>(r1));
            const uint4 u1 = __ldcs(reinterpret_cast<const uint4 *>(r1 + N));
            __stcs(reinterpret_cast<uint4 *>(out + m0 * ldo + c0 * 8), silu_mul_chunk(lut, g0, u0, mode));
            __stcs(reinterpret_cast<uint4 *>(out + m1 * ldo + c1 * 8), silu_mul_chunk(lut, g1, u1, mode));
            m0 = m1;
            c0 = c1;
            step(m0, c0);
        }
        if (i < total) {
            const uint16_t *r0 = x + m0 * ldx + c0 * 8;
            const uint4 g0 = __ldcs(reinterpret_cast<const uint4 *>(r0));
            const uint4 u0 = __ldcs(reinterpret_cast<const uint4 *>(r0 + N));
            __stcs(reinterpret_cast<uint4 *>(out + m0 * ldo + c0 * 8), silu_mul_chunk(lut, g0, u0, mode));
        }
    } else {
        const int64_t total = static_cast<int64_t>(M) * N;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const int64_t m = i / N, n = i - m * N;
            out[m * ldo + n] = f32_to_bf16(silu_mul_lut_one(lut, x[m * ldx + n], x[m * ldx + N + n], mode));
        }
    }
}

// ---------------------------------------------------------------------------
// gdn_gates: decay and write gates of the gated-delta-net layers
// ---------------------------------------------------------------------------
// PR #8602, the "fused_glu" commit: the write gate is the sigmoid of b and
// the decay gate is -exp(A_log) times the softplus of a + dt_bias, computed in
// fp32 with softplus in its overflow-safe form; PR #9057 ("Changes"): the
// decay gates stay fp32.  For token t,
// head j: x = a + dt_bias[j] (fp32), g = -exp(A_log[j]) * softplus(x) (fp32),
// beta = bf16(sigmoid(b)).  softplus in its stable form: x + log1p(e^-x) for
// x > 0, log1p(e^x) otherwise -- never e^x of a large x -- and sigmoid from
// e^-|y| likewise.  Elementwise; a and b are row-strided views (e.g. columns
// of one projection output).
// One (token, head) of gdn_gates: a, b the inputs, neg_a = -exp(A_log[j]),
// dt = dt_bias[j].
__device__ __forceinline__ void gdn_gate_one(float a, float b, float neg_a, float dt, float &g, uint16_t &beta)
{
    const float x = a + dt;
    const float sp = x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
    g = neg_a * sp;
    // sigmoid without overflow: 1/(1 + e^-y) sends e^-y to +inf in fp32 for
    // y < -88.7 and returns 0, although e^y is still a (subnormal) bf16
    // value down to y ~ -92
    const float ty = expf(-fabsf(b));
    beta = f32_to_bf16((b >= 0.0f ? 1.0f : ty) / (1.0f + ty));
}

// Any shape: one thread per element.
__global__ void __launch_bounds__(256) gdn_gates_kernel(const uint16_t *a, int64_t lda, const uint16_t *b,
                                                        int64_t ldb, const float *A_log, const float *dt_bias,
                                                        float *g, int64_t ldg, uint16_t *beta, int64_t ldbeta,
                                                        int T, int H)
{
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t total = static_cast<int64_t>(T) * H;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / H, j = i - t * H;
        gdn_gate_one(bf16_to_f32(a[t * lda + j]), bf16_to_f32(b[t * ldb + j]), -expf(A_log[j]), dt_bias[j],
                     g[t * ldg + j], beta[t * ldbeta + j]);
    }
}

// Up to kGdnMaxHeads heads, T * ceil(H/8) < 2^31: one thread per (token, 8
// consecutive heads), 32-bit index arithmetic, the heads' -exp(A_log) and
// dt_bias computed once per CTA into shared memory.  vec: H % 8 == 0 and
// every row 16-byte aligned -- 16-byte loads of a and b, 16-byte stores of
// g (two) and beta, all streaming.
constexpr int kGdnMaxHeads = 4096;

__global__ void __launch_bounds__(256) gdn_gates_chunk_kernel(const uint16_t *a, int64_t lda, const uint16_t *b,
                                                              int64_t ldb, const float *A_log, const float *dt_bias,
                                                              float *g, int64_t ldg, uint16_t *beta, int64_t ldbeta,
                                                              int T, int H, int vec)
{
    __shared__ float neg_a_s[kGdnMaxHeads], dt_s[kGdnMaxHeads];
    grid_dependency_wait();
    grid_launch_dependents();
    for (int j = threadIdx.x; j < H; j += blockDim.x) {
        neg_a_s[j] = -expf(A_log[j]);
        dt_s[j] = dt_bias[j];
    }
    __syncthreads();
    const uint32_t hc = static_cast<uint32_t>(H + 7) >> 3;
    const uint32_t items = static_cast<uint32_t>(T) * hc;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < items; i += gridDim.x * blockDim.x) {
        const uint32_t t = i / hc;
        const int j0 = static_cast<int>(i - t * hc) * 8;
        const uint16_t *ar = a + static_cast<int64_t>(t) * lda + j0;
        const uint16_t *br = b + static_cast<int64_t>(t) * ldb + j0;
        float *gr = g + static_cast<int64_t>(t) * ldg + j0;
        uint16_t *betar = beta + static_cast<int64_t>(t) * ldbeta + j0;
        if (vec) {
            const uint4 av = __ldcs(reinterpret_cast<const uint4 *>(ar));
            const uint4 bv = __ldcs(reinterpret_cast<const uint4 *>(br));
            const uint32_t aw[4] = {av.x, av.y, av.z, av.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
            float gv[8];
            uint32_t be[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint16_t lo, hi;
                gdn_gate_one(bf16_lo(aw[q]), bf16_lo(bw[q]), neg_a_s[j0 + 2 * q], dt_s[j0 + 2 * q], gv[2 * q], lo);
                gdn_gate_one(bf16_hi(aw[q]), bf16_hi(bw[q]), neg_a_s[j0 + 2 * q + 1], dt_s[j0 + 2 * q + 1],
                             gv[2 * q + 1], hi);
                be[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            __stcs(reinterpret_cast<float4 *>(gr), make_float4(gv[0], gv[1], gv[2], gv[3]));
            __stcs(reinterpret_cast<float4 *>(gr + 4), make_float4(gv[4], gv[5], gv[6], gv[7]));
            __stcs(reinterpret_cast<uint4 *>(betar), make_uint4(be[0], be[1], be[2], be[3]));
        } else {
            const int n = min(8, H - j0);
            for (int e = 0; e < n; ++e)
                gdn_gate_one(bf16_to_f32(ar[e]), bf16_to_f32(br[e]), neg_a_s[j0 + e], dt_s[j0 + e], gr[e], betar[e]);
        }
    }
}

}  // namespace mbglu
