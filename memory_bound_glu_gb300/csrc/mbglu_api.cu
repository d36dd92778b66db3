// mbglu_api.cu -- the C ABI of libmbglu.so (declared in include/mbglu.h):
// host-side validation, launch planning and dispatch to the sm_103a kernels.
//
// The library is stateless apart from a per-device table of attributes (SM
// count, shared-memory limit) filled on first use under a mutex; it allocates
// nothing and caches nothing derived from the weights (DeepSpeed PR #9057
// commits on stale pointer-keyed caches: in-place weight updates must always
// be seen).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>

#include "mbglu.h"
#include "glu_kernels.cuh"
#include "glu_backward.cuh"
#include "glu_tc.cuh"
#include "glu_slice.cuh"

namespace {

using mbglu::GluParams;

thread_local int t_last_cuda_error = 0;
thread_local int t_last_variant = 0;
thread_local int t_last_single = 0;   // row blocks of the last norm call that ran as the single kernel
thread_local int t_last_bwd = 0;      // the last glu_backward's second step (mbglu_last_backward_path)

enum Variant {
    kNone = 0, kStream = 1, kGeneric = 2, kZeroFill = 3, kTensor = 4, kSiluMul = 5, kGdnGates = 6,
    kRowBlocks = 7,  // a batch above kBlockRows, run as row blocks
    kBackward = 8,   // glu_backward
    kTcGemv = 9,     // the tcgen05 kernel (one pass for batch 17..64)
    kSlice = 10      // the K-slice tensor-core kernel (batch 1..16 where it applies, h in registers)
};
constexpr int kBlockRows = mbglu::kMaxM;   // rows one GEMV kernel takes (its batch tile)

constexpr int kMaxDevices = 64;
constexpr uint32_t kBarRegion = 1024;        // mbarriers, stage -> group table, group counter
static_assert(mbglu::kMaxStreamWarps * 8 * 8 <= mbglu::kSlotGrpOffset, "mbarriers overflow their region");
static_assert(mbglu::kSlotGrpOffset + mbglu::kMaxStreamWarps * 8 * 4 <= mbglu::kCounterOffset,
              "stage table overflows its region");
static_assert(mbglu::kCounterOffset + 4 <= mbglu::kProBarOffset, "counter overlaps the prologue barrier");
static_assert(mbglu::kProBarOffset % 8 == 0 && mbglu::kProBarOffset + 8 <= mbglu::kPieceBarOffset,
              "prologue barrier overlaps the piece barriers");
static_assert(mbglu::kPieceBarOffset % 8 == 0 && mbglu::kPieceBarOffset + mbglu::kMaxStreamWarps * 8 <= mbglu::kPhaseBarOffset,
              "piece barriers overlap the phase barrier");
static_assert(mbglu::kPhaseBarOffset % 8 == 0 && mbglu::kPhaseBarOffset + 8 <= mbglu::kHBarOffset &&
                  mbglu::kHBarOffset % 8 == 0 && mbglu::kHBarOffset + 8 <= kBarRegion,
              "phase barriers outside the region");
constexpr int kMaxStages = 8;
constexpr int kMmaKsCap = 240;               // tensor-core segment: its box (KS + 8) x 8 must be <= 256 wide
constexpr int64_t kNormMaxMK = 81920;        // add_rmsnorm_glu: M*K*2 bytes of normed rows in smem

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;       // max dynamic + static shared memory per block
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Overrides for tuning sweeps only; every default is chosen by plan_stream.
// glu_bwd_mma_kernel: 64-column boxes per warp (2: 128-column slices; 4 measured slower)
constexpr int kBwdNB = 2;

struct Tuning {
    int warps = 0;            // warps per CTA of the streaming kernel (0: automatic)
    int rows = 0;             // rows per stage R in {1,2,4} (0: automatic)
    int ks = 0;               // K-segment length (0: automatic)
    int stages = 0;           // ring depth cap (0: as many as fit, <= 8)
    int smem_kb = 0;          // shared-memory budget cap in KiB (0: device limit)
    int ctas_per_sm = 0;      // 1 or 2 streaming CTAs per SM (0: automatic)
    int hreg = 1;             // batch 1: keep h in registers where K allows
    int waves = 1;            // CTAs per resident CTA slot (grid = SMs * ctas_per_sm * waves)
    int interleave = 0;       // row groups dealt round-robin over CTAs instead of contiguous blocks
    int mma_min_m = 3;        // smallest batch that takes the tensor-core kernel (17: never)
    int mma_ks_min = 192;     // tensor-core plan: shortest K-segment worth one more warp
    int tma = 1;              // tensor-core kernel: whole groups by tensor copy (0: row by row)
    int phases = 0;           // tensor-core kernel: K-phases (0: automatic, 1: never, 2: always where allowed)
    int tc = 1;               // batches of tc_min_m..64 on the tcgen05 kernel (0: row blocks)
    int tc_min_m = 17;        // smallest batch that takes the tcgen05 kernel
    int tc_split = 0;         // tcgen05 kernel: CTAs per tile (0: automatic, 1..4 where the plan allows)
    int bwd_fused = 1;        // backward: steps 2 and 3 in one pass where they apply (0: separate kernels)
    int bwd_mma_min_m = 3;    // backward: smallest batch whose one-pass step takes the tensor cores (17: never)
    int bwd_warps = 0;        // backward on the tensor cores: warps per CTA (0: automatic)
    int slice = 1;            // batches of slice_min_m..8 on the K-slice kernel where it applies (0: never)
    int slice_min_m = 1;      // smallest batch that takes the K-slice kernel
    int slice16 = 1;          // batches of 9..16 on the K-slice kernel where it applies (0: never)
    int slice_spw = 0;        // K-slice kernel: 256-column segments per warp (0: automatic, 1..3)
};

std::atomic<int> g_policy{MBGLU_POLICY_PREFETCH};

int env_int(const char *name, int dflt)
{
    const char *v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

const Tuning &tuning()
{
    static const Tuning t = [] {
        Tuning x;
        x.warps = std::min(mbglu::kMaxStreamWarps, std::max(0, env_int("MBGLU_WARPS", 0)));
        x.rows = env_int("MBGLU_ROWS", 0);
        if (x.rows != 1 && x.rows != 2 && x.rows != 4) x.rows = 0;
        x.ks = std::max(0, env_int("MBGLU_KS", 0)) & ~7;
        x.stages = std::min(kMaxStages, std::max(0, env_int("MBGLU_STAGES", 0)));
        x.smem_kb = std::max(0, env_int("MBGLU_SMEM_KB", 0));
        x.ctas_per_sm = std::min(2, std::max(0, env_int("MBGLU_CTAS_PER_SM", 0)));
        x.hreg = env_int("MBGLU_HREG", 1) != 0;
        x.waves = std::min(16, std::max(1, env_int("MBGLU_WAVES", 1)));
        x.interleave = env_int("MBGLU_INTERLEAVE", 0) != 0;
        x.mma_min_m = std::min(17, std::max(1, env_int("MBGLU_MMA_MIN_M", 3)));
        x.mma_ks_min = std::max(16, env_int("MBGLU_MMA_KS_MIN", 192));
        x.tma = env_int("MBGLU_TMA", 1) != 0;
        x.phases = std::min(2, std::max(0, env_int("MBGLU_PHASES", 0)));
        x.tc = env_int("MBGLU_TC", 1) != 0;
        x.tc_min_m = std::min(65, std::max(1, env_int("MBGLU_TC_MIN_M", 17)));
        x.tc_split = std::min(mbglu::kTcMaxSplit, std::max(0, env_int("MBGLU_TC_SPLIT", 0)));
        x.bwd_fused = env_int("MBGLU_BWD_FUSED", 1) != 0;
        x.bwd_mma_min_m = std::min(17, std::max(1, env_int("MBGLU_BWD_MMA_MIN_M", 3)));
        x.bwd_warps = std::min(mbglu::bwd_mma_warps(kBwdNB), std::max(0, env_int("MBGLU_BWD_WARPS", 0)));
        x.slice = env_int("MBGLU_SLICE", 1) != 0;
        x.slice_min_m = std::min(9, std::max(1, env_int("MBGLU_SLICE_MIN_M", 1)));
        x.slice16 = env_int("MBGLU_SLICE16", 1) != 0;
        x.slice_spw = std::min(3, std::max(0, env_int("MBGLU_SLICE_SPW", 0)));
        return x;
    }();
    return t;
}

mbglu_status cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return MBGLU_ERR_CUDA;
}

template <int MB, int R, bool NORM, bool HREG>
cudaError_t allow_smem(int optin)
{
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, mbglu::glu_stream_kernel<MB, R, NORM, HREG>);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mbglu::glu_stream_kernel<MB, R, NORM, HREG>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, optin - static_cast<int>(a.sharedSizeBytes));
}

// (MB, R, HREG) tiles instantiated: R * MB <= 16 keeps the accumulators in
// registers; h lives in registers only at batch 1.
#define MBGLU_FOR_EACH_TILE(X)                                                                          \
    X(1, 1, false) X(1, 2, false) X(1, 4, false) X(2, 1, false) X(2, 2, false) X(2, 4, false)         \
    X(4, 1, false) X(4, 2, false) X(4, 4, false) X(8, 1, false) X(8, 2, false) X(16, 1, false)        \
    X(1, 1, true) X(1, 2, true) X(1, 4, true)

cudaError_t allow_all_stream_kernels(int optin)
{
    cudaError_t e = cudaSuccess;
#define MBGLU_ALLOW(TMB, TR, TH)                                                  \
    if (e == cudaSuccess) e = allow_smem<TMB, TR, false, TH>(optin);              \
    if (e == cudaSuccess) e = allow_smem<TMB, TR, true, TH>(optin);
    MBGLU_FOR_EACH_TILE(MBGLU_ALLOW)
#undef MBGLU_ALLOW
    return e;
}

template <bool NORM>
cudaError_t allow_smem_mma(int optin)
{
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, mbglu::glu_mma_kernel<NORM>);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mbglu::glu_mma_kernel<NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - static_cast<int>(a.sharedSizeBytes));
}

cudaError_t allow_smem_generic(int optin)
{
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, mbglu::glu_generic_kernel<true>);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mbglu::glu_generic_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - static_cast<int>(a.sharedSizeBytes));
}

constexpr int kBwdHSmemMax = 96 * 1024;   // glu_bwd_w_kernel: h in shared memory up to this (two CTAs per SM)

cudaError_t allow_smem_bwd()
{
    cudaError_t e = cudaSuccess;
#define MBGLU_ALLOW_BWD(MB)                                                                                  \
    if (e == cudaSuccess)                                                                                    \
        e = cudaFuncSetAttribute(mbglu::glu_bwd_w_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 kBwdHSmemMax);
    MBGLU_ALLOW_BWD(1)
    MBGLU_ALLOW_BWD(2)
    MBGLU_ALLOW_BWD(4)
    MBGLU_ALLOW_BWD(8)
    MBGLU_ALLOW_BWD(16)
    MBGLU_ALLOW_BWD(32)
    MBGLU_ALLOW_BWD(64)
#undef MBGLU_ALLOW_BWD
    return e;
}

cudaError_t allow_smem_bwd_rows(int optin)
{
    cudaError_t e = cudaSuccess;
#define MBGLU_ALLOW_ROWS(TMB, TCPT)                                                                           \
    if (e == cudaSuccess)                                                                                     \
        e = cudaFuncSetAttribute(mbglu::glu_bwd_rows_kernel<TMB, TCPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 optin);
    MBGLU_ALLOW_ROWS(1, 1) MBGLU_ALLOW_ROWS(2, 1) MBGLU_ALLOW_ROWS(4, 1) MBGLU_ALLOW_ROWS(8, 1)
    MBGLU_ALLOW_ROWS(1, 2) MBGLU_ALLOW_ROWS(2, 2) MBGLU_ALLOW_ROWS(4, 2)
#undef MBGLU_ALLOW_ROWS
#define MBGLU_ALLOW_HW(TMB)                                                                                      \
    if (e == cudaSuccess)                                                                                        \
        e = cudaFuncSetAttribute(mbglu::glu_bwd_hw_kernel<TMB>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    MBGLU_ALLOW_HW(1) MBGLU_ALLOW_HW(2) MBGLU_ALLOW_HW(4) MBGLU_ALLOW_HW(8)
#undef MBGLU_ALLOW_HW
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mbglu::glu_bwd_mma_kernel<kBwdNB, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mbglu::glu_bwd_mma_kernel<kBwdNB, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin);
    return e;
}

cudaError_t allow_smem_slice(int optin)
{
    cudaError_t e = cudaSuccess;
#define MBGLU_ALLOW_SLICE(TS, TN, TMB)                                                                            \
    if (e == cudaSuccess) {                                                                                       \
        cudaFuncAttributes a{};                                                                                   \
        e = cudaFuncGetAttributes(&a, mbglu::glu_slice_kernel<TS, TN, TMB>);                                     \
        if (e == cudaSuccess)                                                                                     \
            e = cudaFuncSetAttribute(mbglu::glu_slice_kernel<TS, TN, TMB>,                                        \
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,                                 \
                                     optin - static_cast<int>(a.sharedSizeBytes));                               \
    }
    MBGLU_ALLOW_SLICE(1, false, 8) MBGLU_ALLOW_SLICE(2, false, 8) MBGLU_ALLOW_SLICE(3, false, 8)
    MBGLU_ALLOW_SLICE(1, true, 8) MBGLU_ALLOW_SLICE(2, true, 8) MBGLU_ALLOW_SLICE(3, true, 8)
    MBGLU_ALLOW_SLICE(1, false, 16)
#undef MBGLU_ALLOW_SLICE
    return e;
}

cudaError_t allow_smem_tc(int optin)
{
    return cudaFuncSetAttribute(mbglu::glu_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

mbglu_status device_info(const DeviceInfo **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        const cudaError_t errs[] = {allow_all_stream_kernels(d.smem_optin), allow_smem_mma<false>(d.smem_optin),
                                    allow_smem_mma<true>(d.smem_optin), allow_smem_generic(d.smem_optin),
                                    allow_smem_bwd(), allow_smem_bwd_rows(d.smem_optin),
                                    allow_smem_tc(d.smem_optin), allow_smem_slice(d.smem_optin)};
        for (cudaError_t x : errs)
            if (x != cudaSuccess) return cuda_fail(x);
        d.ready = true;
    }
    *out = &d;
    return MBGLU_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [p, p + bytes) and [q, q + bytes_q) intersect
bool overlaps(const void *p, int64_t bytes, const void *q, int64_t bytes_q)
{
    if (bytes <= 0 || bytes_q <= 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + static_cast<uintptr_t>(bytes_q) && b < a + static_cast<uintptr_t>(bytes);
}

int64_t matrix_bytes(int rows, int cols, int64_t ld)
{
    if (rows <= 0 || cols <= 0) return 0;
    return ((static_cast<int64_t>(rows) - 1) * ld + cols) * 2;
}

int batch_tile(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

// Rows per stage: whole rows of ~8 KB or more per bulk copy when the matrix
// rows are contiguous, bounded by R * MB <= 16 accumulators per kind.
int default_rows(int MB, int K, bool contiguous)
{
    const int rmax = MB >= 16 ? 1 : MB >= 8 ? 2 : 4;
    if (!contiguous) return 1;
    int r = 1;
    while (r < rmax && r * K * 2 < 8192) r *= 2;
    return r;
}

struct Plan {
    int MB = 1, R = 1, warps = 4, KS = 0, nseg = 0, stages = 0, grid = 0, ctas_per_sm = 1;
    bool hreg = false;
    uint32_t off_h = 0, off_s = 0, off_carry = 0, off_piece = 0, off_ring = 0, smem = 0;
    int nphase = 1, nsp = 0;   // tensor-core kernel: K staged in nphase phases of nsp segments
};

// Streaming-kernel plan.  Whole rows per stage (K-segments only if a stage of
// R rows does not fit), one CTA per SM, two stages per warp and as many warps
// (<= 8) as then fit: measured on GB300, more warps beat deeper per-warp
// rings (3-5 stages per warp ran 15-40% slower at equal ring bytes).  Rows
// per stage as default_rows, halved while not even one warp fits.  False if
// h plus a two-stage ring cannot fit.
bool plan_stream(const DeviceInfo &d, int M, int N, int K, bool contiguous, bool norm, Plan &pl,
                 bool allow_hreg = true, uint32_t extra = 0, int max_warps = mbglu::kMaxStreamWarps)
{
    const Tuning &t = tuning();
    pl.MB = batch_tile(M);
    pl.hreg = allow_hreg && t.hreg && pl.MB == 1 && K <= 32 * 8 * mbglu::kHregChunks;
    pl.ctas_per_sm = t.ctas_per_sm > 0 ? t.ctas_per_sm : 1;
    const int static_reserve = 2048;  // the kernel's static shared arrays
    // two co-resident CTAs share the SM's shared memory (1 KB of it is
    // reserved per CTA by the hardware)
    int budget = (pl.ctas_per_sm == 2 ? (d.smem_optin + 1024) / 2 - 1024 : d.smem_optin) - static_reserve;
    if (t.smem_kb > 0) budget = std::min(budget, t.smem_kb * 1024 - static_reserve);
    const bool need_hs = !pl.hreg || norm;
    const uint32_t hbytes =
        need_hs ? (static_cast<uint32_t>(pl.MB) * static_cast<uint32_t>(K) * 2u + 127u) & ~127u : 0u;
    const int64_t room = static_cast<int64_t>(budget) - kBarRegion - hbytes - extra;
    if (room <= 0) return false;
    int ks = t.ks > 0 ? std::min(t.ks, ((K + 7) / 8) * 8) : ((K + 7) / 8) * 8;
    pl.R = t.rows > 0 ? t.rows : default_rows(pl.MB, K, contiguous);
    if (pl.R * pl.MB > 16) pl.R = pl.MB >= 16 ? 1 : 16 / pl.MB;
    for (;;) {
        const int64_t stage = static_cast<int64_t>(pl.R) * 4 * ks;
        int best_w = 0, best_s = 0;
        int64_t best_ring = 0;
        const int want_s = t.stages > 0 ? t.stages : 2;
        for (int w = 1; w <= max_warps; ++w) {
            if (t.warps > 0 && w != std::min(t.warps, max_warps)) continue;
            const int sn = static_cast<int>(std::min<int64_t>(want_s, room / (stage * w)));
            if (sn < 2) continue;
            const int64_t ring = stage * w * sn;
            if (ring >= best_ring) {
                best_ring = ring;
                best_w = w;
                best_s = sn;
            }
        }
        if (best_w > 0) {
            pl.warps = best_w;
            pl.stages = best_s;
            break;
        }
        if (pl.R > 1) {
            pl.R /= 2;
            continue;
        }
        if (ks <= 256) return false;
        ks = std::max(256, (ks / 2) & ~7);
    }
    pl.KS = ks;
    pl.nseg = (K + ks - 1) / ks;
    if (pl.hreg && pl.nseg != 1)   // registers hold whole rows of h only
        return plan_stream(d, M, N, K, contiguous, norm, pl, false, extra, max_warps);
    pl.off_h = kBarRegion;
    pl.off_s = kBarRegion + hbytes;
    pl.off_ring = kBarRegion + hbytes + extra;
    pl.smem = pl.off_ring + static_cast<uint32_t>(pl.warps) * pl.stages * 4u * pl.R * static_cast<uint32_t>(ks);
    pl.grid = std::max(1, std::min(d.sm_count * pl.ctas_per_sm * t.waves, N));
    return true;
}

// Tensor-core plan (batch >= mma_min_m, K % 16 == 0): groups of 8 rows, each
// row of a stage padded by 16 bytes; h_s holds M rows plus a zero row (none at
// M = 16, where every A row is real); 2 KB
// per warp for handed-off accumulators; two stages per warp.  For each warp
// count the longest K-segment (multiple of 16, <= 240: the tensor copy's box
// is KS + 8 <= 256 elements wide) that fits is taken;
// the plan is the most warps whose segment is still >= mma_ks_min elements
// (measured on GB300: at equal ring bytes more warps win, while row copies
// under 512 bytes lose), else the warp count with the largest ring.
// Segments are then evened out over K.  False if nothing fits.
// Warp count and K-segment for `room` bytes of hand-off slots and rings: for
// each warp count the longest segment that fits; the most warps whose
// segment is >= mma_ks_min, else the largest ring.  False if nothing fits.
bool choose_mma_ring(int K, int64_t room, int max_warps, int &w_out, int &ks_out, int64_t &ring_out)
{
    const Tuning &t = tuning();
    const int want_s = t.stages > 0 ? t.stages : 2;
    const int64_t piece = mbglu::kPieceBytes;
    const int64_t row_unit = 2 * mbglu::kMmaRows * 2;   // stage bytes per padded element of a row
    const int ks_cap = std::min(kMmaKsCap, K);
    int64_t best_ring = 0;
    int ks_of[mbglu::kMaxStreamWarps + 1] = {};
    int64_t ring_of[mbglu::kMaxStreamWarps + 1] = {};
    if (room <= 0) return false;
    for (int w = 1; w <= max_warps; ++w) {
        if (t.warps > 0 && w != std::min(t.warps, max_warps)) continue;
        const int64_t per_stage = (room / w - piece) / want_s;
        int ks = static_cast<int>(std::min<int64_t>(ks_cap, (per_stage / row_unit - 8) & ~int64_t{15}));
        if (t.ks > 0) ks = (std::min(t.ks, K) & ~15) <= ks ? (std::min(t.ks, K) & ~15) : 0;
        if (ks < 16) continue;
        ks_of[w] = ks;
        ring_of[w] = static_cast<int64_t>(w) * want_s * row_unit * (ks + 8);
        if (ring_of[w] > best_ring) best_ring = ring_of[w];
    }
    if (best_ring == 0) return false;
    int best_w = 0;
    for (int w = max_warps; w >= 1 && best_w == 0; --w)
        if (ring_of[w] > 0 && ks_of[w] >= std::min(t.mma_ks_min, ks_cap)) best_w = w;
    for (int w = max_warps; w >= 1 && best_w == 0; --w)
        if (ring_of[w] == best_ring) best_w = w;
    int ks = ks_of[best_w];
    if (t.ks <= 0) {   // even the segments out: same count, lengths within 16
        const int nseg = (K + ks - 1) / ks;
        ks = ((K + nseg - 1) / nseg + 15) & ~15;
    }
    w_out = best_w;
    ks_out = ks;
    ring_out = ring_of[best_w];
    return true;
}

// Tensor-core plan (batch >= mma_min_m, K % 16 == 0): groups of 8 rows, each
// row of a stage padded by 16 bytes; h_s holds M rows plus a zero row (none at
// M = 16, where every A row is real); 2 KB per warp for handed-off
// accumulators; two stages per warp (choose_mma_ring).  Measured on GB300: at
// equal ring bytes more warps win, row copies under 512 bytes lose.
// K-phases (allow_phases: plain GEMV with 16-byte aligned h): h_s holds about
// half of K, plus 2 KB per group for the accumulators carried between the
// phases; taken where that ring is >= 1.25x the one-phase ring (the phase
// boundary costs a copy of h from L2), e.g. M = 16, K = 4096.  False if
// nothing fits.
bool plan_mma(const DeviceInfo &d, int M, int N, int K, Plan &pl, uint32_t extra = 0,
              int max_warps = mbglu::kMaxStreamWarps, bool allow_phases = false)
{
    const Tuning &t = tuning();
    if (M < t.mma_min_m || K % 16 != 0) return false;
    const int static_reserve = 2048;
    int budget = d.smem_optin - static_reserve;
    if (t.smem_kb > 0) budget = std::min(budget, t.smem_kb * 1024 - static_reserve);
    const uint32_t hrows = static_cast<uint32_t>(M < mbglu::kMaxM ? M + 1 : M);   // + the zero row below 16
    auto h_bytes = [&](int width) -> uint32_t {
        return (hrows * static_cast<uint32_t>(width + 8) * 2u + 127u) & ~127u;
    };
    const int grid = std::max(1, std::min(d.sm_count, N));

    int w1 = 0, ks1 = 0;
    int64_t ring1 = 0;
    const bool ok1 = choose_mma_ring(K, static_cast<int64_t>(budget) - kBarRegion - h_bytes(K) - extra, max_warps,
                                     w1, ks1, ring1);
    int w2 = 0, ks2 = 0, nsp2 = 0;
    int64_t ring2 = 0;
    uint32_t carry2 = 0;
    bool ok2 = false;
    if (allow_phases && t.phases != 1 && extra == 0 && K >= 2 * 16) {
        const int half = ((K + 1) / 2 + 15) & ~15;
        const int64_t groups = t.interleave ? ((N + mbglu::kMmaRows - 1) / mbglu::kMmaRows + grid - 1) / grid
                                            : ((N + grid - 1) / grid + mbglu::kMmaRows - 1) / mbglu::kMmaRows;
        carry2 = static_cast<uint32_t>(groups) * mbglu::kPieceBytes;
        // h_s is reserved for half of K plus up to one segment (phases end on segment boundaries)
        ok2 = choose_mma_ring(K, static_cast<int64_t>(budget) - kBarRegion - h_bytes(half + kMmaKsCap) - carry2,
                              max_warps, w2, ks2, ring2);
        if (ok2) {
            nsp2 = (half + ks2 - 1) / ks2;
            const int nseg2 = (K + ks2 - 1) / ks2;
            ok2 = nsp2 < nseg2 && (nseg2 + nsp2 - 1) / nsp2 <= mbglu::kMaxPhases;
        }
    }
    const bool two = ok2 && (!ok1 || t.phases == 2 || ring2 * 4 >= ring1 * 5);
    if (!ok1 && !two) return false;
    pl.warps = two ? w2 : w1;
    pl.stages = t.stages > 0 ? t.stages : 2;
    pl.KS = two ? ks2 : ks1;
    pl.MB = 16;
    pl.R = mbglu::kMmaRows;
    pl.nseg = (K + pl.KS - 1) / pl.KS;
    pl.nsp = two ? nsp2 : pl.nseg;
    pl.nphase = (pl.nseg + pl.nsp - 1) / pl.nsp;
    const int hw = std::min(K, pl.nsp * pl.KS);   // h_s columns
    pl.off_h = kBarRegion;
    pl.off_s = kBarRegion + h_bytes(hw);
    pl.off_carry = pl.off_s + extra;
    pl.off_piece = pl.off_carry + (pl.nphase > 1 ? carry2 : 0u);
    pl.off_ring = pl.off_piece + static_cast<uint32_t>(pl.warps) * mbglu::kPieceBytes;
    pl.smem = pl.off_ring + static_cast<uint32_t>(pl.warps) * pl.stages * 2u * mbglu::kMmaRows *
                                static_cast<uint32_t>(pl.KS + 8) * 2u;
    pl.grid = grid;
    return true;
}

template <typename... Args>
mbglu_status launch(void (*kernel)(Args...), dim3 grid, dim3 block, uint32_t smem, cudaStream_t stream,
                    bool pdl, const GluParams &p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

mbglu_status launch_mma(void (*kernel)(GluParams, mbglu::MmaMaps), dim3 grid, dim3 block, uint32_t smem,
                        cudaStream_t stream, bool pdl, const GluParams &p, const mbglu::MmaMaps &maps)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p, maps);
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link against libcuda); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Tiled 2-D descriptor of a bf16 [rows][K] matrix with row stride ld, box
// box_k x box_rows; elements past K or rows read as zero.  False if the
// driver rejects it (the caller then takes a path without tensor copies).
// The last 64 descriptors this thread encoded are kept
// (direct-mapped on their arguments): a descriptor holds only the address,
// the shape and the strides, so a kept one is exactly what encoding again
// would give, whatever the memory holds now.
bool encode_2d(mbglu::TensorMap *out, const void *base, int64_t ld, int rows, int K, int box_k, int box_rows,
               CUtensorMapSwizzle swizzle)
{
    static_assert(sizeof(CUtensorMap) == sizeof(mbglu::TensorMap), "tensor map size");
    struct Entry {
        const void *base = nullptr;
        int64_t ld = 0;
        int rows = 0, K = 0, box_k = 0, box_rows = 0, swizzle = -1;
        mbglu::TensorMap map;
    };
    thread_local Entry cache[64];
    const uint64_t hsh = (reinterpret_cast<uintptr_t>(base) >> 8) ^ (static_cast<uint64_t>(ld) * 0x9e3779b1u) ^
                         (static_cast<uint64_t>(rows) << 7) ^ (static_cast<uint64_t>(K) << 17) ^
                         (static_cast<uint64_t>(box_rows) << 3) ^ static_cast<uint64_t>(swizzle);
    Entry &e = cache[(hsh ^ (hsh >> 6) ^ (hsh >> 12)) & 63u];
    if (e.base == base && e.ld == ld && e.rows == rows && e.K == K && e.box_k == box_k && e.box_rows == box_rows &&
        e.swizzle == static_cast<int>(swizzle)) {
        *out = e.map;
        return true;
    }
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn || box_k > 256 || box_rows < 1 || box_rows > 256) return false;
    CUtensorMap m;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem_strides[2] = {1u, 1u};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::memcpy(out, &m, sizeof m);
    e.base = base;
    e.ld = ld;
    e.rows = rows;
    e.K = K;
    e.box_k = box_k;
    e.box_rows = box_rows;
    e.swizzle = static_cast<int>(swizzle);
    e.map = *out;
    return true;
}

bool encode_box_map(mbglu::TensorMap *out, const void *base, int64_t ld, int N, int K, int box_k, int box_rows)
{
    return encode_2d(out, base, ld, N, K, box_k, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_weight_map(mbglu::TensorMap *out, const void *base, int64_t ld, int N, int K, int box_k)
{
    return encode_box_map(out, base, ld, N, K, box_k, mbglu::kMmaRows);
}

// Both weight descriptors for a tensor-core launch; p.tma says whether they
// are used.
mbglu::MmaMaps weight_maps(GluParams &p)
{
    mbglu::MmaMaps maps = {};
    p.tma = (tuning().tma && encode_weight_map(&maps.gate, p.gate, p.ld_gate, p.N, p.K, p.KS + 8) &&
             encode_weight_map(&maps.up, p.up, p.ld_up, p.N, p.K, p.KS + 8))
                ? 1
                : 0;
    return maps;
}

template <bool NORM>
mbglu_status launch_stream(const Plan &pl, const GluParams &p, cudaStream_t stream, bool pdl)
{
    const dim3 grid(pl.grid), block((pl.warps + (p.helper_warp >= 0 ? 1 : 0)) * 32);
#define MBGLU_CASE(TMB, TR, TH)                                                                               \
    if (pl.MB == TMB && pl.R == TR && pl.hreg == TH)                                                             \
        return launch(mbglu::glu_stream_kernel<TMB, TR, NORM, TH>, grid, block, pl.smem, stream, pdl, p);
    MBGLU_FOR_EACH_TILE(MBGLU_CASE)
#undef MBGLU_CASE
    return MBGLU_ERR_SHAPE;  // unreachable: plan_stream only produces listed tiles
}

int generic_grid(const DeviceInfo &d, int N) { return std::max(1, std::min(d.sm_count * 4, (N + 7) / 8)); }

GluParams base_params(int M, int N, int K, int mode)
{
    GluParams p = {};
    p.helper_warp = -1;
    p.nphase = 1;   // the tensor-core planner sets its phases
    p.M = M;
    p.N = N;
    p.K = K;
    p.mode = mode;
    return p;
}

}  // namespace

extern "C" {

int mbglu_abi_version(void) { return MBGLU_ABI_VERSION; }

mbglu_status mbglu_set_launch_policy(int policy)
{
    if (policy != MBGLU_POLICY_SERIAL && policy != MBGLU_POLICY_PDL && policy != MBGLU_POLICY_PREFETCH)
        return MBGLU_ERR_MODE;
    g_policy.store(policy, std::memory_order_relaxed);
    return MBGLU_OK;
}

int mbglu_get_launch_policy(void) { return g_policy.load(std::memory_order_relaxed); }
int mbglu_last_cuda_error(void) { return t_last_cuda_error; }
int mbglu_last_variant(void) { return t_last_variant; }

int mbglu_last_single_kernel_blocks(void) { return t_last_single; }

int mbglu_last_backward_path(void) { return t_last_bwd; }

mbglu_status gdn_gates(const mbglu_bf16 *a, int64_t lda, const mbglu_bf16 *b, int64_t ldb, const float *A_log,
                       const float *dt_bias, float *g, int64_t ldg, mbglu_bf16 *beta, int64_t ldbeta, int T, int H,
                       cudaStream_t stream)
{
    t_last_variant = kNone;
    if (T < 0 || H < 0) return MBGLU_ERR_SHAPE;
    if (T == 0 || H == 0) return MBGLU_OK;
    if (!a || !b || !A_log || !dt_bias || !g || !beta) return MBGLU_ERR_NULL;
    if (lda < H || ldb < H || ldg < H || ldbeta < H) return MBGLU_ERR_STRIDE;
    if (!aligned(a, 2) || !aligned(b, 2) || !aligned(beta, 2) || !aligned(A_log, 4) || !aligned(dt_bias, 4) ||
        !aligned(g, 4))
        return MBGLU_ERR_ALIGN;
    const int64_t ab = matrix_bytes(T, H, lda), bb = matrix_bytes(T, H, ldb), betab = matrix_bytes(T, H, ldbeta);
    const int64_t gbytes = matrix_bytes(T, H, ldg) * 2, pb = static_cast<int64_t>(H) * 4;   // fp32: twice bf16's
    const void *ins[4] = {a, b, A_log, dt_bias};
    const int64_t inb[4] = {ab, bb, pb, pb};
    for (int k = 0; k < 4; ++k)
        if (overlaps(g, gbytes, ins[k], inb[k]) || overlaps(beta, betab, ins[k], inb[k])) return MBGLU_ERR_ALIAS;
    if (overlaps(g, gbytes, beta, betab)) return MBGLU_ERR_ALIAS;
    const DeviceInfo *d = nullptr;
    mbglu_status st = device_info(&d);
    if (st != MBGLU_OK) return st;
    const int policy = g_policy.load(std::memory_order_relaxed);
    // (token, 8 heads) per thread where the heads fit shared memory and the
    // item count 32 bits; one element per thread otherwise
    const int64_t chunks = static_cast<int64_t>(T) * ((H + 7) / 8);
    const bool by_chunk = H <= mbglu::kGdnMaxHeads && chunks < (int64_t{1} << 31);
    const int vec = H % 8 == 0 && aligned(a, 16) && aligned(b, 16) && aligned(g, 16) && aligned(beta, 16) &&
                    lda % 8 == 0 && ldb % 8 == 0 && ldg % 4 == 0 && ldbeta % 8 == 0;
    const int64_t work = by_chunk ? chunks : static_cast<int64_t>(T) * H;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(d->sm_count) * 8,
                                                                            (work + 255) / 256)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = policy != MBGLU_POLICY_SERIAL ? 1 : 0;
    const uint16_t *a16 = reinterpret_cast<const uint16_t *>(a), *b16 = reinterpret_cast<const uint16_t *>(b);
    uint16_t *beta16 = reinterpret_cast<uint16_t *>(beta);
    const cudaError_t e =
        by_chunk ? cudaLaunchKernelEx(&cfg, mbglu::gdn_gates_chunk_kernel, a16, lda, b16, ldb, A_log, dt_bias, g, ldg,
                                      beta16, ldbeta, T, H, vec)
                 : cudaLaunchKernelEx(&cfg, mbglu::gdn_gates_kernel, a16, lda, b16, ldb, A_log, dt_bias, g, ldg,
                                      beta16, ldbeta, T, H);
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_variant = kGdnGates;
    return MBGLU_OK;
}

mbglu_status silu_mul(const mbglu_bf16 *x, int64_t ldx, mbglu_bf16 *out, int64_t ldo, int M, int N,
                      mbglu_mode mode, cudaStream_t stream)
{
    t_last_variant = kNone;
    if (mode != MBGLU_MODE_FUSED && mode != MBGLU_MODE_HF) return MBGLU_ERR_MODE;
    if (M < 0 || N < 0 || N > INT32_MAX / 2) return MBGLU_ERR_SHAPE;   // 2N columns must fit an int
    if (M == 0 || N == 0) return MBGLU_OK;
    if (!x || !out) return MBGLU_ERR_NULL;
    if (ldx < 2 * static_cast<int64_t>(N) || ldo < N) return MBGLU_ERR_STRIDE;
    if (!aligned(x, 2) || !aligned(out, 2)) return MBGLU_ERR_ALIGN;
    if (overlaps(out, matrix_bytes(M, N, ldo), x, matrix_bytes(M, 2 * N, ldx)))
        return MBGLU_ERR_ALIAS;
    const DeviceInfo *d = nullptr;
    mbglu_status st = device_info(&d);
    if (st != MBGLU_OK) return st;
    const int policy = g_policy.load(std::memory_order_relaxed);
    const int vec = aligned(x, 16) && aligned(out, 16) && N % 8 == 0 && ldx % 8 == 0 && ldo % 8 == 0;
    const int64_t work = vec ? static_cast<int64_t>(M) * (N / 8) : static_cast<int64_t>(M) * N;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(d->sm_count) * 8,
                                                                            (work + 255) / 256)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = policy != MBGLU_POLICY_SERIAL ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mbglu::silu_mul_kernel, reinterpret_cast<const uint16_t *>(x), ldx,
                                             reinterpret_cast<uint16_t *>(out), ldo, M, N, static_cast<int>(mode), vec);
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_variant = kSiluMul;
    return MBGLU_OK;
}

const char *mbglu_status_string(mbglu_status s)
{
    switch (s) {
    case MBGLU_OK: return "MBGLU_OK";
    case MBGLU_ERR_NULL: return "MBGLU_ERR_NULL: a required pointer is NULL";
    case MBGLU_ERR_SHAPE: return "MBGLU_ERR_SHAPE: unsupported M, N or K";
    case MBGLU_ERR_STRIDE: return "MBGLU_ERR_STRIDE: a leading dimension is smaller than its row";
    case MBGLU_ERR_ALIGN: return "MBGLU_ERR_ALIGN: a pointer is not 2-byte aligned";
    case MBGLU_ERR_MODE: return "MBGLU_ERR_MODE: mode must be MBGLU_MODE_FUSED or MBGLU_MODE_HF";
    case MBGLU_ERR_ALIAS: return "MBGLU_ERR_ALIAS: an output overlaps an input";
    case MBGLU_ERR_CUDA: return "MBGLU_ERR_CUDA: a CUDA runtime call failed";
    case MBGLU_ERR_TIMEOUT: return "MBGLU_ERR_TIMEOUT: a bounded device-side wait gave up";
    default: return "unknown mbglu status";
    }
}

}  // extern "C"

namespace {

// Every argument check of glu_gemv, on the whole call: nothing launches when
// one fails.
mbglu_status check_gemv(const mbglu_bf16 *h, int64_t ldh, const mbglu_bf16 *gate_w, int64_t ld_gate,
                        const mbglu_bf16 *up_w, int64_t ld_up, const mbglu_bf16 *out, int64_t ldo, int M, int N,
                        int K, mbglu_mode mode)
{
    if (mode != MBGLU_MODE_FUSED && mode != MBGLU_MODE_HF) return MBGLU_ERR_MODE;
    if (M < 0 || N < 0 || K < 0 || M > MBGLU_MAX_M) return MBGLU_ERR_SHAPE;
    if (M == 0 || N == 0) return MBGLU_OK;
    if (!out || (K > 0 && (!h || !gate_w || !up_w))) return MBGLU_ERR_NULL;
    if (ldo < N || (K > 0 && (ldh < K || ld_gate < K || ld_up < K))) return MBGLU_ERR_STRIDE;
    if (!aligned(out, 2) || (K > 0 && (!aligned(h, 2) || !aligned(gate_w, 2) || !aligned(up_w, 2))))
        return MBGLU_ERR_ALIGN;
    const int64_t ob = matrix_bytes(M, N, ldo);
    if (K > 0 && (overlaps(out, ob, h, matrix_bytes(M, K, ldh)) || overlaps(out, ob, gate_w, matrix_bytes(N, K, ld_gate)) ||
                  overlaps(out, ob, up_w, matrix_bytes(N, K, ld_up))))
        return MBGLU_ERR_ALIAS;
    return MBGLU_OK;
}

// The backward's first step: the GEMV kernels' epilogue writes dG, dU
// (fp32 [M][N]) from dout instead of out.
struct BwdEpilogue {
    const mbglu_bf16 *dout;
    int64_t ldd;
    float *dG, *dU;
};

// The GEMV on 1 <= M <= kBlockRows rows, N >= 1, arguments already checked.
// bwd != nullptr: K >= 1, and the epilogue is the backward's (out unused).
// Plan of glu_slice_kernel (batch 1..8, K >= 256): K in segments of
// 256 columns, SPW per compute warp (h's fragments for them in registers:
// 32 SPW per lane), W = ceil(segments / SPW) compute warps plus the epilogue
// warp; one CTA per SM over balanced row shares; as many stages per warp
// (2..6) as fit.  The smallest SPW that fits: more warps, each with a shorter
// chain of dependent steps, beat deeper rings (K2560, M = 4: 16.0 us at SPW 1
// with 2 stages, 18.0 at SPW 2 with 5).  Below mma_min_m rows only SPW 1: at
// M = 1-2 it beats the CUDA-core streaming kernel (K2560 N9728, M = 1: 16.18
// against 16.58 us), but SPW 2 does not (K4096: 36.8 against 35.2 us).
bool encode_sw128_map(mbglu::TensorMap *out, const void *base, int64_t ld, int rows, int K, int box_rows);

struct SlicePlan {
    int spw = 1, warps = 1, stages = 0, grid = 1, mb = 8;
    uint32_t off_s = 0, off_ring = 0, smem = 0;
};

// Shared-memory layout and ring depth of one candidate; false if fewer than
// two stages fit.
bool slice_layout(const DeviceInfo &d, int M, int K, bool norm, SlicePlan &c)
{
    const int W = c.warps;
    uint32_t region = static_cast<uint32_t>(mbglu::slice_slots(c.mb)) * static_cast<uint32_t>(W) *
                      mbglu::slice_slot_bytes(c.mb);
    if (norm) region = std::max(region, static_cast<uint32_t>(M) * static_cast<uint32_t>(K + 8) * 2u);
    c.off_s = (1024u + region + 127u) & ~127u;
    uint32_t end = c.off_s;
    if (norm) end = c.off_s + ((static_cast<uint32_t>(K) * 2u + 127u) & ~127u) + 2u * 32u * (W + 1) * 4u;
    c.off_ring = (end + 1023u) & ~1023u;
    // 1024: the base's alignment; 256: the kernel's static shared memory (inv_s)
    const int64_t room = static_cast<int64_t>(d.smem_optin) - 1024 - 256 - c.off_ring;
    if (room <= 0) return false;
    c.stages = static_cast<int>(
        std::min<int64_t>({6, room / (static_cast<int64_t>(W) * mbglu::kSliceStage), 64 / W}));
    if (c.stages < 2) return false;
    c.smem = c.off_ring + static_cast<uint32_t>(W * c.stages) * mbglu::kSliceStage + 1024u;
    return true;
}

// norm: the add_rmsnorm_glu variant, whose h_s[M][K + 8] shares the slots'
// region and whose norm_w and statistic partials follow it at off_s; from
// mma_min_m rows (K2560 N9728 single kernel: M = 4 21.7 against 22.2 us,
// M = 8 23.5 against 24.0; at M = 1 the streaming kernel's 19.6 against 20.6).
// Batch 9..16 (MB = 16, not with the norm): one segment per warp, up to 10
// warps (K2560 N9728 M = 16: 18.5 against 19.9 us).  A cluster pair that
// split K for larger K measured slower than the kernel with h in shared
// memory (K4096 N14336 M = 16: 51.6 against 49.7 us), so K past 2560 stays
// there.
bool plan_slice(const DeviceInfo &d, int M, int N, int K, SlicePlan &sp, bool norm = false)
{
    const Tuning &t = tuning();
    if (!t.slice || M < (norm ? t.mma_min_m : t.slice_min_m) || M > mbglu::kMaxM || K < mbglu::kSliceSeg ||
        K % 8 != 0 || N < 1)
        return false;
    const int nseg = (K + mbglu::kSliceSeg - 1) / mbglu::kSliceSeg;
    if (M > 8) {
        if (norm || !t.slice16) return false;
        SlicePlan c;
        c.mb = 16;
        c.warps = nseg;
        if (c.warps > mbglu::slice_max_warps(1, 16) || !slice_layout(d, M, K, false, c)) return false;
        c.grid = std::max(1, std::min(d.sm_count, (N + 7) / 8));
        sp = c;
        return true;
    }
    const int spw_max = M < t.mma_min_m ? 1 : 3;
    for (int spw = 1; spw <= spw_max; ++spw) {
        if (t.slice_spw && spw != t.slice_spw) continue;
        const int W = (nseg + spw - 1) / spw;
        if (W > mbglu::slice_max_warps(spw) || (W - 1) * spw >= nseg) continue;
        SlicePlan c;
        c.spw = spw;
        c.warps = W;
        if (!slice_layout(d, M, K, norm, c)) continue;
        c.grid = std::max(1, std::min(d.sm_count, (N + 7) / 8));
        sp = c;
        return true;
    }
    return false;
}

template <bool NORM>
mbglu_status launch_slice(const SlicePlan &sp, const GluParams &p, const mbglu::SliceMaps &maps,
                          cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sp.grid);
    cfg.blockDim = dim3(32 * (sp.warps + 1));
    cfg.dynamicSmemBytes = sp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaErrorInvalidValue;
    if (sp.mb > 8) {
        if constexpr (!NORM) e = cudaLaunchKernelEx(&cfg, mbglu::glu_slice_kernel<1, false, 16>, p, maps);
    } else {
        switch (sp.spw) {
            case 1: e = cudaLaunchKernelEx(&cfg, mbglu::glu_slice_kernel<1, NORM, 8>, p, maps); break;
            case 2: e = cudaLaunchKernelEx(&cfg, mbglu::glu_slice_kernel<2, NORM, 8>, p, maps); break;
            default: e = cudaLaunchKernelEx(&cfg, mbglu::glu_slice_kernel<3, NORM, 8>, p, maps); break;
        }
    }
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

mbglu_status gemv_block(const mbglu_bf16 *h, int64_t ldh, const mbglu_bf16 *gate_w, int64_t ld_gate,
                        const mbglu_bf16 *up_w, int64_t ld_up, mbglu_bf16 *out, int64_t ldo, int M, int N, int K,
                        mbglu_mode mode, cudaStream_t stream, const BwdEpilogue *bwd = nullptr)
{
    const DeviceInfo *d = nullptr;
    mbglu_status st = device_info(&d);
    if (st != MBGLU_OK) return st;
    const int policy = g_policy.load(std::memory_order_relaxed);
    const bool pdl = policy != MBGLU_POLICY_SERIAL;

    GluParams p = base_params(M, N, K, static_cast<int>(mode));
    p.prefetch = policy == MBGLU_POLICY_PREFETCH;
    p.out = out;
    p.ldo = ldo;
    if (bwd) {
        p.mode = mbglu::kModeBwd;
        p.dout = bwd->dout;
        p.ldd = bwd->ldd;
        p.dG = bwd->dG;
        p.dU = bwd->dU;
    }
    if (K == 0) {
        const int grid = std::max(1, std::min(d->sm_count, static_cast<int>((static_cast<int64_t>(M) * N + 255) / 256)));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, mbglu::zero_fill_kernel, reinterpret_cast<uint16_t *>(out),
                                                 ldo, M, N);
        if (e != cudaSuccess) return cuda_fail(e);
        t_last_variant = kZeroFill;
        return MBGLU_OK;
    }
    p.h = h;
    p.ldh = ldh;
    p.gate = gate_w;
    p.ld_gate = ld_gate;
    p.up = up_w;
    p.ld_up = ld_up;

    Plan pl;
    const bool bulk_ok = (K % 8 == 0) && aligned(gate_w, 16) && aligned(up_w, 16) && (ld_gate % 8 == 0) &&
                         (ld_up % 8 == 0);
    const bool h_vec = aligned(h, 16) && (ldh % 8 == 0);
    SlicePlan sp;
    mbglu::SliceMaps smaps;
    if (bulk_ok && plan_slice(*d, M, N, K, sp) && encode_sw128_map(&smaps.gate, gate_w, ld_gate, N, K, 8) &&
        encode_sw128_map(&smaps.up, up_w, ld_up, N, K, 8)) {
        p.stages = sp.stages;
        p.off_ring = sp.off_ring;
        p.vec_in = h_vec;
        st = launch_slice<false>(sp, p, smaps, stream, pdl);
        if (st == MBGLU_OK) t_last_variant = kSlice;
        return st;
    }
    if (bulk_ok && plan_mma(*d, M, N, K, pl, 0, mbglu::kMaxStreamWarps, h_vec)) {
        p.KS = pl.KS;
        p.nseg = pl.nseg;
        p.nphase = pl.nphase;
        p.nsp = pl.nsp;
        p.stages = pl.stages;
        p.off_h = pl.off_h;
        p.off_ring = pl.off_ring;
        p.off_piece = pl.off_piece;
        p.off_carry = pl.off_carry;
        p.vec_in = h_vec;
        p.interleave = tuning().interleave;
        const mbglu::MmaMaps maps = weight_maps(p);
        st = launch_mma(mbglu::glu_mma_kernel<false>, dim3(pl.grid), dim3(pl.warps * 32), pl.smem, stream, pdl, p,
                        maps);
        if (st == MBGLU_OK) t_last_variant = kTensor;
        return st;
    }
    const bool fast = bulk_ok && plan_stream(*d, M, N, K, ld_gate == K && ld_up == K, false, pl);
    if (fast) {
        p.KS = pl.KS;
        p.nseg = pl.nseg;
        p.stages = pl.stages;
        p.off_h = pl.off_h;
        p.off_ring = pl.off_ring;
        p.vec_in = aligned(h, 16) && (ldh % 8 == 0);
        p.interleave = tuning().interleave;
        st = launch_stream<false>(pl, p, stream, pdl);
        if (st == MBGLU_OK) t_last_variant = kStream;
        return st;
    }
    st = launch(mbglu::glu_generic_kernel<false>, dim3(generic_grid(*d, N)), dim3(256), 0, stream, pdl, p);
    if (st == MBGLU_OK) t_last_variant = kGeneric;
    return st;
}

// ---- the tcgen05 kernel (batch 17..64 in one pass) ----------------------------

// A 2-D bf16 tensor map [rows][K] (row stride ld elements) with a box of 64 x
// box_rows elements in the 128-byte swizzled layout; rows and columns past the
// tensor arrive as zeros.
bool encode_sw128_map(mbglu::TensorMap *out, const void *base, int64_t ld, int rows, int K, int box_rows)
{
    return encode_2d(out, base, ld, rows, K, mbglu::kTcBox, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

struct TcPlan {
    int Np = 0, nchunk = 0, ntiles = 0, ksplit = 1, stages = 0;
    uint32_t smem = 0;
};

// Batch rows padded to a multiple of 16 (the MMA's N), 64-wide K chunks,
// 128-row tiles; the K split (CTAs per tile, 1..4) that makes the longest
// per-SM queue of work shortest (tiles * split CTAs in waves over the SMs),
// the smaller one on a tie, with at least 2 chunks per CTA; as many stages
// as fit, 2..8.  With a split of s, rank 0's stages must also hold the other
// ranks' partial sums, (s - 1) x 2 Np x 128 fp32.
bool plan_tc(const DeviceInfo &d, int M, int N, int K, TcPlan &pl)
{
    if (M < 1 || M > MBGLU_MAX_M || N < 1 || K < 1) return false;
    pl.Np = (M + 15) / 16 * 16;
    pl.nchunk = (K + mbglu::kTcChunk - 1) / mbglu::kTcChunk;
    pl.ntiles = (N + mbglu::kTcRows - 1) / mbglu::kTcRows;
    const uint32_t sbytes = 2 * mbglu::kTcWBytes + static_cast<uint32_t>(pl.Np) * 128u * mbglu::kTcBoxes;
    const int64_t room = static_cast<int64_t>(d.smem_optin) - mbglu::kTcHeader - mbglu::kTcSmemSlack;
    pl.stages = static_cast<int>(std::min<int64_t>(mbglu::kTcMaxStages, room / sbytes));
    if (pl.stages < 2) return false;
    auto span = [&](int ks) {   // per-SM time in units of one full-K tile
        const int64_t ctas = static_cast<int64_t>(pl.ntiles) * ks;
        return static_cast<double>((ctas + d.sm_count - 1) / d.sm_count) / ks;
    };
    auto allowed = [&](int ks) {
        return pl.nchunk >= 2 * ks && (ks - 1) * 4LL * mbglu::kTcRows * mbglu::tc_part_pitch(pl.Np) <= room;
    };
    pl.ksplit = 1;
    for (int ks = 2; ks <= mbglu::kTcMaxSplit; ++ks)
        if (allowed(ks) && span(ks) < span(pl.ksplit)) pl.ksplit = ks;
    if (tuning().tc_split > 0 && (tuning().tc_split == 1 || allowed(tuning().tc_split))) pl.ksplit = tuning().tc_split;
    // rank 0's stage memory also takes the other ranks' partial sums after its MMAs
    const int64_t parts = (pl.ksplit - 1) * 4LL * mbglu::kTcRows * mbglu::tc_part_pitch(pl.Np);
    pl.smem = mbglu::kTcHeader + mbglu::kTcSmemSlack +
              static_cast<uint32_t>(std::max<int64_t>(static_cast<int64_t>(pl.stages) * sbytes, parts));
    return true;
}

mbglu_status launch_tc(const TcPlan &pl, const mbglu::TcParams &p, const mbglu::TcMaps &maps, cudaStream_t stream,
                       bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.ntiles * pl.ksplit));
    cfg.blockDim = dim3(mbglu::kTcThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (pl.ksplit > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(pl.ksplit);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mbglu::glu_tc_kernel, p, maps);
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

// The batch on the tcgen05 kernel when it applies (tensor copies need
// 16-byte aligned operands and row strides), MBGLU_OK with *done = true;
// otherwise *done = false and nothing is launched.
mbglu_status gemv_tc(const mbglu_bf16 *h, int64_t ldh, const mbglu_bf16 *gate_w, int64_t ld_gate,
                     const mbglu_bf16 *up_w, int64_t ld_up, mbglu_bf16 *out, int64_t ldo, int M, int N, int K,
                     mbglu_mode mode, cudaStream_t stream, bool *done)
{
    *done = false;
    if (!tuning().tc || M < tuning().tc_min_m || K % 8 != 0 || !aligned(h, 16) || !aligned(gate_w, 16) ||
        !aligned(up_w, 16) || ldh % 8 != 0 || ld_gate % 8 != 0 || ld_up % 8 != 0)
        return MBGLU_OK;
    const DeviceInfo *d = nullptr;
    mbglu_status st = device_info(&d);
    if (st != MBGLU_OK) return st;
    TcPlan pl;
    if (!plan_tc(*d, M, N, K, pl)) return MBGLU_OK;
    mbglu::TcMaps maps;
    if (!encode_sw128_map(&maps.gate, gate_w, ld_gate, N, K, mbglu::kTcRows) ||
        !encode_sw128_map(&maps.up, up_w, ld_up, N, K, mbglu::kTcRows) ||
        !encode_sw128_map(&maps.h, h, ldh, M, K, pl.Np))
        return MBGLU_OK;
    const int policy = g_policy.load(std::memory_order_relaxed);
    mbglu::TcParams p = {};
    p.out = reinterpret_cast<uint16_t *>(out);
    p.ldo = ldo;
    p.M = M;
    p.N = N;
    p.K = K;
    p.mode = static_cast<int>(mode);
    p.Np = pl.Np;
    p.nchunk = pl.nchunk;
    p.ksplit = pl.ksplit;
    p.stages = pl.stages;
    p.prefetch = policy == MBGLU_POLICY_PREFETCH;
    st = launch_tc(pl, p, maps, stream, policy != MBGLU_POLICY_SERIAL);
    if (st == MBGLU_OK) {
        *done = true;
        t_last_variant = kTcGemv;
    }
    return st;
}


}  // namespace

extern "C" {

mbglu_status glu_gemv(const mbglu_bf16 *h, int64_t ldh, const mbglu_bf16 *gate_w, int64_t ld_gate,
                      const mbglu_bf16 *up_w, int64_t ld_up, mbglu_bf16 *out, int64_t ldo, int M, int N, int K,
                      mbglu_mode mode, cudaStream_t stream)
{
    t_last_variant = kNone;
    mbglu_status st = check_gemv(h, ldh, gate_w, ld_gate, up_w, ld_up, out, ldo, M, N, K, mode);
    if (st != MBGLU_OK || M == 0 || N == 0) return st;
    if (K > 0 && M >= tuning().tc_min_m) {   // one pass on the tcgen05 kernel where it applies
        bool done = false;
        st = gemv_tc(h, ldh, gate_w, ld_gate, up_w, ld_up, out, ldo, M, N, K, mode, stream, &done);
        if (st != MBGLU_OK || done) return st;
    }
    if (M <= kBlockRows) return gemv_block(h, ldh, gate_w, ld_gate, up_w, ld_up, out, ldo, M, N, K, mode, stream);
    // a batch above one kernel's tile: row blocks of kBlockRows, the remainder
    // last, each a full pass over the weights (rows are independent, and every
    // kernel's result for a row does not depend on the rows beside it)
    for (int m0 = 0; m0 < M; m0 += kBlockRows) {
        const int mb = std::min(kBlockRows, M - m0);
        st = gemv_block(K > 0 ? h + static_cast<int64_t>(m0) * ldh : h, ldh, gate_w, ld_gate, up_w, ld_up,
                        out + static_cast<int64_t>(m0) * ldo, ldo, mb, N, K, mode, stream);
        if (st != MBGLU_OK) {
            t_last_variant = kNone;
            return st;
        }
    }
    t_last_variant = kRowBlocks;
    return MBGLU_OK;
}

}  // extern "C"

namespace {

int bwd_splits(int N) { return std::max(1, std::min(mbglu::kBwdMaxSplits, N / 256)); }

constexpr int kBwdMaxParts = 256;   // glu_bwd_rows_kernel: most CTAs (partials of grad_h per pass)

int batch_tile_wide(int M) { return M <= 16 ? batch_tile(M) : M <= 32 ? 32 : 64; }

// Plan of glu_bwd_rows_kernel: one CTA per SM (at most kBwdMaxParts, at most
// N), T = 32 * ceil(K / 8 / CPT / 32) <= 512 threads owning CPT 8-column
// chunks each, stages of R rows of both matrices (>= 16 KB), as many stages
// (2..16) as fit beside the share's dG and dU.  Passes of 8 rows (4 with two
// chunks per thread) keep the accumulators in registers.
struct BwdRowsPlan {
    int grid = 0, threads = 0, cpt = 1, R = 1, S = 0, rows_cta = 0, pass_rows = 8;
    uint32_t off_ring = 0, smem = 0;
};

bool plan_bwd_rows(const DeviceInfo &d, int N, int K, const void *gate_w, int64_t ld_gate, const void *up_w,
                   int64_t ld_up, BwdRowsPlan &rp)
{
    if (K % 8 != 0 || !aligned(gate_w, 16) || !aligned(up_w, 16) || ld_gate % 8 != 0 || ld_up % 8 != 0) return false;
    const int nchunk = K / 8;
    rp.cpt = (nchunk + mbglu::kBwdRowsThreads - 1) / mbglu::kBwdRowsThreads;
    if (rp.cpt > 2) return false;
    rp.threads = 32 * ((nchunk + 32 * rp.cpt - 1) / (32 * rp.cpt));
    rp.pass_rows = rp.cpt == 1 ? 8 : 4;
    rp.grid = std::max(1, std::min({d.sm_count, kBwdMaxParts, N}));
    rp.rows_cta = (N + rp.grid - 1) / rp.grid;
    const uint32_t dgu = 2u * static_cast<uint32_t>(rp.pass_rows) * static_cast<uint32_t>(rp.rows_cta) * 4u;
    rp.off_ring = (256u + dgu + 127u) & ~127u;
    rp.R = std::max(1, std::min(rp.rows_cta, (16384 + 4 * K - 1) / (4 * K)));
    const int64_t stage = 4ll * rp.R * K;
    const int64_t room = static_cast<int64_t>(d.smem_optin) - rp.off_ring;
    rp.S = static_cast<int>(std::min<int64_t>(16, room / stage));
    if (rp.S < 2) return false;
    rp.smem = rp.off_ring + static_cast<uint32_t>(rp.S * stage);
    return true;
}

// Plan of glu_bwd_hw_kernel (steps 2 and 3 in one pass, M <= 8): K in
// 256-column slices, one warp each; at most bwd_hw_warps(MB) warps per CTA,
// so K may be cut into column groups (CTAs sharing one row share); row
// shares so that all CTAs make about one wave; stages of R = 8 rows, as many
// (2..8) as fit beside the share's dG and dU.
struct BwdHwPlan {
    int MB = 1, cg = 1, warps = 1, shares = 1, rows_cta = 0, R = 8, S = 0;
    uint32_t off_ring = 0, smem = 0;
};

bool plan_bwd_hw(const DeviceInfo &d, int M, int N, int K, const void *h, int64_t ldh, const void *gate_w,
                 int64_t ld_gate, const void *up_w, int64_t ld_up, const void *grad_gate, int64_t ldgg,
                 const void *grad_up, int64_t ldgu, BwdHwPlan &hp)
{
    if (M > 8 || K % 8 != 0 || !aligned(h, 16) || ldh % 8 != 0 || !aligned(gate_w, 16) || !aligned(up_w, 16) ||
        ld_gate % 8 != 0 || ld_up % 8 != 0 || !aligned(grad_gate, 16) || !aligned(grad_up, 16) || ldgg % 8 != 0 ||
        ldgu % 8 != 0)
        return false;
    hp.MB = batch_tile(M);
    const int wtot = (K + mbglu::kBwdSlice - 1) / mbglu::kBwdSlice;
    const int wmax = mbglu::bwd_hw_warps(hp.MB);
    hp.cg = (wtot + wmax - 1) / wmax;
    hp.warps = (wtot + hp.cg - 1) / hp.cg;
    hp.shares = std::max(1, std::min(N, d.sm_count / hp.cg));
    hp.rows_cta = (N + hp.shares - 1) / hp.shares;
    const uint32_t dgu = 2u * static_cast<uint32_t>(hp.MB) * static_cast<uint32_t>(hp.rows_cta) * 4u;
    hp.off_ring = (256u + dgu + 127u) & ~127u;
    const int64_t room = static_cast<int64_t>(d.smem_optin) - hp.off_ring;
    for (int R = 8; R >= 2; R /= 2) {   // the tallest stage of which two per warp fit
        hp.R = std::min(R, hp.rows_cta);
        const int64_t stage = 2ll * hp.R * mbglu::kBwdSlice * 2;
        hp.S = static_cast<int>(std::min<int64_t>({8, room / (hp.warps * stage), 32 / hp.warps}));
        if (hp.S >= 2) {
            hp.smem = hp.off_ring + static_cast<uint32_t>(hp.warps * hp.S * stage);
            return true;
        }
    }
    return false;
}

mbglu_status launch_bwd_hw(const BwdHwPlan &hp, const mbglu::BwdParams &q, const mbglu::BwdMaps &maps,
                           cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(hp.shares * hp.cg);
    cfg.blockDim = dim3(32 * hp.warps);
    cfg.dynamicSmemBytes = hp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_policy.load(std::memory_order_relaxed) != MBGLU_POLICY_SERIAL ? 1 : 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (hp.MB) {
        case 1: e = cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_hw_kernel<1>, q, maps); break;
        case 2: e = cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_hw_kernel<2>, q, maps); break;
        case 4: e = cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_hw_kernel<4>, q, maps); break;
        default: e = cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_hw_kernel<8>, q, maps); break;
    }
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

// Plan of glu_bwd_mma_kernel (steps 2 and 3 on the tensor cores, M <= 16 in
// a batch tile MB of 8 or 16 rows):
// K in slices of 64 NB columns, one warp each; W warps per CTA cut K into
// cg column groups, and the SMs into row shares of about N / (SMs / cg) rows;
// stages of 16 rows, as many (2..4) as fit beside the staged dG, dU.  Of the
// warp counts that fit, the most warps (each warp's chain of dependent steps
// is what bounds the pass), then the most stages.
struct BwdMmaPlan {
    int NB = 2, MB = 8, cg = 1, warps = 1, shares = 1, rows_cta = 0, rows_pad = 0, S = 0;
    uint32_t off_nm = 0, off_ring = 0, smem = 0;
};

bool plan_bwd_mma(const DeviceInfo &d, int M, int N, int K, const void *h, int64_t ldh, const void *gate_w,
                  int64_t ld_gate, const void *up_w, int64_t ld_up, const void *grad_gate, int64_t ldgg,
                  const void *grad_up, int64_t ldgu, BwdMmaPlan &mp)
{
    if (M > 16 || K % 8 != 0 || !aligned(gate_w, 16) || !aligned(up_w, 16) || ld_gate % 8 != 0 ||
        ld_up % 8 != 0 || !aligned(grad_gate, 16) || !aligned(grad_up, 16) || ldgg % 8 != 0 || ldgu % 8 != 0)
        return false;
    const int NB = kBwdNB;
    const int MB = M > 8 ? 16 : 8;
    const int pitch = mbglu::bwd_mma_pitch(MB);
    // the workspace holds max(256 min(M, 8), 48 min(M, 16)) rows of K partials
    const int parts_cap = std::max(kBwdMaxParts * std::min(M, 8), static_cast<int>(mbglu::kBwdMaxSplits) * M) / M;
    const int slice = 64 * NB;
    const int wtot = (K + slice - 1) / slice;
    const int wmax = std::min(tuning().bwd_warps > 0 ? tuning().bwd_warps : mbglu::bwd_mma_warps(NB, MB),
                              mbglu::bwd_mma_warps(NB, MB));
    const int wmin = tuning().bwd_warps > 0 ? tuning().bwd_warps : 1;
    const int64_t stage = 2ll * NB * mbglu::kBwdMmaBox;
    bool found = false;
    int64_t best = -1;
    for (int w = wmax; w >= wmin; --w) {
        BwdMmaPlan c;
        c.NB = NB;
        c.MB = MB;
        c.cg = (wtot + w - 1) / w;
        c.warps = (wtot + c.cg - 1) / c.cg;   // the same groups, balanced
        if (c.warps != w) continue;
        c.shares = std::max(1, std::min({(N + 15) / 16, d.sm_count / c.cg, parts_cap}));
        c.rows_cta = (N + c.shares - 1) / c.shares;
        c.rows_pad = (c.rows_cta + 15) / 16 * 16;
        c.off_nm = 512;
        c.off_ring = (c.off_nm + 4u * static_cast<uint32_t>(pitch) * static_cast<uint32_t>(c.rows_pad) + 1023u) &
                     ~1023u;
        const int64_t room = static_cast<int64_t>(d.smem_optin) - 1024 - c.off_ring;   // 1024: base alignment
        if (room <= 0) continue;
        c.S = static_cast<int>(std::min<int64_t>({4, room / (c.warps * stage), 64 / c.warps}));
        if (c.S < 2) continue;
        c.smem = c.off_ring + static_cast<uint32_t>(c.warps * c.S * stage) + 1024u;
        const int64_t score = 16ll * c.warps + c.S;
        if (score > best) {
            best = score;
            mp = c;
            found = true;
        }
    }
    return found;
}

mbglu_status launch_bwd_mma(const BwdMmaPlan &mp, const mbglu::BwdParams &q, const mbglu::BwdMaps &maps,
                            cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(mp.shares * mp.cg);
    cfg.blockDim = dim3(32 * mp.warps);
    cfg.dynamicSmemBytes = mp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_policy.load(std::memory_order_relaxed) != MBGLU_POLICY_SERIAL ? 1 : 0;
    const cudaError_t e = mp.MB > 8 ? cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_mma_kernel<kBwdNB, 16>, q, maps)
                                    : cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_mma_kernel<kBwdNB, 8>, q, maps);
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

mbglu_status launch_bwd_rows(const BwdRowsPlan &rp, int MB, const mbglu::BwdParams &q, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rp.grid);
    cfg.blockDim = dim3(rp.threads);
    cfg.dynamicSmemBytes = rp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_policy.load(std::memory_order_relaxed) != MBGLU_POLICY_SERIAL ? 1 : 0;
    cudaError_t e = cudaErrorInvalidValue;
#define MBGLU_BWD_ROWS(TMB, TCPT)                                                             \
    if (MB == TMB && rp.cpt == TCPT) e = cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_rows_kernel<TMB, TCPT>, q);
    MBGLU_BWD_ROWS(1, 1) MBGLU_BWD_ROWS(2, 1) MBGLU_BWD_ROWS(4, 1) MBGLU_BWD_ROWS(8, 1)
    MBGLU_BWD_ROWS(1, 2) MBGLU_BWD_ROWS(2, 2) MBGLU_BWD_ROWS(4, 2)
#undef MBGLU_BWD_ROWS
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

int64_t round256(int64_t b) { return (b + 255) & ~static_cast<int64_t>(255); }

mbglu_status launch_plain(cudaError_t e)
{
    return e == cudaSuccess ? MBGLU_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

size_t glu_backward_workspace_bytes(int M, int N, int K)
{
    if (M <= 0 || N <= 0 || K <= 0 || M > MBGLU_MAX_M) return 0;
    // dG, dU; then the grad_h partials of one pass: up to kBwdMaxParts CTAs
    // of the rows kernel at 8 rows, or kBwdMaxSplits splits at kBlockRows rows
    const int64_t parts = std::max<int64_t>(static_cast<int64_t>(kBwdMaxParts) * std::min(M, 8),
                                            static_cast<int64_t>(mbglu::kBwdMaxSplits) * std::min(M, kBlockRows));
    return static_cast<size_t>(round256(2 * static_cast<int64_t>(M) * N * 4) + round256(parts * K * 4));
}

mbglu_status glu_backward(const mbglu_bf16 *h, int64_t ldh, const mbglu_bf16 *gate_w, int64_t ld_gate,
                          const mbglu_bf16 *up_w, int64_t ld_up, const mbglu_bf16 *dout, int64_t ldd,
                          mbglu_bf16 *grad_h, int64_t ldgh, mbglu_bf16 *grad_gate, int64_t ldgg,
                          mbglu_bf16 *grad_up, int64_t ldgu, int M, int N, int K, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream)
{
    t_last_variant = kNone;
    t_last_bwd = 0;
    if (M < 0 || N < 0 || K < 0 || M > MBGLU_MAX_M) return MBGLU_ERR_SHAPE;
    const bool want_h = grad_h != nullptr, want_w = grad_gate != nullptr || grad_up != nullptr;
    if (want_w && (!grad_gate || !grad_up)) return MBGLU_ERR_NULL;
    if (K == 0) return MBGLU_OK;   // every gradient has K columns
    // shapes where one factor is empty: the gradients that remain are sums of nothing
    const bool full = M > 0 && N > 0;
    if (full && (!h || !gate_w || !up_w || !dout || !workspace)) return MBGLU_ERR_NULL;
    if ((M > 0 && want_h && ldgh < K) || (N > 0 && want_w && (ldgg < K || ldgu < K))) return MBGLU_ERR_STRIDE;
    if (full && (ldh < K || ld_gate < K || ld_up < K || ldd < N)) return MBGLU_ERR_STRIDE;
    if (!aligned(h, 2) || !aligned(gate_w, 2) || !aligned(up_w, 2) || !aligned(dout, 2) || !aligned(grad_h, 2) ||
        !aligned(grad_gate, 2) || !aligned(grad_up, 2) || !aligned(workspace, 16))
        return MBGLU_ERR_ALIGN;
    const size_t need = glu_backward_workspace_bytes(M, N, K);
    if (full && workspace_bytes < need) return MBGLU_ERR_SHAPE;
    // outputs against inputs and one another
    const int64_t hb = matrix_bytes(M, K, ldh), gb = matrix_bytes(N, K, ld_gate), ub = matrix_bytes(N, K, ld_up);
    const int64_t db = matrix_bytes(M, N, ldd);
    const int64_t ghb = want_h ? matrix_bytes(M, K, ldgh) : 0;
    const int64_t ggb = want_w ? matrix_bytes(N, K, ldgg) : 0, gub = want_w ? matrix_bytes(N, K, ldgu) : 0;
    const int64_t wsb = full ? static_cast<int64_t>(need) : 0;
    const void *ins[4] = {h, gate_w, up_w, dout};
    const int64_t inb[4] = {full ? hb : 0, full ? gb : 0, full ? ub : 0, full ? db : 0};
    const void *outs[4] = {grad_h, grad_gate, grad_up, workspace};
    const int64_t outb[4] = {ghb, ggb, gub, wsb};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 4; ++j)
            if (overlaps(outs[i], outb[i], ins[j], inb[j])) return MBGLU_ERR_ALIAS;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], outb[i], outs[j], outb[j])) return MBGLU_ERR_ALIAS;
    }
    if (M == 0 && N == 0) return MBGLU_OK;
    if (!full) {   // N == 0: grad_h = 0; M == 0: grad_gate = grad_up = 0
        cudaError_t e = cudaSuccess;
        if (N == 0 && want_h)
            e = cudaMemset2DAsync(grad_h, static_cast<size_t>(ldgh) * 2, 0, static_cast<size_t>(K) * 2, M, stream);
        if (e == cudaSuccess && M == 0 && want_w) {
            e = cudaMemset2DAsync(grad_gate, static_cast<size_t>(ldgg) * 2, 0, static_cast<size_t>(K) * 2, N, stream);
            if (e == cudaSuccess)
                e = cudaMemset2DAsync(grad_up, static_cast<size_t>(ldgu) * 2, 0, static_cast<size_t>(K) * 2, N, stream);
        }
        return launch_plain(e);
    }

    const DeviceInfo *d = nullptr;
    mbglu_status st = device_info(&d);
    if (st != MBGLU_OK) return st;
    float *dG = static_cast<float *>(workspace);
    float *dU = dG + static_cast<int64_t>(M) * N;
    float *part = reinterpret_cast<float *>(static_cast<char *>(workspace) + round256(2 * static_cast<int64_t>(M) * N * 4));

    // 1) dG, dU: the forward kernels with the backward epilogue, per block of
    //    up to kBlockRows rows (the weights stay in L2 for step 2)
    for (int m0 = 0; m0 < M; m0 += kBlockRows) {
        const int mb = std::min(kBlockRows, M - m0);
        const BwdEpilogue be = {dout + static_cast<int64_t>(m0) * ldd, ldd, dG + static_cast<int64_t>(m0) * N,
                                dU + static_cast<int64_t>(m0) * N};
        st = gemv_block(h + static_cast<int64_t>(m0) * ldh, ldh, gate_w, ld_gate, up_w, ld_up, nullptr, 0, mb, N, K,
                        MBGLU_MODE_FUSED, stream, &be);
        if (st != MBGLU_OK) return st;
    }

    mbglu::BwdParams q = {};
    q.h = h;
    q.ldh = ldh;
    q.gate = gate_w;
    q.ld_gate = ld_gate;
    q.up = up_w;
    q.ld_up = ld_up;
    q.part = part;
    q.grad_h = grad_h;
    q.ldgh = ldgh;
    q.grad_gate = grad_gate;
    q.ldgg = ldgg;
    q.grad_up = grad_up;
    q.ldgu = ldgu;
    q.N = N;
    q.K = K;
    q.ldm = N;
    q.vec_w = aligned(gate_w, 8) && aligned(up_w, 8) && ld_gate % 4 == 0 && ld_up % 4 == 0;
    cudaError_t e = cudaSuccess;
    // 2 + 3 in one pass over the rows where it applies (aligned; M <= 8 on
    // the CUDA cores, M <= 16 on the tensor cores): grad_h partials and both
    // weight gradients, then the partials' sum.  From bwd_mma_min_m rows on,
    // the pass runs on the tensor cores.
    BwdMmaPlan mp;
    mbglu::BwdMaps mmaps;
    if (want_h && want_w && tuning().bwd_fused && M >= tuning().bwd_mma_min_m &&
        plan_bwd_mma(*d, M, N, K, h, ldh, gate_w, ld_gate, up_w, ld_up, grad_gate, ldgg, grad_up, ldgu, mp) &&
        encode_sw128_map(&mmaps.gate, gate_w, ld_gate, N, K, 16) &&
        encode_sw128_map(&mmaps.up, up_w, ld_up, N, K, 16)) {
        q.M = M;
        q.dG = dG;
        q.dU = dU;
        q.rows_cta = mp.rows_cta;
        q.rows_pad = mp.rows_pad;
        q.col_groups = mp.cg;
        q.S = mp.S;
        q.off_nm = mp.off_nm;
        q.off_ring = mp.off_ring;
        st = launch_bwd_mma(mp, q, mmaps, stream);
        if (st != MBGLU_OK) return st;
        t_last_bwd = 3;
        const int64_t warps = static_cast<int64_t>(M) * (K / 8);
        const int rgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(d->sm_count * 8, (warps + 7) / 8)));
        const int vec_store = aligned(grad_h, 16) && ldgh % 8 == 0;
        mbglu::glu_bwd_h_reduce8_kernel<<<rgrid, 256, 0, stream>>>(q, mp.shares, vec_store);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
        t_last_variant = kBackward;
        return MBGLU_OK;
    }
    BwdHwPlan hp;
    mbglu::BwdMaps hmaps;
    if (want_h && want_w && tuning().bwd_fused &&
        plan_bwd_hw(*d, M, N, K, h, ldh, gate_w, ld_gate, up_w, ld_up, grad_gate, ldgg, grad_up, ldgu, hp) &&
        encode_box_map(&hmaps.gate, gate_w, ld_gate, N, K, mbglu::kBwdSlice, hp.R) &&
        encode_box_map(&hmaps.up, up_w, ld_up, N, K, mbglu::kBwdSlice, hp.R)) {
        q.M = M;
        q.dG = dG;
        q.dU = dU;
        q.rows_cta = hp.rows_cta;
        q.col_groups = hp.cg;
        q.R = hp.R;
        q.S = hp.S;
        q.off_ring = hp.off_ring;
        st = launch_bwd_hw(hp, q, hmaps, stream);
        if (st != MBGLU_OK) return st;
        t_last_bwd = 2;
        const int64_t warps = static_cast<int64_t>(M) * (K / 8);
        const int rgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(d->sm_count * 8, (warps + 7) / 8)));
        const int vec_store = aligned(grad_h, 16) && ldgh % 8 == 0;
        mbglu::glu_bwd_h_reduce8_kernel<<<rgrid, 256, 0, stream>>>(q, hp.shares, vec_store);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
        t_last_variant = kBackward;
        return MBGLU_OK;
    }
    // 2) grad_h: partials, then their sum in order; passes of up to 8 rows
    //    (the rows kernel) or kBlockRows rows (the column-block kernel)
    if (want_h) {
        BwdRowsPlan rp;
        const bool rows_ok = plan_bwd_rows(*d, N, K, gate_w, ld_gate, up_w, ld_up, rp);
        const int pass = rows_ok ? rp.pass_rows : kBlockRows;
        for (int m0 = 0; m0 < M; m0 += pass) {
            const int mb = std::min(pass, M - m0);
            q.M = mb;
            q.dG = dG + static_cast<int64_t>(m0) * N;
            q.dU = dU + static_cast<int64_t>(m0) * N;
            q.grad_h = grad_h + static_cast<int64_t>(m0) * ldgh;
            int nparts = 0;
            if (rows_ok) {
                q.R = rp.R;
                q.S = rp.S;
                q.off_ring = rp.off_ring;
                q.rows_cta = rp.rows_cta;
                st = launch_bwd_rows(rp, batch_tile(mb), q, stream);
                if (st != MBGLU_OK) return st;
                nparts = rp.grid;
            } else {
                nparts = bwd_splits(N);
                const dim3 grid((K + mbglu::kBwdCols - 1) / mbglu::kBwdCols, nparts);
                const int MB = batch_tile(mb);
                const size_t smem = static_cast<size_t>(std::max(2 * mb * mbglu::kBwdRowChunk, MB * 4 * 128)) * 4;
                switch (MB) {
                    case 1: mbglu::glu_bwd_h_kernel<1><<<grid, 256, smem, stream>>>(q); break;
                    case 2: mbglu::glu_bwd_h_kernel<2><<<grid, 256, smem, stream>>>(q); break;
                    case 4: mbglu::glu_bwd_h_kernel<4><<<grid, 256, smem, stream>>>(q); break;
                    case 8: mbglu::glu_bwd_h_kernel<8><<<grid, 256, smem, stream>>>(q); break;
                    default: mbglu::glu_bwd_h_kernel<16><<<grid, 256, smem, stream>>>(q); break;
                }
                if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
            }
            if (rows_ok) {   // one warp per (row, 8 columns), the lanes over the partials
                const int64_t warps = static_cast<int64_t>(mb) * (K / 8);
                const int rgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(d->sm_count * 8, (warps + 7) / 8)));
                const int vec_store = aligned(grad_h, 16) && ldgh % 8 == 0;
                mbglu::glu_bwd_h_reduce8_kernel<<<rgrid, 256, 0, stream>>>(q, nparts, vec_store);
            } else {
                const int rgrid = static_cast<int>(std::max<int64_t>(
                    1, std::min<int64_t>(d->sm_count * 4, (static_cast<int64_t>(mb) * K + 255) / 256)));
                mbglu::glu_bwd_h_reduce_kernel<<<rgrid, 256, 0, stream>>>(q, nparts);
            }
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
        }
    }
    // 3) grad_gate, grad_up: the outer products over all M rows, h in shared
    //    memory where it fits
    const int wcpt = (K / 8 + mbglu::kBwdRowsThreads - 1) / mbglu::kBwdRowsThreads;   // chunks per thread
    if (want_w && K % 8 == 0 && (M <= 8 && wcpt == 1 || M <= 4 && wcpt == 2) &&
        aligned(grad_gate, 16) && aligned(grad_up, 16) && ldgg % 8 == 0 && ldgu % 8 == 0 && aligned(h, 16) &&
        ldh % 8 == 0) {
        // the main path: whole rows per CTA, h in registers
        q.M = M;
        q.dG = dG;
        q.dU = dU;
        const int cpt = wcpt;
        const int threads = 32 * ((K / 8 + 32 * cpt - 1) / (32 * cpt));
        const int grid = std::max(1, std::min(2 * d->sm_count, N));
        q.rows_cta = (N + grid - 1) / grid;
        const size_t smem = 2u * 8u * static_cast<size_t>(q.rows_cta) * 4u;
        const int MB = batch_tile(M);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = g_policy.load(std::memory_order_relaxed) != MBGLU_POLICY_SERIAL ? 1 : 0;
        e = cudaErrorInvalidValue;
#define MBGLU_BWD_W(TMB, TCPT)                                                                   \
        if (MB == TMB && cpt == TCPT) e = cudaLaunchKernelEx(&cfg, mbglu::glu_bwd_w_rows_kernel<TMB, TCPT>, q);
        MBGLU_BWD_W(1, 1) MBGLU_BWD_W(2, 1) MBGLU_BWD_W(4, 1) MBGLU_BWD_W(8, 1)
        MBGLU_BWD_W(1, 2) MBGLU_BWD_W(2, 2) MBGLU_BWD_W(4, 2)
#undef MBGLU_BWD_W
        if (e != cudaSuccess) return cuda_fail(e);
    } else if (want_w) {
        q.M = M;
        q.dG = dG;
        q.dU = dU;
        const int64_t hbytes = static_cast<int64_t>(M) * K * 2;
        q.h_smem = hbytes <= kBwdHSmemMax;
        q.vec_out = K % 8 == 0 && aligned(grad_gate, 16) && aligned(grad_up, 16) && ldgg % 8 == 0 && ldgu % 8 == 0 &&
                    (q.h_smem || (aligned(h, 16) && ldh % 8 == 0));
        const size_t smem = q.h_smem ? static_cast<size_t>(hbytes) : 0;
        const int wgrid = std::max(1, std::min(N, d->sm_count * 2));
        switch (batch_tile_wide(M)) {
            case 1: mbglu::glu_bwd_w_kernel<1><<<wgrid, 256, smem, stream>>>(q); break;
            case 2: mbglu::glu_bwd_w_kernel<2><<<wgrid, 256, smem, stream>>>(q); break;
            case 4: mbglu::glu_bwd_w_kernel<4><<<wgrid, 256, smem, stream>>>(q); break;
            case 8: mbglu::glu_bwd_w_kernel<8><<<wgrid, 256, smem, stream>>>(q); break;
            case 16: mbglu::glu_bwd_w_kernel<16><<<wgrid, 256, smem, stream>>>(q); break;
            case 32: mbglu::glu_bwd_w_kernel<32><<<wgrid, 256, smem, stream>>>(q); break;
            default: mbglu::glu_bwd_w_kernel<64><<<wgrid, 256, smem, stream>>>(q); break;
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    }
    t_last_variant = kBackward;
    t_last_bwd = 1;
    return MBGLU_OK;
}

}  // extern "C"

namespace {

// Every argument check of the add_rmsnorm_glu entry points, on the whole call.
mbglu_status check_norm(const mbglu_bf16 *x, const mbglu_bf16 *residual, const mbglu_bf16 *norm_w,
                        const mbglu_bf16 *gate_w, int64_t ld_gate, const mbglu_bf16 *up_w, int64_t ld_up,
                        const mbglu_bf16 *out, int64_t ldo, int M, int N, int K, mbglu_mode mode, const int *ws)
{
    if (mode != MBGLU_MODE_FUSED && mode != MBGLU_MODE_HF) return MBGLU_ERR_MODE;
    if (M < 0 || N < 0 || K <= 0 || M > MBGLU_MAX_M) return MBGLU_ERR_SHAPE;
    if (static_cast<int64_t>(std::min(M, kBlockRows)) * K > kNormMaxMK) return MBGLU_ERR_SHAPE;
    if (M == 0) return MBGLU_OK;
    if (!x || !residual || !norm_w || (N > 0 && (!gate_w || !up_w || !out))) return MBGLU_ERR_NULL;
    if (N > 0 && (ld_gate < K || ld_up < K || ldo < N)) return MBGLU_ERR_STRIDE;
    if (!aligned(x, 2) || !aligned(residual, 2) || !aligned(norm_w, 2) ||
        (N > 0 && (!aligned(gate_w, 2) || !aligned(up_w, 2) || !aligned(out, 2))))
        return MBGLU_ERR_ALIGN;
    const int64_t xb = static_cast<int64_t>(M) * K * 2, nb = static_cast<int64_t>(K) * 2;
    const int64_t gb = matrix_bytes(N, K, ld_gate), ub = matrix_bytes(N, K, ld_up), ob = matrix_bytes(M, N, ldo);
    if (x != residual && overlaps(x, xb, residual, xb)) return MBGLU_ERR_ALIAS;
    if (overlaps(residual, xb, norm_w, nb) || overlaps(residual, xb, gate_w, gb) || overlaps(residual, xb, up_w, ub))
        return MBGLU_ERR_ALIAS;
    if (N > 0 && (overlaps(out, ob, x, xb) || overlaps(out, ob, residual, xb) || overlaps(out, ob, norm_w, nb) ||
                  overlaps(out, ob, gate_w, gb) || overlaps(out, ob, up_w, ub)))
        return MBGLU_ERR_ALIAS;
    if (ws) {
        const int64_t wsb = MBGLU_WORKSPACE_BYTES;
        if (overlaps(ws, wsb, x, xb) || overlaps(ws, wsb, residual, xb) || overlaps(ws, wsb, norm_w, nb) ||
            (N > 0 && (overlaps(ws, wsb, gate_w, gb) || overlaps(ws, wsb, up_w, ub) || overlaps(ws, wsb, out, ob))))
            return MBGLU_ERR_ALIAS;
    }
    return MBGLU_OK;
}

// add_rmsnorm_glu on 1 <= M <= kBlockRows rows, arguments already checked.
// ws == nullptr: residual-add kernel, then the GEMV with the norm prologue.
// ws != nullptr: one kernel (the add is formed in shared memory, residual
// written back by the last CTA), where the fast kernels apply; otherwise the
// two-kernel path.
mbglu_status norm_block(const mbglu_bf16 *x, mbglu_bf16 *residual, const mbglu_bf16 *norm_w, float eps,
                        const mbglu_bf16 *gate_w, int64_t ld_gate, const mbglu_bf16 *up_w, int64_t ld_up,
                        mbglu_bf16 *out, int64_t ldo, int M, int N, int K, mbglu_mode mode, int *ws,
                        cudaStream_t stream)
{
    const DeviceInfo *d = nullptr;
    mbglu_status st = device_info(&d);
    if (st != MBGLU_OK) return st;
    const int policy = g_policy.load(std::memory_order_relaxed);
    const bool pdl = policy != MBGLU_POLICY_SERIAL;

    GluParams p = base_params(M, N, K, static_cast<int>(mode));
    p.gate = gate_w;
    p.ld_gate = ld_gate;
    p.up = up_w;
    p.ld_up = ld_up;
    p.out = out;
    p.ldo = ldo;
    p.s = residual;
    p.norm_w = norm_w;
    p.eps = eps;
    p.vec_in = (K % 8 == 0) && aligned(residual, 16) && aligned(norm_w, 16);
    p.prefetch = policy == MBGLU_POLICY_PREFETCH;
    p.interleave = tuning().interleave;
    const bool bulk_ok = (K % 8 == 0) && aligned(gate_w, 16) && aligned(up_w, 16) && (ld_gate % 8 == 0) &&
                         (ld_up % 8 == 0) && p.vec_in;

    // single kernel: needs the fast kernels, 16-byte aligned x, and N > 0
    // norm_w in shared memory, then the statistic's per-thread partials
    const uint32_t nwbytes = ((static_cast<uint32_t>(K) * 2u + 127u) & ~127u) + mbglu::kNormPartBytes;
    if (ws && N > 0 && bulk_ok && aligned(x, 16)) {
        const uint32_t sbytes = nwbytes;   // s is formed in place where the residual rows land
        Plan pl;
        p.fused = 1;
        p.x = x;
        p.residual = residual;
        p.ws = ws;
        SlicePlan sp;
        mbglu::SliceMaps smaps;
        if (plan_slice(*d, M, N, K, sp, true) && encode_sw128_map(&smaps.gate, gate_w, ld_gate, N, K, 8) &&
            encode_sw128_map(&smaps.up, up_w, ld_up, N, K, 8)) {   // the epilogue warp writes the residual slice
            p.stages = sp.stages;
            p.off_s = sp.off_s;
            p.off_ring = sp.off_ring;
            st = launch_slice<true>(sp, p, smaps, stream, pdl);
            if (st == MBGLU_OK) {
                t_last_variant = kSlice;
                ++t_last_single;
            }
            return st;
        }
        if (plan_mma(*d, M, N, K, pl, sbytes)) {   // + the helper warp: up to kMaxStreamWarps + 1 warps
            p.KS = pl.KS;
            p.nseg = pl.nseg;
            p.stages = pl.stages;
            p.off_h = pl.off_h;
            p.off_s = pl.off_s;
            p.off_ring = pl.off_ring;
            p.off_piece = pl.off_piece;
            p.off_carry = pl.off_carry;
            p.nphase = pl.nphase;
            p.nsp = pl.nsp;
            p.helper_warp = pl.warps;   // one extra warp writes the residual slice
            const mbglu::MmaMaps maps = weight_maps(p);
            st = launch_mma(mbglu::glu_mma_kernel<true>, dim3(pl.grid), dim3((pl.warps + 1) * 32), pl.smem, stream,
                            pdl, p, maps);
            if (st == MBGLU_OK) {
                t_last_variant = kTensor;
                ++t_last_single;
            }
            return st;
        }
        if (plan_stream(*d, M, N, K, true, true, pl, true, sbytes, mbglu::kMaxStreamWarps - 1)) {
            p.KS = pl.KS;
            p.nseg = pl.nseg;
            p.stages = pl.stages;
            p.off_h = pl.off_h;
            p.off_s = pl.off_s;
            p.off_ring = pl.off_ring;
            p.helper_warp = pl.warps;   // one extra warp writes the residual slice
            st = launch_stream<true>(pl, p, stream, pdl);
            if (st == MBGLU_OK) {
                t_last_variant = kStream;
                ++t_last_single;
            }
            return st;
        }
        p.fused = 0;
        p.x = nullptr;
        p.residual = nullptr;
        p.ws = nullptr;
        p.helper_warp = -1;
    }

    // 1) residual <- bf16(x + residual); it waits for its predecessor before
    //    reading and releases the GEMV launch at once.
    {
        const int64_t count = static_cast<int64_t>(M) * K;
        const int vec = aligned(x, 16) && aligned(residual, 16) && (count % 8 == 0);
        const int64_t work = vec ? count / 8 : count;
        const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(d->sm_count, (work + 255) / 256)));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, mbglu::residual_add_kernel, reinterpret_cast<const uint16_t *>(x),
                                                 reinterpret_cast<uint16_t *>(residual), count, vec);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (N == 0) {
        t_last_variant = kNone;
        return MBGLU_OK;
    }

    // 2) the GEMV with the norm prologue, as a programmatic dependent launch
    Plan pl;
    SlicePlan sp;
    mbglu::SliceMaps smaps;
    if (bulk_ok && plan_slice(*d, M, N, K, sp, true) && encode_sw128_map(&smaps.gate, gate_w, ld_gate, N, K, 8) &&
        encode_sw128_map(&smaps.up, up_w, ld_up, N, K, 8)) {
        p.stages = sp.stages;
        p.off_s = sp.off_s;
        p.off_ring = sp.off_ring;
        st = launch_slice<true>(sp, p, smaps, stream, pdl);
        if (st == MBGLU_OK) t_last_variant = kSlice;
        return st;
    }
    if (bulk_ok && plan_mma(*d, M, N, K, pl, nwbytes)) {
        p.KS = pl.KS;
        p.nseg = pl.nseg;
        p.stages = pl.stages;
        p.off_h = pl.off_h;
        p.off_s = pl.off_s;
        p.off_ring = pl.off_ring;
        p.off_piece = pl.off_piece;
        p.off_carry = pl.off_carry;
        p.nphase = pl.nphase;
        p.nsp = pl.nsp;
        const mbglu::MmaMaps maps = weight_maps(p);
        st = launch_mma(mbglu::glu_mma_kernel<true>, dim3(pl.grid), dim3(pl.warps * 32), pl.smem, stream, pdl, p,
                        maps);
        if (st == MBGLU_OK) t_last_variant = kTensor;
        return st;
    }
    const bool fast = bulk_ok && plan_stream(*d, M, N, K, true, true, pl, true, nwbytes);
    if (fast) {
        p.KS = pl.KS;
        p.nseg = pl.nseg;
        p.stages = pl.stages;
        p.off_h = pl.off_h;
        p.off_s = pl.off_s;
        p.off_ring = pl.off_ring;
        st = launch_stream<true>(pl, p, stream, pdl);
        if (st == MBGLU_OK) t_last_variant = kStream;
        return st;
    }
    p.vec_in = 0;
    const uint32_t smem = static_cast<uint32_t>(M) * static_cast<uint32_t>(K) * 2u;
    st = launch(mbglu::glu_generic_kernel<true>, dim3(generic_grid(*d, N)), dim3(256), smem, stream, pdl, p);
    if (st == MBGLU_OK) t_last_variant = kGeneric;
    return st;
}

mbglu_status add_rmsnorm_glu_impl(const mbglu_bf16 *x, mbglu_bf16 *residual, const mbglu_bf16 *norm_w, float eps,
                                  const mbglu_bf16 *gate_w, int64_t ld_gate, const mbglu_bf16 *up_w, int64_t ld_up,
                                  mbglu_bf16 *out, int64_t ldo, int M, int N, int K, mbglu_mode mode, int *ws,
                                  cudaStream_t stream)
{
    t_last_variant = kNone;
    t_last_single = 0;
    mbglu_status st = check_norm(x, residual, norm_w, gate_w, ld_gate, up_w, ld_up, out, ldo, M, N, K, mode, ws);
    if (st != MBGLU_OK || M == 0) return st;
    if (M <= kBlockRows)
        return norm_block(x, residual, norm_w, eps, gate_w, ld_gate, up_w, ld_up, out, ldo, M, N, K, mode, ws, stream);
    // row blocks, as glu_gemv: the add, the statistic and the normed row are
    // per row.  Consecutive blocks share the workspace, which every completed
    // single-kernel call leaves zero.
    for (int m0 = 0; m0 < M; m0 += kBlockRows) {
        const int mb = std::min(kBlockRows, M - m0);
        const int64_t xo = static_cast<int64_t>(m0) * K;
        st = norm_block(x + xo, residual + xo, norm_w, eps, gate_w, ld_gate, up_w, ld_up,
                        N > 0 ? out + static_cast<int64_t>(m0) * ldo : out, ldo, mb, N, K, mode, ws, stream);
        if (st != MBGLU_OK) {
            t_last_variant = kNone;
            return st;
        }
    }
    t_last_variant = N > 0 ? kRowBlocks : kNone;   // N == 0: the residual adds alone, as for one block
    return MBGLU_OK;
}

}  // namespace

extern "C" {

mbglu_status add_rmsnorm_glu(const mbglu_bf16 *x, mbglu_bf16 *residual, const mbglu_bf16 *norm_w, float eps,
                             const mbglu_bf16 *gate_w, const mbglu_bf16 *up_w, mbglu_bf16 *out, int M, int N, int K,
                             mbglu_mode mode, cudaStream_t stream)
{
    return add_rmsnorm_glu_impl(x, residual, norm_w, eps, gate_w, K, up_w, K, out, N, M, N, K, mode, nullptr, stream);
}

mbglu_status add_rmsnorm_glu_strided(const mbglu_bf16 *x, mbglu_bf16 *residual, const mbglu_bf16 *norm_w, float eps,
                                     const mbglu_bf16 *gate_w, int64_t ld_gate, const mbglu_bf16 *up_w, int64_t ld_up,
                                     mbglu_bf16 *out, int64_t ldo, int M, int N, int K, mbglu_mode mode,
                                     void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    t_last_variant = kNone;
    t_last_single = 0;
    if (workspace) {
        if (workspace_bytes < MBGLU_WORKSPACE_BYTES) return MBGLU_ERR_SHAPE;
        if (!aligned(workspace, 16)) return MBGLU_ERR_ALIGN;
    }
    return add_rmsnorm_glu_impl(x, residual, norm_w, eps, gate_w, ld_gate, up_w, ld_up, out, ldo, M, N, K, mode,
                                static_cast<int *>(workspace), stream);
}

mbglu_status add_rmsnorm_glu_ws(const mbglu_bf16 *x, mbglu_bf16 *residual, const mbglu_bf16 *norm_w, float eps,
                                const mbglu_bf16 *gate_w, const mbglu_bf16 *up_w, mbglu_bf16 *out, int M, int N,
                                int K, mbglu_mode mode, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream)
{
    t_last_variant = kNone;
    t_last_single = 0;
    if (!workspace) return MBGLU_ERR_NULL;
    if (workspace_bytes < MBGLU_WORKSPACE_BYTES) return MBGLU_ERR_SHAPE;
    if (!aligned(workspace, 16)) return MBGLU_ERR_ALIGN;
    return add_rmsnorm_glu_impl(x, residual, norm_w, eps, gate_w, K, up_w, K, out, N, M, N, K, mode,
                                static_cast<int *>(workspace), stream);
}

mbglu_status mbglu_read_device_error(int *word)
{
    if (!word) return MBGLU_ERR_NULL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    int w = 0;
    if ((e = cudaMemcpyFromSymbol(&w, mbglu::g_device_error, sizeof w)) != cudaSuccess) return cuda_fail(e);
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(mbglu::g_device_error, &zero, sizeof zero)) != cudaSuccess) return cuda_fail(e);
    *word = w;
    return MBGLU_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// add_rmsnorm_glu_noalloc: the single-kernel add_rmsnorm_glu for callers that
// cannot allocate device memory.  Its scratch -- the two arrival counters the
// single kernel needs -- lives in this file-scope device array instead of a
// caller-provided workspace.  Every GPU that loads the library holds it until
// the process exits.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) int g_noalloc_scratch[MBGLU_NOALLOC_SCRATCH_BYTES / sizeof(int)];
static_assert(MBGLU_WORKSPACE_BYTES <= MBGLU_NOALLOC_SCRATCH_BYTES, "the array must hold one workspace");

std::mutex g_noalloc_mu;
int *g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};

// The identity of the current context (0 if the driver cannot tell): a
// cudaDeviceReset destroys the context and a new one gets a new identity,
// so an address kept from the old context is never reused.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static const std::pair<GetCurrent, GetId> fns = [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            a = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            b = nullptr;
        return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!fns.first || !fns.second || fns.first(&ctx) != CUDA_SUCCESS || !ctx || fns.second(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// The array's device address on the current device.  In host code the name
// g_noalloc_scratch is only a host-side stand-in, so the address is asked of
// the runtime (with the device current) and kept per device together with the
// context it belongs to; a new context (after cudaDeviceReset) looks it up again.
mbglu_status noalloc_scratch(int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    // 0 when no context is current on this thread yet: the address is then
    // looked up (which makes one current) and looked up again next time
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev] || ctx == 0 || g_noalloc_ctx[dev] != ctx) {
        int *ptr = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        g_noalloc_ptr[dev] = ptr;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return MBGLU_OK;
}

}  // namespace

extern "C" mbglu_status add_rmsnorm_glu_noalloc(const mbglu_bf16 *x, mbglu_bf16 *residual, const mbglu_bf16 *norm_w,
                                                float eps, const mbglu_bf16 *gate_w, const mbglu_bf16 *up_w,
                                                mbglu_bf16 *out, int M, int N, int K, mbglu_mode mode,
                                                cudaStream_t stream)
{
    t_last_variant = kNone;
    t_last_single = 0;
    // the scratch this call needs must fit the array (the single kernel needs
    // one workspace whatever the shapes; the check states the limit)
    const size_t need = MBGLU_WORKSPACE_BYTES;
    if (need > MBGLU_NOALLOC_SCRATCH_BYTES) return MBGLU_ERR_SHAPE;
    int *scratch = nullptr;
    mbglu_status st = noalloc_scratch(&scratch);
    if (st != MBGLU_OK) return st;
    // the counters must start at zero; the array keeps whatever the last call
    // (on any stream) left there, so clear them, in stream order
    const cudaError_t e = cudaMemsetAsync(scratch, 0, need, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return add_rmsnorm_glu_ws(x, residual, norm_w, eps, gate_w, up_w, out, M, N, K, mode, scratch, need, stream);
}

// Diagnostics: the first `count` words of the current device's no-allocation
// scratch array, after the device has finished its work.
extern "C" mbglu_status mbglu_noalloc_scratch_read(int *words, int count)
{
    if (!words) return MBGLU_ERR_NULL;
    if (count < 0 || count * sizeof(int) > MBGLU_NOALLOC_SCRATCH_BYTES) return MBGLU_ERR_SHAPE;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    if (count == 0) return MBGLU_OK;
    if ((e = cudaMemcpyFromSymbol(words, g_noalloc_scratch, count * sizeof(int))) != cudaSuccess) return cuda_fail(e);
    return MBGLU_OK;
}
