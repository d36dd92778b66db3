/*
 * mbglu.h -- C ABI of libmbglu.so: the decode-step dual-weight GLU GEMV on
 * GB300 (sm_103a).
 *
 *   out[m, n] = SiLU( sum_k h[m,k] * gate_w[n,k] ) * ( sum_k h[m,k] * up_w[n,k] )
 *
 * for a small batch (1 <= M <= 64) of bf16 hidden rows, reading the two
 * nn.Linear-layout weight matrices in place (no concatenated copy), with an
 * optional fused residual-add + zero-centred RMSNorm in front
 * (add_rmsnorm_glu and its one-kernel, strided and no-allocation forms).
 * Beside it, two ops of the same fused segment: silu_mul, the GLU epilogue
 * alone on projections a concatenated-weight GEMM has computed, and
 * gdn_gates, the gates of the gated-delta-net layers.
 *
 * Sources (DeepSpeed pull requests, as printed on their web pages):
 *   [8602/PlanB]   PR #8602 "feat(rollout): HybridEngineRollout graph capture
 *                  + segment-KI for Qwen3.5 hybrid", comment "Plan B:
 *                  Dual-Weight GEMV -- Investigation Results & Implementation"
 *                  (sections "Plan B Design: kernel adapts to the weights",
 *                  "Why cuBLAS-level performance is achievable at b=1").
 *   [8602/fused_glu] PR #8602 commit "expr(segment-ki): native CUDA fused_glu
 *                  kernel + GPU perf matrix" (single vs double rounding).
 *   [9057/Changes] PR #9057 "fix(module-inject): preserve HF precision
 *                  boundaries in segKI kernels", section "Changes"; its
 *                  commit "decode attention ... real row stride" (pass the
 *                  true row stride, fail closed on a mismatch).
 *
 * Conventions for every entry point:
 *   - bf16 values are passed as raw 16-bit patterns (mbglu_bf16).
 *   - Matrices are row-major; ld* are row strides in ELEMENTS, the K (inner)
 *     dimension is contiguous.
 *   - All data pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller (any allocator).  The library allocates nothing
 *     per call and keeps no state derived from the weights, so in-place
 *     weight updates are always seen.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream); no
 *     host synchronisation, no host reads of device data.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-zero status other than MBGLU_ERR_CUDA means nothing was launched
 *     (MBGLU_ERR_CUDA may follow kernels of the same call that did launch).
 *     No C++ exception crosses this boundary.
 *   - The fast kernels stream both weight matrices through shared memory
 *     with bulk asynchronous copies; they need gate_w/up_w 16-byte aligned,
 *     ld_gate and ld_up multiples of 8, and K a multiple of 8.  Other
 *     2-byte-aligned inputs run on a slower generic kernel with identical
 *     arithmetic rules.
 *   - Results are bitwise deterministic run to run (no atomics in any sum)
 *     and do not depend on where a row falls in the matrix.
 *   - A batch of 17..64 rows (PR #9057, the commit squashing the A100
 *     optimisation session, runs decode at batch 8, 32 and 64) runs in one
 *     pass over the weights on the fifth-generation tensor cores where
 *     glu_gemv's operands are 16-byte aligned with row strides that are
 *     multiples of 8 elements and K % 8 == 0.  Otherwise, and in the
 *     add_rmsnorm_glu entry points, it runs as row blocks of MBGLU_BLOCK_M =
 *     16 rows, the remainder last, each block a full pass over both weights
 *     (M = 64 streams them four times); each row's result is then the one a
 *     call on that row alone gives.
 */
#ifndef MBGLU_H
#define MBGLU_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MBGLU_ABI_VERSION 2
#define MBGLU_MAX_M 64     /* batch rows per call */
#define MBGLU_BLOCK_M 16   /* batch rows per pass over the weights */

typedef uint16_t mbglu_bf16;   /* raw bf16 bits */

/*
 * Rounding mode of the GLU epilogue.
 *  MBGLU_MODE_FUSED  single rounding: out = bf16( SiLU(g) * u ), g and u fp32
 *                    accumulations, SiLU and the product in fp32.
 *                    [8602/PlanB] kernel listing; [8602/fused_glu].
 *  MBGLU_MODE_HF     HF-boundary rounding, as the bf16 composite
 *                    F.silu(h @ Wg.T) * (h @ Wu.T) materialises it:
 *                    gb = bf16(g), ub = bf16(u), sb = bf16(SiLU(gb)) with SiLU
 *                    in fp32, out = bf16(sb * ub).
 *                    [8602/PlanB] b>1 fallback; [9057/Changes]: the GLU
 *                    keeps the bf16 roundings of HF's own code.
 * SiLU(x) = x / (1 + exp(-x)) with the precise expf and IEEE division,
 * evaluated from e^-|x| so that no intermediate overflows (silu_mul takes a
 * correctly rounded reciprocal in place of the division).
 */
typedef enum { MBGLU_MODE_FUSED = 0, MBGLU_MODE_HF = 1 } mbglu_mode;

typedef int mbglu_status;
#define MBGLU_OK            0
#define MBGLU_ERR_NULL      1   /* a required pointer is NULL */
#define MBGLU_ERR_SHAPE     2   /* M, N or K negative; M > MBGLU_MAX_M; K == 0 with the norm;
                                   add_rmsnorm_glu with one pass's rows above its shared-memory limit */
#define MBGLU_ERR_STRIDE    3   /* a leading dimension smaller than the row it holds */
#define MBGLU_ERR_ALIGN     4   /* a pointer not 2-byte aligned */
#define MBGLU_ERR_MODE      5   /* mode is neither FUSED nor HF */
#define MBGLU_ERR_ALIAS     6   /* an output overlaps an input it must not overlap */
#define MBGLU_ERR_CUDA      7   /* a CUDA runtime call failed; see mbglu_last_cuda_error() */
#define MBGLU_ERR_TIMEOUT   8   /* a bounded device-side wait gave up (reported by
                                   mbglu_read_device_error, never by a launch) */

/*
 * glu_gemv -- the dual-weight GLU GEMV.  [8602/PlanB] "Plan B Design": both
 * nn.Linear weights are used where they lie, the dot products accumulate in
 * fp32, and each output feature is SiLU of its gate product times its up
 * product.
 *
 *   h       [M, K] bf16, row stride ldh >= K          (read)
 *   gate_w  [N, K] bf16, row stride ld_gate >= K      (read, in place)
 *   up_w    [N, K] bf16, row stride ld_up >= K        (read, in place)
 *   out     [M, N] bf16, row stride ldo >= N          (written)
 *   0 <= M <= MBGLU_MAX_M, N >= 0, K >= 0.
 *   M == 0 or N == 0: no-op, MBGLU_OK.  K == 0: out = +0 (SiLU(0) * 0).
 *   out must not overlap h, gate_w or up_w (MBGLU_ERR_ALIAS).
 * Row strides are explicit because decode code slices operands out of fused
 * buffers ([9057/Changes] strided-view fixes: pass the real row stride, fail
 * closed on a mismatch).
 */
mbglu_status glu_gemv(const mbglu_bf16 *h, int64_t ldh,
                      const mbglu_bf16 *gate_w, int64_t ld_gate,
                      const mbglu_bf16 *up_w, int64_t ld_up,
                      mbglu_bf16 *out, int64_t ldo,
                      int M, int N, int K, mbglu_mode mode,
                      cudaStream_t stream);

/*
 * glu_backward -- the gradients of glu_gemv's exact composite
 * out = SiLU(h gate_w^T) * (h up_w^T) for an upstream gradient dout.
 * [8602/PlanB] "Plan B Design": the autograd wrapper works on the model's
 * own weight tensors, so their gradients land on those tensors (the
 * "Verification Results" compare them with the composite's).  In fp32 from
 * the bf16 operands:
 *   g, u     = the forward's dot products (fp32 accumulation)
 *   dG       = dout * u * SiLU'(g),  dU = dout * SiLU(g)        [M, N] fp32
 *   grad_h    = dG gate_w + dU up_w                              [M, K]
 *   grad_gate = dG^T h,  grad_up = dU^T h                        [N, K]
 * each gradient rounded once to bf16.  The HF mode's roundings have no
 * gradient of their own (casts pass gradients through), so this is the
 * backward of both modes.
 *   h, gate_w, up_w  as glu_gemv                              (read)
 *   dout     [M, N] bf16, row stride ldd >= N                 (read)
 *   grad_h   [M, K] bf16, row stride ldgh >= K, or NULL to skip it
 *   grad_gate, grad_up  [N, K] bf16, row strides ldgg, ldgu >= K; both
 *            NULL to skip them, or both given
 *   workspace  device memory of glu_backward_workspace_bytes(M, N, K)
 *            bytes, 16-byte aligned, owned by the caller; its contents are
 *            undefined afterwards
 *   0 <= M <= MBGLU_MAX_M, N >= 0, K >= 0.  K == 0: no-op.  M == 0 or
 *   N == 0: the gradients that remain are written as zeros (no workspace
 *   needed).  Batches above 16 rows compute dG and dU per 16-row block and
 *   grad_h per 8-row pass; the weight gradients sum over all M rows at once.
 * Outputs must not overlap the inputs, one another or the workspace
 * (MBGLU_ERR_ALIAS).  Asynchronous on `stream`; no allocation; the sums run
 * in a fixed order, so results are bitwise deterministic.
 */
size_t glu_backward_workspace_bytes(int M, int N, int K);
mbglu_status glu_backward(const mbglu_bf16 *h, int64_t ldh,
                          const mbglu_bf16 *gate_w, int64_t ld_gate,
                          const mbglu_bf16 *up_w, int64_t ld_up,
                          const mbglu_bf16 *dout, int64_t ldd,
                          mbglu_bf16 *grad_h, int64_t ldgh,
                          mbglu_bf16 *grad_gate, int64_t ldgg,
                          mbglu_bf16 *grad_up, int64_t ldgu,
                          int M, int N, int K,
                          void *workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * add_rmsnorm_glu -- residual add + zero-centred RMSNorm, then glu_gemv on
 * the normed rows.  [9057/Changes]: the residual add and the RMSNorm keep
 * HF's bf16 roundings, and the zero-centred scale (1 + w) is formed in fp32.
 *
 *   x         [M, K] bf16, contiguous                        (read)
 *   residual  [M, K] bf16, contiguous                        (read, then
 *             overwritten with s = bf16(x + residual): the updated residual
 *             stream the next layer needs)
 *   norm_w    [K] bf16                                       (read)
 *   eps       added to the mean square inside the root (e.g. 1e-6)
 *   gate_w, up_w  [N, K] bf16, contiguous (row stride K)     (read, in place)
 *   out       [M, N] bf16, contiguous                        (written)
 * Per row, in fp32:  var = mean_k s^2;  h = bf16( (s * rsqrt(var + eps)) *
 * (1 + (float)norm_w) );  then out = GLU(h) in `mode` (mode affects only
 * the GLU epilogue; s and h round to bf16 in both modes).
 *   1 <= K, 0 <= M <= MBGLU_MAX_M, and the rows of one pass must fit the
 *   kernel's shared-memory budget: min(M, MBGLU_BLOCK_M)*K <= 81920 (K <= 5120
 *   once M >= 16).
 *   out must not overlap any input; residual must not overlap x partially,
 *   nor norm_w, gate_w, up_w (MBGLU_ERR_ALIAS).  residual == x is allowed.
 * Two kernels run on `stream`: the residual add, then the GEMV, which reads
 * residual only after the add has completed (see the launch policy below
 * for what each may do before its predecessor has finished); above
 * MBGLU_BLOCK_M rows, the two per row block.
 */
mbglu_status add_rmsnorm_glu(const mbglu_bf16 *x, mbglu_bf16 *residual,
                             const mbglu_bf16 *norm_w, float eps,
                             const mbglu_bf16 *gate_w, const mbglu_bf16 *up_w,
                             mbglu_bf16 *out, int M, int N, int K,
                             mbglu_mode mode, cudaStream_t stream);

/*
 * add_rmsnorm_glu_ws -- the same operation and arguments as add_rmsnorm_glu,
 * as ONE kernel: every CTA forms s = bf16(x + residual) in shared memory for
 * the row statistic and arrives on a counter in `workspace` once it holds the
 * residual rows; at its end each CTA, after all have arrived (no CTA reads
 * residual any more), writes its slice of s to residual; the last one returns
 * the counters to zero.  Saves the residual-add launch and its dependency on
 * the critical path.
 *   workspace        device memory of at least MBGLU_WORKSPACE_BYTES,
 *                    16-byte aligned, owned by the caller, ALL ZERO before its
 *                    first use (cudaMemset once); every completed call leaves
 *                    it zero again.
 *   Calls that may run at the same time (on different streams, or in
 *   concurrently launched graphs) need different workspaces; consecutive
 *   calls on one stream may share one.  A call that does not complete (a
 *   bounded wait gave up, see mbglu_read_device_error) may leave it non-zero:
 *   zero it again before reuse.
 * Where the single kernel does not apply (operands not 16-byte aligned,
 * K % 8 != 0, or M*K*2 bytes of s not fitting beside the weight ring) the
 * call runs the two-kernel path of add_rmsnorm_glu and leaves the workspace
 * untouched.  Errors as add_rmsnorm_glu, plus MBGLU_ERR_NULL for a NULL
 * workspace, MBGLU_ERR_SHAPE for workspace_bytes < MBGLU_WORKSPACE_BYTES,
 * MBGLU_ERR_ALIGN, MBGLU_ERR_ALIAS if it overlaps an operand.
 */
#define MBGLU_WORKSPACE_BYTES 256
mbglu_status add_rmsnorm_glu_ws(const mbglu_bf16 *x, mbglu_bf16 *residual,
                                const mbglu_bf16 *norm_w, float eps,
                                const mbglu_bf16 *gate_w, const mbglu_bf16 *up_w,
                                mbglu_bf16 *out, int M, int N, int K,
                                mbglu_mode mode, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * add_rmsnorm_glu_strided -- add_rmsnorm_glu (or, with a workspace,
 * add_rmsnorm_glu_ws) on weights and an output with explicit row strides:
 * gate_w and up_w [N][K] with row strides ld_gate, ld_up >= K, out [M][N]
 * with row stride ldo >= N (elements), e.g. views into a packed parameter
 * buffer or a wider activation buffer.  PR #9057, the decode-attention
 * stride commit: kernels take the true row stride instead of assuming a
 * contiguous tensor, and reject a stride that cannot hold the row.  x,
 * residual and norm_w stay contiguous.  workspace: NULL runs the two-kernel
 * path; otherwise as add_rmsnorm_glu_ws (MBGLU_WORKSPACE_BYTES, 16-byte
 * aligned, zero before first use).  Errors as add_rmsnorm_glu_ws, plus
 * MBGLU_ERR_STRIDE for ld_gate < K, ld_up < K or ldo < N.  Strides that are
 * not multiples of 8 elements run the generic kernel.
 */
mbglu_status add_rmsnorm_glu_strided(const mbglu_bf16 *x, mbglu_bf16 *residual,
                                     const mbglu_bf16 *norm_w, float eps,
                                     const mbglu_bf16 *gate_w, int64_t ld_gate,
                                     const mbglu_bf16 *up_w, int64_t ld_up,
                                     mbglu_bf16 *out, int64_t ldo, int M, int N, int K,
                                     mbglu_mode mode, void *workspace, size_t workspace_bytes,
                                     cudaStream_t stream);

/*
 * add_rmsnorm_glu_noalloc -- add_rmsnorm_glu_ws for callers that cannot
 * allocate device memory: code running where the memory is owned by someone
 * else (a serving runtime's planner, a plugin host, a framework that hands
 * out only the tensors of the op), or where cudaMalloc is not allowed at all
 * (inside stream capture, in paths that must not synchronise the device).
 * No counterpart on the pages: it exists for such callers only.
 * Same arguments as add_rmsnorm_glu; the caller still provides every input and
 * output.  The workspace the single kernel needs comes from a fixed device
 * array inside the library, MBGLU_NOALLOC_SCRATCH_BYTES per GPU, held by every
 * GPU that loads the library until the process exits; a call needing more
 * than that returns MBGLU_ERR_SHAPE.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it with the identity of the device's
 *     context: make that first call before any stream capture on that device.
 *     After a cudaDeviceReset the next call sees a new context and looks the
 *     address up again (so that call, too, belongs outside stream capture).
 *   - Each call clears the counters with a stream-ordered cudaMemsetAsync
 *     before its kernel, because the array keeps what the last call left.
 *   - All calls share the one array: calls that may overlap on the GPU (on
 *     different streams, or in concurrently running graphs) race on it and
 *     give wrong results.  Use add_rmsnorm_glu_ws with one workspace per stream
 *     for that.
 * Falls back to the two-kernel path (scratch untouched) exactly where
 * add_rmsnorm_glu_ws does.  Errors as add_rmsnorm_glu_ws.
 */
#define MBGLU_NOALLOC_SCRATCH_BYTES 256
mbglu_status add_rmsnorm_glu_noalloc(const mbglu_bf16 *x, mbglu_bf16 *residual,
                                     const mbglu_bf16 *norm_w, float eps,
                                     const mbglu_bf16 *gate_w, const mbglu_bf16 *up_w,
                                     mbglu_bf16 *out, int M, int N, int K,
                                     mbglu_mode mode, cudaStream_t stream);

/*
 * silu_mul -- the GLU epilogue alone, on projections computed elsewhere: the
 * prefill / large-batch route, where one GEMM on a concatenated [gate; up]
 * weight leaves both projections side by side.  DeepSpeed PR #8602, commit
 * "expr(segment-ki): native CUDA fused_glu kernel + GPU perf matrix": a fused
 * silu-mul kernel on the "halves layout", with single rounding against the
 * composite's double rounding.
 *   x    [M][2N] bf16, row stride ldx >= 2N elements: the gate projection in
 *        columns [0, N), the up projection in columns [N, 2N).
 *   out  [M][N] bf16, row stride ldo >= N elements; must not overlap x.
 *   mode MBGLU_MODE_FUSED: out = bf16(SiLU(g) * u), one rounding;
 *        MBGLU_MODE_HF:    out = bf16(bf16(SiLU(g)) * u), F.silu(g) * u on
 *        bf16 tensors (g and u are bf16 already).
 * Device pointers owned by the caller; asynchronous on `stream`, no
 * allocation, capturable.  Any M >= 0 (no batch limit).  M == 0 or N == 0 is
 * a no-op.  Errors: MBGLU_ERR_MODE, MBGLU_ERR_SHAPE (M or N negative, or 2N
 * beyond INT32_MAX),
 * MBGLU_ERR_NULL, MBGLU_ERR_STRIDE (ldx < 2N or ldo < N), MBGLU_ERR_ALIGN (a
 * pointer not 2-byte aligned), MBGLU_ERR_ALIAS (out overlaps x),
 * MBGLU_ERR_CUDA.  16-byte aligned rows with N % 8 == 0 take the vectorised
 * path; anything else runs element by element, with the same results.
 */
mbglu_status silu_mul(const mbglu_bf16 *x, int64_t ldx, mbglu_bf16 *out, int64_t ldo,
                      int M, int N, mbglu_mode mode, cudaStream_t stream);

/*
 * gdn_gates -- the decay and write gates of the gated-delta-net layers, which
 * the same segment-KI work fuses beside the GLU.  DeepSpeed PR #8602, the
 * commit adding gdn_gates: a sigmoid write gate and the decay gate
 * -exp(A_log) * softplus(a + dt_bias), computed in fp32 with the stable
 * softplus form, on strided input; PR #9057 "Changes": the decay gates stay
 * fp32.  For token t < T and head j < H:
 *   x = a[t][j] + dt_bias[j]                 (fp32 addition; a is bf16)
 *   g[t][j]    = -exp(A_log[j]) * softplus(x)   fp32, softplus(x) = log(1 + e^x)
 *                                                 in its stable form
 *   beta[t][j] = bf16(sigmoid(b[t][j]))         one rounding
 *   a, b     [T][H] bf16 with row strides lda, ldb >= H (views into a wider
 *            projection output are fine);
 *   A_log, dt_bias  [H] fp32 (bf16 parameters widen exactly);
 *   g        [T][H] fp32, row stride ldg >= H; beta [T][H] bf16, ldbeta >= H;
 *            neither may overlap an input or the other output.
 * Device pointers owned by the caller; asynchronous on `stream`; no
 * allocation.  T == 0 or H == 0 is a no-op.  Errors: MBGLU_ERR_SHAPE (T or H
 * negative), MBGLU_ERR_NULL, MBGLU_ERR_STRIDE, MBGLU_ERR_ALIGN (bf16 pointers
 * not 2-byte, fp32 pointers not 4-byte aligned), MBGLU_ERR_ALIAS,
 * MBGLU_ERR_CUDA.
 */
mbglu_status gdn_gates(const mbglu_bf16 *a, int64_t lda, const mbglu_bf16 *b, int64_t ldb,
                       const float *A_log, const float *dt_bias,
                       float *g, int64_t ldg, mbglu_bf16 *beta, int64_t ldbeta,
                       int T, int H, cudaStream_t stream);

/*
 * Launch policy, process-wide (default MBGLU_POLICY_PREFETCH).  It decides how
 * a call's kernels are ordered after the kernel that precedes them on the
 * stream; results are identical under every policy.
 *   MBGLU_POLICY_SERIAL    plain stream-ordered launches.
 *   MBGLU_POLICY_PDL       programmatic dependent launch: the kernels may be
 *                          scheduled while the preceding kernel drains, but
 *                          read and write nothing in global memory before it
 *                          has completed.
 *   MBGLU_POLICY_PREFETCH  as PDL, and the first weight stages (gate_w and
 *                          up_w only) are requested before that wait, so a
 *                          decode step's back-to-back calls overlap one call's
 *                          tail with the next call's ramp.  Contract: the
 *                          kernel immediately preceding a call on its stream
 *                          must not write gate_w / up_w after releasing its
 *                          dependents early (kernels that do not use
 *                          programmatic dependent launch never do: they
 *                          release at completion).  Use SERIAL or PDL around
 *                          custom early-releasing kernels that update weights.
 * Returns MBGLU_ERR_MODE for an unknown value.
 */
#define MBGLU_POLICY_SERIAL   0
#define MBGLU_POLICY_PDL      1
#define MBGLU_POLICY_PREFETCH 2
mbglu_status mbglu_set_launch_policy(int policy);
int mbglu_get_launch_policy(void);

/* Human-readable name of a status code (static storage). */
const char *mbglu_status_string(mbglu_status s);

/* MBGLU_ABI_VERSION of the loaded library. */
int mbglu_abi_version(void);

/* cudaError_t of the most recent failing CUDA call made by this library on
 * the calling host thread (0 if none). */
int mbglu_last_cuda_error(void);

/* Which kernel the calling thread's last successful call launched:
 * 0 none (no-op), 1 streaming kernel (CUDA-core FMA), 2 generic kernel,
 * 3 zero fill, 4 tensor-core kernel with h in shared memory (batch >= 3),
 * 5 silu_mul, 6 gdn_gates, 7 row blocks (a batch above MBGLU_BLOCK_M: one
 * of 1, 2, 4, 10 per block), 8 glu_backward, 9 the tcgen05 kernel (a batch
 * above MBGLU_BLOCK_M in one pass), 10 the K-slice tensor-core kernel (h's
 * fragments in registers, batch 1..16). */
int mbglu_last_variant(void);

/* Which kernels the calling thread's last glu_backward took for the
 * gradients' second step: 0 none (the call launched no such step), 1 the
 * separate grad_h and weight-gradient kernels, 2 one pass on the CUDA cores
 * (M <= 2, or the tensor-core pass off), 3 one pass on the tensor cores
 * (M = 3..16; mma.sync; dG and dU enter as three bf16 terms, exact for
 * normal fp32 values).  The one-pass kernels need K % 8 == 0, 16-byte
 * aligned weights and weight gradients with row strides of whole 16-byte
 * units, and M <= 8 (CUDA cores) or M <= 16 (tensor cores). */
int mbglu_last_backward_path(void);

/* How many row blocks of the calling thread's last add_rmsnorm_glu* call ran
 * as the single kernel (the workspace / no-allocation paths); 0 when every
 * block took the two-kernel path or the call launched nothing. */
int mbglu_last_single_kernel_blocks(void);

/* Diagnostics: copies the first `count` ints of the current device's
 * add_rmsnorm_glu_noalloc scratch array to host memory `words`, after a
 * cudaDeviceSynchronize.  SYNCHRONOUS.  MBGLU_ERR_NULL for a null `words`,
 * MBGLU_ERR_SHAPE for count < 0 or beyond MBGLU_NOALLOC_SCRATCH_BYTES,
 * MBGLU_ERR_CUDA on a CUDA failure. */
mbglu_status mbglu_noalloc_scratch_read(int *words, int count);

/*
 * Reads and clears the device error word of the current device.  Kernels
 * never trap: a bounded wait that gives up records MBGLU_ERR_TIMEOUT here and
 * the kernel returns.  SYNCHRONOUS: waits for the device to finish its work.
 * Returns MBGLU_OK or MBGLU_ERR_CUDA; *word receives the recorded code.
 */
mbglu_status mbglu_read_device_error(int *word);

#ifdef __cplusplus
}
#endif

#endif /* MBGLU_H */
