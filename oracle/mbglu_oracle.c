/*
 * mbglu_oracle.c -- plain, slow, fp64 CPU oracle for the dual-weight GLU GEMV
 * and its fused residual-add + zero-centred RMSNorm prologue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that the tests, the smoke check and the
 * benchmark's CPU-baseline leg can check the CUDA library against an
 * independent, obviously-correct statement of what it computes.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Sources (DeepSpeed pull requests, as printed on their web pages):
 *   [8602/PlanB]  PR #8602 "feat(rollout): HybridEngineRollout graph capture
 *                 + segment-KI for Qwen3.5 hybrid", comment "Plan B:
 *                 Dual-Weight GEMV -- Investigation Results & Implementation",
 *                 section "Plan B Design: kernel adapts to the weights".
 *   [8602/fused_glu] PR #8602 commit "expr(segment-ki): native CUDA fused_glu
 *                 kernel + GPU perf matrix" (single vs double rounding).
 *   [8602/old-ki] PR #8602 commit "expr(old-ki): KV cache write-back +
 *                 numerics bisection" (RMSNorm must not accumulate in bf16).
 *   [9057/Changes] PR #9057 "fix(module-inject): preserve HF precision
 *                 boundaries in segKI kernels", section "Changes".
 *
 * Every floating-point step below is done in IEEE binary64 with
 * -ffp-contract=off, so the result is the same on every host.  bf16 values
 * travel as their raw 16-bit patterns (uint16_t).
 *
 * Parity pins: every function here is pinned by the CPU test suite against
 * exact rational arithmetic, arbitrary-precision SiLU, closed forms and a
 * library composite; none is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ABI_VERSION 1

enum { ORACLE_MODE_FUSED = 0, ORACLE_MODE_HF = 1 };

int oracle_abi_version(void) { return ORACLE_ABI_VERSION; }

/* ------------------------------------------------------------------------ */
/* bf16 <-> binary64                                                         */
/* ------------------------------------------------------------------------ */

/* Exact widening: a bf16 pattern is the top half of a binary32 pattern. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a binary64 value to the nearest bf16, ties to even, directly from the
 * double's bits (no detour through binary32, which would round twice).
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored significand bits.
 * Normal numbers have 8 significant bits; below 2^-126 the spacing is fixed
 * at 2^-133 (subnormals).  Results beyond the largest finite bf16 round to
 * +-inf as IEEE round-to-nearest prescribes.  NaN maps to a quiet NaN with
 * the input's sign.  [8602/PlanB]: the kernel's single final rounding is
 * __float2bfloat16_rn, i.e. round-to-nearest-even.
 */
uint16_t oracle_bf16_round(double x)
{
    uint64_t u;
    memcpy(&u, &x, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 63) << 15);
    const int bexp = (int)((u >> 52) & 0x7ff);
    const uint64_t frac = u & ((UINT64_C(1) << 52) - 1);

    if (bexp == 0x7ff)                      /* inf or NaN */
        return (uint16_t)(sign | (frac ? 0x7fc0 : 0x7f80));
    if (bexp == 0 && frac == 0)             /* +-0 */
        return sign;

    /* value = sig * 2^(e - 52) with sig < 2^53 */
    uint64_t sig;
    int e;
    if (bexp == 0) {                        /* binary64 subnormal */
        sig = frac;
        e = -1022;
    } else {
        sig = frac | (UINT64_C(1) << 52);
        e = bexp - 1023;
    }

    /* exponent of one bf16 unit in the last place at this magnitude */
    const int q = (e >= -126) ? (e - 7) : -133;
    const int shift = 52 + q - e;           /* >= 45 */
    uint64_t n;
    if (shift >= 54) {
        n = 0;                              /* below half a unit: rounds to 0 */
    } else {
        n = sig >> shift;
        const uint64_t rem = sig & ((UINT64_C(1) << shift) - 1);
        const uint64_t half = UINT64_C(1) << (shift - 1);
        if (rem > half || (rem == half && (n & 1)))
            n += 1;
    }

    uint32_t bits;
    if (q == -133) {
        bits = (uint32_t)n;                 /* subnormal; n == 128 is 2^-126 */
    } else {
        /* n in [128, 256]; a carry to 256 moves into the exponent field */
        const int64_t b = ((int64_t)(e + 127) << 7) + (int64_t)n - 128;
        bits = (b >= 0x7f80) ? 0x7f80u : (uint32_t)b;
    }
    return (uint16_t)(sign | bits);
}

/* oracle_bf16_round over an array: out[i] = oracle_bf16_round(x[i]). */
void oracle_bf16_round_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}

/* ------------------------------------------------------------------------ */
/* SiLU                                                                      */
/* ------------------------------------------------------------------------ */

/*
 * SiLU(x) = x * sigmoid(x) = x / (1 + e^-x).  The pages use the name only
 * ([8602/PlanB] applies SILU(gate_acc) to the gate dot product; its b>1
 * fallback calls F.silu); this is the standard definition F.silu computes.
 */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* ------------------------------------------------------------------------ */
/* GLU GEMV                                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *h;
    int64_t ldh;
    const uint16_t *gate_w;
    int64_t ld_gate;
    const uint16_t *up_w;
    int64_t ld_up;
    uint16_t *out;
    int64_t ldo;
    int M, N, K, mode;
    double *G, *U, *Ag, *Au;   /* optional [M*N] diagnostics, row-major */
    int n0, n1;                /* this worker's output features */
} glu_job;

/*
 * For each batch row m and output feature n ([8602/PlanB]: the listed
 * kernel gives every output feature a warp of its own):
 *   G = sum_k h[m,k] * W_gate[n,k]      (the gate dot product)
 *   U = sum_k h[m,k] * W_up[n,k]        (the up dot product)
 * Each bf16 x bf16 product is exact in binary64 (8 + 8 significant bits), and
 * the sum runs in k order.
 *
 * mode FUSED ([8602/PlanB] kernel listing; [8602/fused_glu], the fused
 * kernel rounds once where the composite rounds twice):
 * out = bf16( SiLU(G) * U ), one rounding at the end.
 *
 * mode HF ([8602/PlanB] b>1 fallback F.silu(hidden @ gate_w.T) *
 * (hidden @ up_w.T) on bf16 tensors; [9057/Changes]: the GLU keeps the bf16
 * roundings of HF's own code): every tensor the bf16 composite materialises
 * is rounded --
 *   gb = bf16(G), ub = bf16(U), sb = bf16(SiLU(gb)), out = bf16(sb * ub).
 */
static void glu_rows(const glu_job *j)
{
    for (int m = 0; m < j->M; ++m) {
        const uint16_t *hrow = j->h + (int64_t)m * j->ldh;
        for (int n = j->n0; n < j->n1; ++n) {
            const uint16_t *grow = j->gate_w + (int64_t)n * j->ld_gate;
            const uint16_t *urow = j->up_w + (int64_t)n * j->ld_up;
            double G = 0.0, U = 0.0, Ag = 0.0, Au = 0.0;
            for (int k = 0; k < j->K; ++k) {
                const double hk = oracle_bf16_to_double(hrow[k]);
                const double pg = hk * oracle_bf16_to_double(grow[k]);
                const double pu = hk * oracle_bf16_to_double(urow[k]);
                G += pg;
                U += pu;
                Ag += fabs(pg);
                Au += fabs(pu);
            }
            uint16_t o;
            if (j->mode == ORACLE_MODE_FUSED) {
                o = oracle_bf16_round(oracle_silu(G) * U);
            } else {
                const uint16_t gb = oracle_bf16_round(G);
                const uint16_t ub = oracle_bf16_round(U);
                const uint16_t sb = oracle_bf16_round(oracle_silu(oracle_bf16_to_double(gb)));
                o = oracle_bf16_round(oracle_bf16_to_double(sb) * oracle_bf16_to_double(ub));
            }
            j->out[(int64_t)m * j->ldo + n] = o;
            const int64_t d = (int64_t)m * j->N + n;
            if (j->G) j->G[d] = G;
            if (j->U) j->U[d] = U;
            if (j->Ag) j->Ag[d] = Ag;
            if (j->Au) j->Au[d] = Au;
        }
    }
}

static void *glu_worker(void *arg)
{
    glu_rows((const glu_job *)arg);
    return NULL;
}

/*
 * Returns 0 on success, -1 on bad arguments.  The output features are split
 * into contiguous ranges, one per thread; every output is computed by
 * exactly the code above, so the thread count changes nothing but the wall
 * time.
 */
int oracle_glu_gemv(const uint16_t *h, int64_t ldh,
                    const uint16_t *gate_w, int64_t ld_gate,
                    const uint16_t *up_w, int64_t ld_up,
                    uint16_t *out, int64_t ldo,
                    int M, int N, int K, int mode,
                    double *G, double *U, double *Ag, double *Au,
                    int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (mode != ORACLE_MODE_FUSED && mode != ORACLE_MODE_HF) return -1;
    if (M == 0 || N == 0) return 0;
    if (!out || (K > 0 && (!h || !gate_w || !up_w))) return -1;
    if (ldo < N || (K > 0 && (ldh < K || ld_gate < K || ld_up < K))) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = N;
    if (nthreads > 256) nthreads = 256;

    glu_job jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < nthreads; ++t) {
        glu_job *j = &jobs[t];
        j->h = h; j->ldh = ldh;
        j->gate_w = gate_w; j->ld_gate = ld_gate;
        j->up_w = up_w; j->ld_up = ld_up;
        j->out = out; j->ldo = ldo;
        j->M = M; j->N = N; j->K = K; j->mode = mode;
        j->G = G; j->U = U; j->Ag = Ag; j->Au = Au;
        j->n0 = (int)(((int64_t)N * t) / nthreads);
        j->n1 = (int)(((int64_t)N * (t + 1)) / nthreads);
    }
    if (nthreads == 1) {
        glu_rows(&jobs[0]);
        return 0;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, glu_worker, &jobs[t]) != 0) break;
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    for (int t = started; t < nthreads; ++t) glu_rows(&jobs[t]);  /* any that did not start */
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Residual add + zero-centred RMSNorm                                       */
/* ------------------------------------------------------------------------ */

/*
 * For each row m ([9057/Changes]: the residual add and the RMSNorm keep HF's
 * bf16 roundings, and the zero-centred scale (1 + w) is formed in fp32;
 * [8602/old-ki] the statistic must not be accumulated in bf16):
 *   s[k]  = bf16(x[k] + r[k])                      the updated residual stream
 *   var   = (1/K) * sum_k s[k]^2
 *   h[k]  = bf16( s[k] / sqrt(var + eps) * (1 + w[k]) )
 * eps is the caller's binary32 value, widened exactly.  s_out receives the
 * residual sum, h_out the normed hidden row that feeds the GLU GEMV.
 * Returns 0, or -1 on bad arguments (K == 0 has no mean).
 */
int oracle_add_rmsnorm(const uint16_t *x, const uint16_t *residual,
                       const uint16_t *norm_w, float eps,
                       int M, int K, uint16_t *s_out, uint16_t *h_out)
{
    if (M < 0 || K <= 0) return -1;
    if (M == 0) return 0;
    if (!x || !residual || !norm_w || !s_out || !h_out) return -1;
    const double e = (double)eps;
    for (int m = 0; m < M; ++m) {
        const uint16_t *xr = x + (int64_t)m * K;
        const uint16_t *rr = residual + (int64_t)m * K;
        uint16_t *sr = s_out + (int64_t)m * K;
        uint16_t *hr = h_out + (int64_t)m * K;
        double ss = 0.0;
        for (int k = 0; k < K; ++k) {
            sr[k] = oracle_bf16_round(oracle_bf16_to_double(xr[k]) +
                                      oracle_bf16_to_double(rr[k]));
            const double sv = oracle_bf16_to_double(sr[k]);
            ss += sv * sv;
        }
        const double var = ss / (double)K;
        const double rms = sqrt(var + e);
        for (int k = 0; k < K; ++k) {
            const double sv = oracle_bf16_to_double(sr[k]);
            const double scale = 1.0 + oracle_bf16_to_double(norm_w[k]);
            hr[k] = oracle_bf16_round(sv / rms * scale);
        }
    }
    return 0;
}

/*
 * The whole fused segment: residual add + norm, then the GLU GEMV on the
 * normed rows.  residual is in/out: it receives s = bf16(x + residual).
 * mode selects the GLU epilogue only; s and h round to bf16 in both modes.
 * Returns 0, -1 on bad arguments, -2 if host memory ran out.
 */
int oracle_add_rmsnorm_glu(const uint16_t *x, uint16_t *residual,
                           const uint16_t *norm_w, float eps,
                           const uint16_t *gate_w, const uint16_t *up_w,
                           uint16_t *out, int M, int N, int K, int mode,
                           uint16_t *h_out, int nthreads)
{
    if (M < 0 || N < 0 || K <= 0) return -1;
    if (M == 0) return 0;
    const size_t cnt = (size_t)M * (size_t)K;
    uint16_t *s = (uint16_t *)malloc(cnt * sizeof *s);
    uint16_t *h = h_out ? h_out : (uint16_t *)malloc(cnt * sizeof *h);
    if (!s || !h) { free(s); if (!h_out) free(h); return -2; }
    int rc = oracle_add_rmsnorm(x, residual, norm_w, eps, M, K, s, h);
    if (rc == 0 && N > 0)
        rc = oracle_glu_gemv(h, K, gate_w, K, up_w, K, out, N, M, N, K, mode,
                             NULL, NULL, NULL, NULL, nthreads);
    if (rc == 0) memcpy(residual, s, cnt * sizeof *s);
    free(s);
    if (!h_out) free(h);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* silu_mul: the GLU epilogue on projections already computed              */
/* ------------------------------------------------------------------------ */

/*
 * The standalone epilogue of the prefill / large-batch route
 * ([8602/fused_glu]: a native kernel that applies SiLU and the product to
 * the two halves of each row in place, rounding once where the composite
 * rounds twice).  Each row of x holds both projections side by side, as a GEMM on
 * the concatenated [gate; up] weight leaves them: the gate half in columns
 * [0, N) and the up half in columns [N, 2N).  For every m < M, n < N:
 *   g = x[m, n], u = x[m, N + n]                 (bf16, exact in binary64)
 *   mode FUSED: out = bf16( SiLU(g) * u )        one rounding
 *   mode HF:    out = bf16( bf16(SiLU(g)) * u )  F.silu(g) * u on bf16 tensors
 * g and u are bf16 already, so the HF rounding of the two projections is the
 * identity here.  ldx >= 2N and ldo >= N are row strides in elements.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_silu_mul(const uint16_t *x, int64_t ldx, uint16_t *out, int64_t ldo, int M, int N, int mode)
{
    if (M < 0 || N < 0) return -1;
    if (mode != ORACLE_MODE_FUSED && mode != ORACLE_MODE_HF) return -1;
    if (M == 0 || N == 0) return 0;
    if (!x || !out || ldx < 2 * (int64_t)N || ldo < N) return -1;
    for (int m = 0; m < M; ++m) {
        const uint16_t *gate = x + (int64_t)m * ldx;
        const uint16_t *up = gate + N;
        for (int n = 0; n < N; ++n) {
            const double g = oracle_bf16_to_double(gate[n]);
            const double u = oracle_bf16_to_double(up[n]);
            uint16_t o;
            if (mode == ORACLE_MODE_FUSED) {
                o = oracle_bf16_round(oracle_silu(g) * u);
            } else {
                const uint16_t sb = oracle_bf16_round(oracle_silu(g));
                o = oracle_bf16_round(oracle_bf16_to_double(sb) * u);
            }
            out[(int64_t)m * ldo + n] = o;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* gdn_gates: the decay and write gates of the gated-delta-net layers       */
/* ------------------------------------------------------------------------ */

/*
 * The gates the same segment-KI work fuses beside the GLU ([8602/fused_glu],
 * the gdn_gates commit: the sigmoid write gate and the decay gate
 * -exp(A_log) * softplus(a + dt_bias) computed in fp32 with the stable
 * softplus form, on strided inputs read in place; [9057/Changes]: the decay
 * gates stay fp32).  For every token t < T and head j < H:
 *   x    = fp32( a[t, j] + dt_bias[j] )       the binary32 addition the fp32
 *                                             math performs (a is bf16)
 *   g    = -exp(A_log[j]) * softplus(x)       returned in binary64
 *   beta = bf16( sigmoid(b[t, j]) )           one rounding
 * with softplus(x) = log(1 + e^x) (PyTorch's F.softplus returns x itself for
 * x > 20, which differs from log(1 + e^x) by less than 2^-64 relative) and
 * sigmoid(y) = 1 / (1 + e^-y).  The exact values are computed in binary64;
 * the stable forms (x + log1p(e^-x) for x > 0) keep every digit.
 * Returns 0, or -1 on bad arguments.
 */
static double oracle_softplus(double x)
{
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

int oracle_gdn_gates(const uint16_t *a, int64_t lda, const uint16_t *b, int64_t ldb,
                     const float *A_log, const float *dt_bias,
                     double *g, uint16_t *beta, int T, int H)
{
    if (T < 0 || H < 0) return -1;
    if (T == 0 || H == 0) return 0;
    if (!a || !b || !A_log || !dt_bias || !g || !beta || lda < H || ldb < H) return -1;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < H; ++j) {
            const float x = (float)oracle_bf16_to_double(a[(int64_t)t * lda + j]) + dt_bias[j];
            g[(int64_t)t * H + j] = -exp((double)A_log[j]) * oracle_softplus((double)x);
            const double y = oracle_bf16_to_double(b[(int64_t)t * ldb + j]);
            beta[(int64_t)t * H + j] = oracle_bf16_round(1.0 / (1.0 + exp(-y)));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward of the dual-weight GLU GEMV                                      */
/* ------------------------------------------------------------------------ */

/*
 * [8602/PlanB]: the autograd wrapper saves (hidden, gate_w, up_w) so that
 * the gradients reach the original Parameters; its three gradients matched
 * the composite F.silu(h @ Wg.T) * (h @ Wu.T) exactly in fp32 (section
 * "Verification Results").
 * So the backward is the gradient of out = SiLU(G) * U with G = h . Wg[n],
 * U = h . Wu[n], for an upstream gradient dout [M][N]:
 *   SiLU'(G) = s (1 + G (1 - s)),  s = 1 / (1 + e^-G)
 *   dG[m,n]  = dout[m,n] * U * SiLU'(G)
 *   dU[m,n]  = dout[m,n] * SiLU(G)
 *   grad_h[m,k]  = sum_n dG[m,n] Wg[n,k] + dU[m,n] Wu[n,k]   (n in order)
 *   grad_Wg[n,k] = sum_m dG[m,n] h[m,k]                     (m in order)
 *   grad_Wu[n,k] = sum_m dU[m,n] h[m,k]
 * Everything in binary64 on the exact bf16 inputs; the gradients are returned
 * in binary64 ([M][K], [N][K], [N][K], row-major, contiguous).
 */
typedef struct {
    const uint16_t *h, *gate_w, *up_w, *dout;
    int64_t ldh, ld_gate, ld_up, ldd;
    int M, N, K;
    double *dG, *dU;                 /* [M][N] scratch */
    double *grad_h, *grad_gate, *grad_up;
    int lo, hi;                      /* this worker's n (phase 1) or k (phase 2) range */
} bwd_job;

static void bwd_rows(const bwd_job *j)   /* phase 1: dG, dU, and the weight gradients of rows [lo, hi) */
{
    for (int n = j->lo; n < j->hi; ++n) {
        const uint16_t *grow = j->gate_w + (int64_t)n * j->ld_gate;
        const uint16_t *urow = j->up_w + (int64_t)n * j->ld_up;
        for (int m = 0; m < j->M; ++m) {
            const uint16_t *hrow = j->h + (int64_t)m * j->ldh;
            double G = 0.0, U = 0.0;
            for (int k = 0; k < j->K; ++k) {
                const double hk = oracle_bf16_to_double(hrow[k]);
                G += hk * oracle_bf16_to_double(grow[k]);
                U += hk * oracle_bf16_to_double(urow[k]);
            }
            const double s = 1.0 / (1.0 + exp(-G));
            const double d = oracle_bf16_to_double(j->dout[(int64_t)m * j->ldd + n]);
            j->dG[(int64_t)m * j->N + n] = d * U * (s * (1.0 + G * (1.0 - s)));
            j->dU[(int64_t)m * j->N + n] = d * oracle_silu(G);
        }
        for (int k = 0; k < j->K; ++k) {
            double sg = 0.0, su = 0.0;
            for (int m = 0; m < j->M; ++m) {
                const double hk = oracle_bf16_to_double(j->h[(int64_t)m * j->ldh + k]);
                sg += j->dG[(int64_t)m * j->N + n] * hk;
                su += j->dU[(int64_t)m * j->N + n] * hk;
            }
            j->grad_gate[(int64_t)n * j->K + k] = sg;
            j->grad_up[(int64_t)n * j->K + k] = su;
        }
    }
}

static void bwd_cols(const bwd_job *j)   /* phase 2: grad_h for columns [lo, hi) */
{
    for (int m = 0; m < j->M; ++m)
        for (int k = j->lo; k < j->hi; ++k) {
            double acc = 0.0;
            for (int n = 0; n < j->N; ++n) {
                acc += j->dG[(int64_t)m * j->N + n] * oracle_bf16_to_double(j->gate_w[(int64_t)n * j->ld_gate + k]);
                acc += j->dU[(int64_t)m * j->N + n] * oracle_bf16_to_double(j->up_w[(int64_t)n * j->ld_up + k]);
            }
            j->grad_h[(int64_t)m * j->K + k] = acc;
        }
}

static void *bwd_rows_worker(void *arg) { bwd_rows((const bwd_job *)arg); return NULL; }
static void *bwd_cols_worker(void *arg) { bwd_cols((const bwd_job *)arg); return NULL; }

/* Splits [0, total) over nthreads workers running fn; the split changes only the wall time. */
static void bwd_run(bwd_job *base, int total, int nthreads, void *(*fn)(void *))
{
    bwd_job jobs[256];
    pthread_t tids[256];
    if (nthreads > total) nthreads = total;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *base;
        jobs[t].lo = (int)(((int64_t)total * t) / nthreads);
        jobs[t].hi = (int)(((int64_t)total * (t + 1)) / nthreads);
    }
    for (int t = 0; t < nthreads; ++t) {
        if (nthreads == 1 || pthread_create(&tids[t], NULL, fn, &jobs[t]) != 0) break;
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    for (int t = started; t < nthreads; ++t) fn(&jobs[t]);
}

/* Returns 0, or -1 on bad arguments (the scratch is the caller's dG, dU [M][N]). */
int oracle_glu_backward(const uint16_t *h, int64_t ldh, const uint16_t *gate_w, int64_t ld_gate,
                        const uint16_t *up_w, int64_t ld_up, const uint16_t *dout, int64_t ldd,
                        int M, int N, int K, double *dG, double *dU,
                        double *grad_h, double *grad_gate, double *grad_up, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0 || K == 0) return 0;
    if (!h || !gate_w || !up_w || !dout || !dG || !dU || !grad_h || !grad_gate || !grad_up) return -1;
    if (ldh < K || ld_gate < K || ld_up < K || ldd < N) return -1;
    bwd_job base = {h, gate_w, up_w, dout, ldh, ld_gate, ld_up, ldd, M, N, K, dG, dU,
                    grad_h, grad_gate, grad_up, 0, 0};
    bwd_run(&base, N, nthreads, bwd_rows_worker);   /* every dG, dU before any grad_h */
    bwd_run(&base, K, nthreads, bwd_cols_worker);
    return 0;
}
