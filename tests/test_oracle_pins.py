"""Pins for the fp64 CPU oracle: checks against things other than itself.

Each test ties the oracle to exact rational arithmetic, 120-bit SiLU, a
closed form, an invariant or a library routine, so that a plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a
wrong tie rule) fails at least one of them.  ``test_oracle_mutations.py``
plants such slips in a copy of the oracle and checks they are caught.

Method sources: DeepSpeed PR #8602 "Plan B: Dual-Weight GEMV" (kernel listing:
fp32 dot products, SiLU(gate)*up, one round-to-nearest-even to bf16; b>1
fallback F.silu(h@Wg.T)*(h@Wu.T) on bf16 tensors) and PR #9057 "Changes"
(the residual sum, the normed row and the GLU's intermediates round to bf16
as HF's modules do; the zero-centred norm scale is formed in fp32).
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import glu_inputs as gi
from exact_ref import (bf16_bits_to_fraction, fraction_to_mpf, glu_exact, mpf_to_fraction, rmsnorm_exact_row,
                       rne_bf16, silu_exact)
import tolerance as tol

mpmath = pytest.importorskip("mpmath")
EPS32 = float(np.float32(1e-6))


def f2b(x: float) -> int:
    """bf16 pattern of a value known to be exactly representable."""
    b = struct.unpack("<I", struct.pack("<f", x))[0]
    assert b & 0xFFFF == 0, x
    return b >> 16


# --------------------------------------------------------------------------
# bf16 rounding and widening
# --------------------------------------------------------------------------

def test_bf16_widening_matches_torch_for_all_patterns(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = gi.from_bits(pats).to(torch.float64).numpy()
    got = np.array([oracle_lib.oracle_bf16_to_double(int(p)) for p in pats])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def _random_doubles(rng, n):
    # magnitudes across the whole bf16 range, incl. subnormal and overflow
    e = rng.integers(-140, 130, size=n)
    m = rng.random(n) + 1.0
    s = rng.choice([-1.0, 1.0], size=n)
    return s * np.ldexp(m, e)


def _ties_and_edges():
    vals = []
    for b in [0x0001, 0x0002, 0x007F, 0x0080, 0x0081, 0x3F80, 0x3F81, 0x4049, 0x7F7E, 0x7F7F, 0x00FF]:
        lo = bf16_bits_to_fraction(b)
        hi = bf16_bits_to_fraction(b + 1) if b + 1 < 0x7F80 else Fraction(2) ** 128
        mid = (lo + hi) / 2
        for q in (mid, mid + (hi - lo) / 1024, mid - (hi - lo) / 1024, lo, (lo + mid) / 2):
            f = float(q)
            if Fraction(f) == q:   # exactly representable in binary64
                vals.extend([f, -f])
    vals += [2.0 ** -134, 2.0 ** -133, 3 * 2.0 ** -134, 2.0 ** -150, 1e-300, 5e-324,
             3.4028234663852886e38, 3.3961775292304416e38, 3.3961775292304417e38, 1e39, 1e308]
    return vals


def test_bf16_round_equals_bruteforce_nearest_even(oracle_lib):
    """Random doubles + constructed ties: oracle == exhaustive-table RNE."""
    rng = np.random.default_rng(1234)
    vals = list(_random_doubles(rng, 4000)) + _ties_and_edges()
    for v in vals:
        got = oracle_lib.oracle_bf16_round(float(v))
        want = rne_bf16(Fraction(float(v)))
        if want == 0 and v < 0:
            want = 0x8000   # a negative value that rounds to zero keeps its sign
        assert got == want, (v, hex(got), hex(want))


def test_bf16_round_matches_torch_on_float32_values(oracle_lib):
    """For binary32 inputs a single rounding equals torch's float32->bf16."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(20000, generator=g) * (10.0 ** torch.randint(-30, 30, (20000,), generator=g).float())
    x = torch.cat([x, torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -130, 3e38])])
    want = gi.bits(x.to(torch.bfloat16))
    got = np.array([oracle_lib.oracle_bf16_round(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_round_specials(oracle_lib):
    assert oracle_lib.oracle_bf16_round(float("inf")) == 0x7F80
    assert oracle_lib.oracle_bf16_round(float("-inf")) == 0xFF80
    assert oracle_lib.oracle_bf16_round(float("nan")) & 0x7FFF > 0x7F80
    assert oracle_lib.oracle_bf16_round(-0.0) == 0x8000
    assert oracle_lib.oracle_bf16_round(0.0) == 0x0000
    assert oracle_lib.oracle_bf16_round(1.0) == 0x3F80
    # 1 + 2^-8 is the tie between 1 and 1 + 2^-7: goes to the even pattern (1)
    assert oracle_lib.oracle_bf16_round(1.0 + 2 ** -8) == 0x3F80
    assert oracle_lib.oracle_bf16_round(1.0 + 3 * 2 ** -8) == 0x3F82


# --------------------------------------------------------------------------
# SiLU
# --------------------------------------------------------------------------

def _all_finite_bf16():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return pats[(pats & 0x7FFF) < 0x7F80]


@pytest.mark.slow
def test_silu_exhaustive_over_bf16_gate_values(oracle_lib):
    """K=1, h=[1], W_gate[:,0] = every finite bf16, W_up = 1:
    out = bf16(SiLU(g)) for every g, against 120-bit SiLU rounded by brute
    force.  Same in HF mode (g and u=1 are already bf16)."""
    g = _all_finite_bf16()
    N = g.size
    h = np.array([[f2b(1.0)]], dtype=np.uint16)
    gw = g.reshape(N, 1)
    uw = np.full((N, 1), f2b(1.0), dtype=np.uint16)
    out_f = oracle.glu_gemv(h, gw, uw, "fused", lib=oracle_lib)
    out_h = oracle.glu_gemv(h, gw, uw, "hf", lib=oracle_lib)
    want = np.empty(N, dtype=np.uint16)
    for i, b in enumerate(g):
        v = rne_bf16(silu_exact(bf16_bits_to_fraction(int(b))))
        if v == 0 and (int(b) & 0x8000):
            v = 0x8000   # SiLU of a negative value that rounds to zero: -0
        want[i] = v
    # +0 and -0 are one point (G = 0 + (-0) sums to +0)
    for out in (out_f[0], out_h[0]):
        assert np.array_equal(tol.ordered(out), tol.ordered(want)), np.flatnonzero(out != want)[:10]
        nz = (want & 0x7FFF) != 0
        assert np.array_equal(out[nz], want[nz])


def test_silu_closed_forms(oracle_lib):
    assert oracle_lib.oracle_silu(0.0) == 0.0
    for x in (-5.0, -1.0, -0.25, 0.5, 1.0, 3.0, 20.0):
        want = float(silu_exact(Fraction(x)))
        assert abs(oracle_lib.oracle_silu(x) - want) <= 4 * abs(want) * 2 ** -53
    # SiLU(x) - SiLU(-x) = x
    for x in (0.3, 1.7, 6.0):
        assert abs(oracle_lib.oracle_silu(x) - oracle_lib.oracle_silu(-x) - x) < 1e-15 * max(1, x)


# --------------------------------------------------------------------------
# Dot products and epilogues against exact arithmetic
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["fused", "hf"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 3, 4), (2, 3, 4), (3, 2, 5), (2, 5, 8)])
def test_glu_exact_small_integers(oracle_lib, mode, shape):
    """Small-integer operands: G and U are exact integers; the output is the
    brute-force rounding of the 120-bit SiLU(G)*U (or the HF chain)."""
    M, N, K = shape
    h = gi.small_int_bf16((M, K), seed=11 + M)
    gw = gi.small_int_bf16((N, K), seed=23 + N)
    uw = gi.small_int_bf16((N, K), seed=37 + K, lo=-3, hi=3)
    out, diag = oracle.glu_gemv(h, gw, uw, mode, diagnostics=True, lib=oracle_lib)
    want, Gx, Ux = glu_exact(h, gw, uw, mode)
    nz = (want & 0x7FFF) != 0
    assert np.array_equal(out[nz], want[nz])
    assert np.all((out[~nz] & 0x7FFF) == 0)
    for m in range(M):
        for n in range(N):
            assert Fraction(diag["G"][m, n]) == Gx[m][n]
            assert Fraction(diag["U"][m, n]) == Ux[m][n]


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_glu_exact_random_normal(oracle_lib, mode):
    """N(0,1) bf16 operands, K<=8: the binary64 sums are still exact."""
    for seed, (M, N, K) in enumerate([(1, 6, 7), (2, 4, 8), (3, 5, 3)]):
        h = gi.bits(gi.normal_bf16((M, K), 1.0, seed, "pin-h"))
        gw = gi.bits(gi.normal_bf16((N, K), 0.5, seed, "pin-g"))
        uw = gi.bits(gi.normal_bf16((N, K), 0.5, seed, "pin-u"))
        out, diag = oracle.glu_gemv(h, gw, uw, mode, diagnostics=True, lib=oracle_lib)
        want, Gx, Ux = glu_exact(h, gw, uw, mode)
        assert np.array_equal(out, want)
        assert all(Fraction(diag["G"][m, n]) == Gx[m][n] for m in range(M) for n in range(N))
        assert all(Fraction(diag["U"][m, n]) == Ux[m][n] for m in range(M) for n in range(N))


def test_glu_abs_sums(oracle_lib):
    h = gi.small_int_bf16((2, 6), seed=3)
    gw = gi.small_int_bf16((3, 6), seed=4)
    uw = gi.small_int_bf16((3, 6), seed=5)
    _, d = oracle.glu_gemv(h, gw, uw, "fused", diagnostics=True, lib=oracle_lib)
    hf = tol.bf16_bits_to_f64(h)
    assert np.array_equal(d["Ag"], np.abs(hf) @ np.abs(tol.bf16_bits_to_f64(gw)).T)
    assert np.array_equal(d["Au"], np.abs(hf) @ np.abs(tol.bf16_bits_to_f64(uw)).T)


# --------------------------------------------------------------------------
# Closed forms and invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_zero_weights_give_positive_zero(oracle_lib, mode):
    h = gi.bits(gi.normal_bf16((3, 64), 1.0, 0, "z-h"))
    z = np.zeros((17, 64), dtype=np.uint16)
    out = oracle.glu_gemv(h, z, z, mode, lib=oracle_lib)
    assert np.all(out == 0)


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_zero_hidden_gives_zero(oracle_lib, mode):
    h = np.zeros((2, 48), dtype=np.uint16)
    w = gi.bits(gi.normal_bf16((9, 48), 1.0, 0, "zh-w"))
    out = oracle.glu_gemv(h, w, w, mode, lib=oracle_lib)
    assert np.all((out & 0x7FFF) == 0)


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_identity_rows(oracle_lib, mode):
    """N = K, W_gate = W_up = I: out_i = SiLU(h_i) * h_i (fused: one rounding;
    HF: bf16(bf16(SiLU(h_i)) * h_i))."""
    K = 40
    hb = gi.bits(gi.normal_bf16((2, K), 2.0, 5, "id-h"))
    eye = gi.bits(torch.eye(K, dtype=torch.bfloat16))
    out = oracle.glu_gemv(hb, eye, eye, mode, lib=oracle_lib)
    for m in range(2):
        for i in range(K):
            hi = bf16_bits_to_fraction(int(hb[m, i]))
            if mode == "fused":
                want = rne_bf16(silu_exact(hi) * hi)
            else:
                want = rne_bf16(bf16_bits_to_fraction(rne_bf16(silu_exact(hi))) * hi)
            if hi == 0:
                assert out[m, i] & 0x7FFF == 0
            else:
                assert out[m, i] == want, (m, i)


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_swapping_gate_and_up_moves_only_the_silu(oracle_lib, mode):
    """glu(h, W_up, W_gate) = bf16(SiLU(U) * G): the roles of the two dot
    products swap and nothing else changes."""
    M, N, K = 2, 33, 96
    h = gi.bits(gi.normal_bf16((M, K), 1.0, 2, "sw-h"))
    gw = gi.bits(gi.normal_bf16((N, K), 0.1, 2, "sw-g"))
    uw = gi.bits(gi.normal_bf16((N, K), 0.1, 2, "sw-u"))
    _, d = oracle.glu_gemv(h, gw, uw, mode, diagnostics=True, lib=oracle_lib)
    out_sw, d_sw = oracle.glu_gemv(h, uw, gw, mode, diagnostics=True, lib=oracle_lib)
    assert np.array_equal(d_sw["G"], d["U"]) and np.array_equal(d_sw["U"], d["G"])
    for m in range(M):
        for n in range(N):
            G, U = Fraction(d["G"][m, n]), Fraction(d["U"][m, n])
            if mode == "fused":
                want = rne_bf16(silu_exact(U) * G)
            else:
                ub = bf16_bits_to_fraction(rne_bf16(U))
                gb = bf16_bits_to_fraction(rne_bf16(G))
                want = rne_bf16(bf16_bits_to_fraction(rne_bf16(silu_exact(ub))) * gb)
            assert out_sw[m, n] == want


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_power_of_two_scaling_of_up(oracle_lib, mode):
    """W_up -> 2*W_up doubles every output exactly (scaling by 2 commutes with
    round-to-nearest-even away from overflow and subnormals)."""
    M, N, K = 2, 50, 128
    h = gi.bits(gi.normal_bf16((M, K), 1.0, 3, "p2-h"))
    gw = gi.bits(gi.normal_bf16((N, K), 0.1, 3, "p2-g"))
    u = gi.normal_bf16((N, K), 0.1, 3, "p2-u")
    o1 = oracle.glu_gemv(h, gw, gi.bits(u), mode, lib=oracle_lib)
    o2 = oracle.glu_gemv(h, gw, gi.bits(u * 2), mode, lib=oracle_lib)
    v1, v2 = tol.bf16_bits_to_f64(o1), tol.bf16_bits_to_f64(o2)
    ok = np.abs(v1) > 2.0 ** -120
    assert ok.mean() > 0.9
    assert np.array_equal(v2[ok], 2 * v1[ok])


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_row_permutation_permutes_outputs(oracle_lib, mode):
    M, N, K = 3, 41, 72
    h = gi.bits(gi.normal_bf16((M, K), 1.0, 4, "pm-h"))
    gw = gi.bits(gi.normal_bf16((N, K), 0.1, 4, "pm-g"))
    uw = gi.bits(gi.normal_bf16((N, K), 0.1, 4, "pm-u"))
    perm = np.random.default_rng(0).permutation(N)
    o = oracle.glu_gemv(h, gw, uw, mode, lib=oracle_lib)
    op = oracle.glu_gemv(h, gw[perm], uw[perm], mode, lib=oracle_lib)
    assert np.array_equal(op, o[:, perm])


def test_thread_count_does_not_change_results(oracle_lib):
    M, N, K = 2, 257, 300
    h = gi.bits(gi.normal_bf16((M, K), 1.0, 6, "th-h"))
    gw = gi.bits(gi.normal_bf16((N, K), 0.06, 6, "th-g"))
    uw = gi.bits(gi.normal_bf16((N, K), 0.06, 6, "th-u"))
    a = oracle.glu_gemv(h, gw, uw, "hf", nthreads=1, lib=oracle_lib)
    b = oracle.glu_gemv(h, gw, uw, "hf", nthreads=7, lib=oracle_lib)
    assert np.array_equal(a, b)


def test_empty_shapes(oracle_lib):
    h = np.zeros((0, 8), dtype=np.uint16)
    w = np.zeros((4, 8), dtype=np.uint16)
    assert oracle.glu_gemv(h, w, w, lib=oracle_lib).shape == (0, 4)
    # K == 0: empty sums, SiLU(0) * 0 = +0
    h0 = np.zeros((2, 0), dtype=np.uint16)
    w0 = np.zeros((3, 0), dtype=np.uint16)
    assert np.all(oracle.glu_gemv(h0, w0, w0, "hf", lib=oracle_lib) == 0)
    assert np.all(oracle.glu_gemv(h0, w0, w0, "fused", lib=oracle_lib) == 0)


# --------------------------------------------------------------------------
# Library composite cross-checks
# --------------------------------------------------------------------------

def test_fused_matches_float64_torch_composite(oracle_lib):
    """F.silu(h@Wg.T) * (h@Wu.T) in float64 (a BLAS sum, another order), then
    one brute-force rounding: equal away from near-ties."""
    M, N, K = 2, 64, 256
    h = gi.normal_bf16((M, K), 1.0, 8, "c64-h")
    gw = gi.normal_bf16((N, K), 0.0625, 8, "c64-g")
    uw = gi.normal_bf16((N, K), 0.0625, 8, "c64-u")
    out = oracle.glu_gemv(gi.bits(h), gi.bits(gw), gi.bits(uw), "fused", lib=oracle_lib)
    h64, g64, u64 = (t.to(torch.float64) for t in (h, gw, uw))
    ref = (torch.nn.functional.silu(h64 @ g64.T) * (h64 @ u64.T)).numpy()
    want = np.array([[rne_bf16(Fraction(float(v))) for v in row] for row in ref], dtype=np.uint16)
    assert np.mean(out == want) >= 0.999
    assert tol.ulp_distance(out, want).max() <= 1


def test_hf_matches_bf16_torch_composite(oracle_lib):
    """The HF composite on bf16 CPU tensors (fp32 accumulation inside the
    matmul, bf16 tensors between ops) agrees within the parity bar."""
    M, N, K = 4, 512, 1024
    h = gi.normal_bf16((M, K), 1.0, 9, "cbf-h")
    gw = gi.normal_bf16((N, K), 1 / 32, 9, "cbf-g")
    uw = gi.normal_bf16((N, K), 1 / 32, 9, "cbf-u")
    out, diag = oracle.glu_gemv(gi.bits(h), gi.bits(gw), gi.bits(uw), "hf", diagnostics=True, lib=oracle_lib)
    ref = torch.nn.functional.silu(h @ gw.T) * (h @ uw.T)
    tau = tol.conditioning_floor(diag, K, "hf")
    st = tol.compare(gi.bits(ref), out, tau)
    assert tol.passes(st), st
    assert st["exact_frac"] > 0.95


# --------------------------------------------------------------------------
# Residual add + zero-centred RMSNorm
# --------------------------------------------------------------------------

def test_norm_against_high_precision(oracle_lib):
    M, K = 3, 96
    x = gi.bits(gi.normal_bf16((M, K), 1.0, 10, "n-x"))
    r = gi.bits(gi.normal_bf16((M, K), 1.0, 10, "n-r"))
    w = gi.bits(gi.normal_bf16((K,), 0.1, 10, "n-w"))
    s, h = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
    for m in range(M):
        ws, wh = rmsnorm_exact_row(x[m], r[m], w, EPS32)
        assert list(s[m]) == ws
        assert list(h[m]) == wh


def test_norm_small_rows_eps_matters(oracle_lib):
    """Rows with mean(s^2) near eps: the eps term is visible in h."""
    M, K = 2, 32
    x = gi.bits(gi.normal_bf16((M, K), 1e-3, 17, "ne-x"))
    r = np.zeros((M, K), dtype=np.uint16)
    w = gi.bits(gi.normal_bf16((K,), 0.1, 17, "ne-w"))
    _, h = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
    for m in range(M):
        _, wh = rmsnorm_exact_row(x[m], r[m], w, EPS32)
        assert list(h[m]) == wh
    _, h_noeps = oracle.add_rmsnorm(x, r, w, 0.0, lib=oracle_lib)
    assert not np.array_equal(h, h_noeps)


def test_norm_zero_weight_is_plain_rmsnorm(oracle_lib):
    """norm_w = 0 gives (1 + 0) = 1: h = bf16(s / sqrt(mean(s^2) + eps))."""
    K = 64
    x = gi.bits(gi.normal_bf16((1, K), 1.0, 12, "nz-x"))
    r = np.zeros((1, K), dtype=np.uint16)
    w = np.zeros((K,), dtype=np.uint16)
    s, h = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
    assert np.array_equal(s, x)
    xv = tol.bf16_bits_to_f64(x[0])
    ref = xv / np.sqrt(np.mean(xv * xv) + EPS32)
    want = np.array([rne_bf16(Fraction(float(v))) for v in ref], dtype=np.uint16)
    assert tol.ulp_distance(h[0], want).max() == 0


def test_norm_constant_row(oracle_lib):
    """s = c everywhere: h = bf16(c / sqrt(c^2 + eps))."""
    K = 128
    for c in (0.5, -3.0, 1e-3):
        cb = oracle_lib.oracle_bf16_round(c)
        x = np.full((1, K), cb, dtype=np.uint16)
        r = np.zeros((1, K), dtype=np.uint16)
        w = np.zeros((K,), dtype=np.uint16)
        _, h = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
        cv = bf16_bits_to_fraction(cb)
        val = fraction_to_mpf(cv) / mpmath.sqrt(fraction_to_mpf(cv * cv + Fraction(EPS32)))
        assert np.all(h == rne_bf16(mpf_to_fraction(val)))


def test_norm_cancelled_residual_gives_zero(oracle_lib):
    """x = -residual: s = +0 everywhere, var = 0, h = 0 / sqrt(eps) = 0."""
    K = 80
    x = gi.bits(gi.normal_bf16((2, K), 1.0, 13, "nc-x"))
    r = x ^ np.uint16(0x8000)
    w = gi.bits(gi.normal_bf16((K,), 0.1, 13, "nc-w"))
    s, h = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
    assert np.all(s == 0) and np.all(h == 0)


def test_residual_sum_is_one_correct_rounding(oracle_lib):
    M, K = 4, 200
    x = gi.bits(gi.normal_bf16((M, K), 1.0, 14, "rs-x"))
    r = gi.bits(gi.normal_bf16((M, K), 3.0, 14, "rs-r"))
    w = np.zeros((K,), dtype=np.uint16)
    s, _ = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
    want = np.array([[rne_bf16(bf16_bits_to_fraction(int(a)) + bf16_bits_to_fraction(int(b)))
                      for a, b in zip(xr, rr)] for xr, rr in zip(x, r)], dtype=np.uint16)
    nz = (want & 0x7FFF) != 0
    assert np.array_equal(s[nz], want[nz])
    assert np.all((s[~nz] & 0x7FFF) == 0)


def test_norm_matches_fp32_torch_formula(oracle_lib):
    """HF's zero-centred RMSNorm in fp32 torch (x.float(); rsqrt(mean+eps);
    *(1+w.float()); to bf16): within one bf16 step, nearly always equal."""
    M, K = 8, 2560
    x = gi.normal_bf16((M, K), 1.0, 15, "nt-x")
    r = gi.normal_bf16((M, K), 1.0, 15, "nt-r")
    w = gi.normal_bf16((K,), 0.1, 15, "nt-w")
    s, h = oracle.add_rmsnorm(gi.bits(x), gi.bits(r), gi.bits(w), 1e-6, lib=oracle_lib)
    st = (x + r)  # bf16 add on CPU: one rounding
    assert np.array_equal(gi.bits(st), s)
    sf = st.float()
    ref = (sf * torch.rsqrt(sf.pow(2).mean(-1, keepdim=True) + 1e-6)) * (1.0 + w.float())
    d = tol.ulp_distance(gi.bits(ref.to(torch.bfloat16)), h)
    assert d.max() <= 1 and np.mean(d == 0) > 0.99


def test_fused_segment_is_norm_then_glu(oracle_lib):
    M, N, K = 2, 40, 64
    x = gi.bits(gi.normal_bf16((M, K), 1.0, 16, "fs-x"))
    r = gi.bits(gi.normal_bf16((M, K), 1.0, 16, "fs-r"))
    w = gi.bits(gi.normal_bf16((K,), 0.1, 16, "fs-w"))
    gw = gi.bits(gi.normal_bf16((N, K), 0.125, 16, "fs-g"))
    uw = gi.bits(gi.normal_bf16((N, K), 0.125, 16, "fs-u"))
    out, res, h = oracle.add_rmsnorm_glu(x, r, w, 1e-6, gw, uw, "hf", lib=oracle_lib)
    s2, h2 = oracle.add_rmsnorm(x, r, w, 1e-6, lib=oracle_lib)
    assert np.array_equal(res, s2) and np.array_equal(h, h2)
    want, _, _ = glu_exact(h2, gw, uw, "hf")
    assert np.array_equal(out, want)


# ---------------------------------------------------------------------------
# silu_mul (halves layout): the standalone epilogue
# ---------------------------------------------------------------------------

def _silu_mul_exact(g_bits, u_bits, mode):
    """Exactly rounded silu_mul from arbitrary-precision SiLU (exact_ref)."""
    out = np.zeros(len(g_bits), dtype=np.uint16)
    for i, (gb, ub) in enumerate(zip(g_bits, u_bits)):
        g, u = bf16_bits_to_fraction(int(gb)), bf16_bits_to_fraction(int(ub))
        if mode == "fused":
            out[i] = rne_bf16(silu_exact(g) * u)
        else:
            sb = bf16_bits_to_fraction(rne_bf16(silu_exact(g)))
            out[i] = rne_bf16(sb * u)
    return out


def _same_up_to_zero_sign(a, b):
    a, b = np.asarray(a), np.asarray(b)
    zero = ((a & 0x7FFF) == 0) & ((b & 0x7FFF) == 0)
    return bool(np.all((a == b) | zero))


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_silu_mul_matches_exact_rounding(mode):
    """Every output is the correctly rounded value of the exact SiLU(g) * u
    (FUSED) or of bf16(SiLU(g)) * u (HF), over N(0, 2) draws, SiLU's far
    negative tail and small integers."""
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(11)
    g = np.concatenate([gi.bits(gi.normal_bf16((200,), 2.0, 0, "smx-g")),
                        gi.bits(torch.tensor(-rng.uniform(20, 95, 40), dtype=torch.float32).to(torch.bfloat16)),
                        gi.small_int_bf16((20,), seed=3, lo=-4, hi=4)])
    u = np.concatenate([gi.bits(gi.normal_bf16((200,), 2.0, 0, "smx-u")),
                        gi.bits(gi.normal_bf16((40,), 1.0, 0, "smx-u2")),
                        gi.small_int_bf16((20,), seed=4, lo=-4, hi=4)])
    x = np.concatenate([g, u])[None, :]
    got = oracle.silu_mul(x, mode)[0]
    assert _same_up_to_zero_sign(got, _silu_mul_exact(g, u, mode))


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_silu_mul_equals_glu_gemv_with_k_one(mode):
    """With K = 1 and h = 1 the GEMV's dot products are exactly the weights,
    so glu_gemv (pinned on its own above) must give silu_mul's bits."""
    N = 300
    g = gi.bits(gi.normal_bf16((N,), 3.0, 0, "smk-g"))
    u = gi.bits(gi.normal_bf16((N,), 1.0, 0, "smk-u"))
    h = np.array([[0x3F80]], dtype=np.uint16)   # 1.0
    want = oracle.glu_gemv(h, g[:, None].copy(), u[:, None].copy(), mode)[0]
    got = oracle.silu_mul(np.concatenate([g, u])[None, :], mode)[0]
    assert np.array_equal(got, want)


def test_silu_mul_halves_orientation_strides_and_closed_forms():
    one, m20, zero = 0x3F80, gi.bits(torch.tensor([-20.0]).to(torch.bfloat16))[0], 0x0000
    # gate half first: SiLU(-20) * 1 is tiny; SiLU(1) * -20 is not
    a = oracle.silu_mul(np.array([[m20, one]], dtype=np.uint16), "fused")[0, 0]
    b = oracle.silu_mul(np.array([[one, m20]], dtype=np.uint16), "fused")[0, 0]
    assert abs(oracle.bf16_to_float(int(a))) < 1e-7
    assert abs(oracle.bf16_to_float(int(b)) - (-20.0 / (1.0 + math.exp(-1.0)))) < 0.06
    # u = 0 -> zero; g = 0 -> zero; g = 100 -> SiLU(g) = g (to binary64) so out = bf16(g * u)
    x = np.array([[one, zero, 0x42C8, one, 0x4000, 0x4000]], dtype=np.uint16)   # g = 1, 0, 100; u = 1, 2, 2
    out = oracle.silu_mul(x, "hf")[0]
    assert oracle.bf16_to_float(int(out[1])) == 0.0
    assert oracle.bf16_to_float(int(out[2])) == 200.0
    # a row stride wider than 2N is honoured; the padding is never read
    M, N = 3, 5
    wide = np.full((M, 2 * N + 3), 0x7FC0, dtype=np.uint16)   # NaN padding
    body = gi.bits(gi.normal_bf16((M, 2 * N), 1.0, 0, "sms"))
    wide[:, :2 * N] = body
    assert np.array_equal(oracle.silu_mul(wide[:, :2 * N], "fused"), oracle.silu_mul(body, "fused"))


# ---------------------------------------------------------------------------
# gdn_gates: beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias)
# ---------------------------------------------------------------------------

def _gdn_inputs(T=7, H=24, seed=0):
    rng = np.random.default_rng(seed)
    a = gi.bits(torch.tensor(rng.normal(0, 3, (T, H)), dtype=torch.float32).to(torch.bfloat16))
    b = gi.bits(torch.tensor(rng.normal(0, 3, (T, H)), dtype=torch.float32).to(torch.bfloat16))
    A_log = rng.normal(0, 1, H).astype(np.float32)
    dt_bias = rng.normal(0, 1, H).astype(np.float32)
    return a, b, A_log, dt_bias


def test_gdn_gates_match_arbitrary_precision():
    """g against mpmath at 120 bits on x = fp32(a + dt_bias) (numpy's IEEE
    float32 addition), beta against exact rounding of the exact sigmoid."""
    mpmath = pytest.importorskip("mpmath")
    a, b, A_log, dt_bias = _gdn_inputs()
    g, beta = oracle.gdn_gates(a, b, A_log, dt_bias)
    af = (a.astype(np.uint32) << 16).view(np.float32)
    bf = (b.astype(np.uint32) << 16).view(np.float32)
    x = (af + dt_bias[None, :]).astype(np.float32)          # binary32 addition
    with mpmath.workprec(120):
        for t in range(a.shape[0]):
            for j in range(a.shape[1]):
                xe = mpmath.mpf(float(x[t, j]))
                ge = -mpmath.exp(mpmath.mpf(float(A_log[j]))) * mpmath.log(1 + mpmath.exp(xe))
                assert abs(g[t, j] - float(ge)) <= 1e-15 * abs(float(ge))
                ye = mpmath.mpf(float(bf[t, j]))
                se = 1 / (1 + mpmath.exp(-ye))
                assert beta[t, j] == rne_bf16(mpf_to_fraction(se)), (t, j)


def test_gdn_gates_closed_forms_and_tails():
    bits = lambda v: gi.bits(torch.tensor(v, dtype=torch.float32).to(torch.bfloat16))   # noqa: E731
    a = bits([[0.0, 1000.0, -80.0, 40.0]])
    b = bits([[0.0, 3.0, -3.0, 100.0]])
    A_log = np.array([0.0, 0.0, 1.0, np.log(2.0)], dtype=np.float32)
    dt = np.zeros(4, dtype=np.float32)
    g, beta = oracle.gdn_gates(a, b, A_log, dt)
    assert abs(g[0, 0] + math.log(2.0)) < 1e-15                                 # softplus(0) = ln 2
    assert abs(g[0, 1] + 1000.0) < 1e-12                                        # softplus(x) -> x, no overflow
    assert abs(g[0, 2] / (-math.e * math.exp(-80.0)) - 1) < 1e-12              # softplus(x) -> e^x
    assert abs(g[0, 3] / (-float(np.exp(np.float32(np.log(2.0)), dtype=np.float64)) * 40.0) - 1) < 1e-15
    assert beta[0, 0] == 0x3F00                                                 # sigmoid(0) = 1/2
    s3 = oracle.bf16_to_float(int(beta[0, 1])) + oracle.bf16_to_float(int(beta[0, 2]))
    assert abs(s3 - 1.0) <= 2 ** -8                                              # sigmoid(-y) = 1 - sigmoid(y)
    assert beta[0, 3] == 0x3F80                                                 # rounds to 1


# ---------------------------------------------------------------------------
# backward of the dual-weight GLU GEMV
# ---------------------------------------------------------------------------

def _bwd_inputs(M=3, N=20, K=24, seed=0):
    h = gi.bits(gi.normal_bf16((M, K), 1.0, seed, "bw-h"))
    gw = gi.bits(gi.normal_bf16((N, K), 0.3, seed, "bw-g"))
    uw = gi.bits(gi.normal_bf16((N, K), 0.3, seed, "bw-u"))
    d = gi.bits(gi.normal_bf16((M, N), 1.0, seed, "bw-d"))
    return h, gw, uw, d


def _f64(bits_):
    return torch.from_numpy((np.asarray(bits_, np.uint32) << 16).view(np.float32).astype(np.float64))


def test_glu_backward_matches_fp64_autograd():
    """The three gradients against PyTorch autograd of the fp64 composite
    F.silu(h @ Wg.T) * (h @ Wu.T) on the same (exact) inputs."""
    h, gw, uw, d = _bwd_inputs()
    gh, gg, gu = oracle.glu_backward(h, gw, uw, d)
    ht, gt, ut = (_f64(a).requires_grad_(True) for a in (h, gw, uw))
    out = torch.nn.functional.silu(ht @ gt.T) * (ht @ ut.T)
    rh, rg, ru = torch.autograd.grad(out, (ht, gt, ut), grad_outputs=_f64(d))
    for got, ref in ((gh, rh), (gg, rg), (gu, ru)):
        ref = ref.numpy()
        assert np.abs(got - ref).max() <= 1e-12 * np.abs(ref).max()


def test_glu_backward_finite_differences():
    """Central differences of sum(dout * out) in binary64 along a few
    coordinates of h, Wg and Wu."""
    h, gw, uw, d = _bwd_inputs(M=2, N=6, K=5, seed=1)
    gh, gg, gu = oracle.glu_backward(h, gw, uw, d)
    H, G, U, D = (_f64(a).numpy() for a in (h, gw, uw, d))

    def f(H_, G_, U_):
        g = H_ @ G_.T
        return float(np.sum(D * (g / (1 + np.exp(-g))) * (H_ @ U_.T)))

    eps = 1e-6
    for arr, grad, idx in ((H, gh, (1, 3)), (G, gg, (4, 2)), (U, gu, (0, 0)), (U, gu, (5, 4))):
        p, m = arr.copy(), arr.copy()
        p[idx] += eps
        m[idx] -= eps
        args_p = [p if arr is x else x for x in (H, G, U)]
        args_m = [m if arr is x else x for x in (H, G, U)]
        fd = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def test_glu_backward_closed_forms_and_threads():
    h, gw, uw, d = _bwd_inputs(seed=2)
    gh, gg, gu = oracle.glu_backward(h, gw, uw, np.zeros_like(d))
    assert not gh.any() and not gg.any() and not gu.any()             # no upstream gradient
    gh, gg, gu = oracle.glu_backward(h, gw, np.zeros_like(uw), d)      # up_w = 0: U = 0
    assert not gh.any() and not gg.any() and gu.any()                  # only dWu = (dout*SiLU(G))^T h
    a = oracle.glu_backward(h, gw, uw, d, nthreads=1)
    b = oracle.glu_backward(h, gw, uw, d, nthreads=7)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
