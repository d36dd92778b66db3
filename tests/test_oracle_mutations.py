"""Planted mistakes in a copy of the oracle must be caught by its pins.

Each case copies ``oracle/mbglu_oracle.c`` to a temporary directory, applies
one textual slip of the kind a hand-written oracle might carry (a wrong sign,
a dropped term, a transposed operand, a wrong tie rule, a wrong index, a
missing epsilon), builds it with the oracle's own flags, and runs a compact
set of the pins from ``test_oracle_pins.py`` against it.  The unmodified
source must pass the same set.  Everything runs on the CPU.
"""
import math
import os
import shutil
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import glu_inputs as gi
from exact_ref import bf16_bits_to_fraction, glu_exact, rmsnorm_exact_row, rne_bf16, silu_exact

pytest.importorskip("mpmath")
EPS32 = float(np.float32(1e-6))

MUTATIONS = {
    "silu_sign": ("x / (1.0 + exp(-x))", "x / (1.0 + exp(x))"),
    "dropped_first_term": ("for (int k = 0; k < j->K; ++k) {\n                const double hk = oracle_bf16_to_double(hrow[k]);\n                const double pg",
                           "for (int k = 1; k < j->K; ++k) {\n                const double hk = oracle_bf16_to_double(hrow[k]);\n                const double pg"),
    "up_reads_gate": ("const double pu = hk * oracle_bf16_to_double(urow[k]);",
                      "const double pu = hk * oracle_bf16_to_double(grow[k]);"),
    "hf_up_rounds_gate": ("const uint16_t ub = oracle_bf16_round(U);", "const uint16_t ub = oracle_bf16_round(G);"),
    "hf_silu_on_unrounded_gate": ("oracle_silu(oracle_bf16_to_double(gb))", "oracle_silu(G)"),
    "fused_rounds_twice": ("o = oracle_bf16_round(oracle_silu(G) * U);",
                           "o = oracle_bf16_round(oracle_bf16_to_double(oracle_bf16_round(oracle_silu(G))) * U);"),
    "ties_away": ("(rem == half && (n & 1))", "(rem == half)"),
    "no_subnormals": ("(e >= -126) ? (e - 7) : -133", "(e - 7)"),
    "batch_row_index": ("hrow = j->h + (int64_t)m * j->ldh;\n        for (int n = j->n0;",
                        "hrow = j->h;\n        for (int n = j->n0;"),
    "norm_mean_divisor": ("ss / (double)K", "ss / (double)(K + 1)"),
    "norm_scale_not_centred": ("1.0 + oracle_bf16_to_double(norm_w[k])", "oracle_bf16_to_double(norm_w[k])"),
    "norm_eps_dropped": ("sqrt(var + e)", "sqrt(var)"),
    "residual_sign": ("oracle_bf16_to_double(xr[k]) +", "oracle_bf16_to_double(xr[k]) -"),
    "silu_mul_halves_swapped": ("const double g = oracle_bf16_to_double(gate[n]);",
                                "const double g = oracle_bf16_to_double(up[n]);"),
    "silu_mul_hf_unrounded_silu": ("o = oracle_bf16_round(oracle_bf16_to_double(sb) * u);",
                                   "o = oracle_bf16_round(oracle_silu(g) * u);"),
    "gdn_softplus_unstable": ("return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));", "return log1p(exp(x));"),
    "gdn_sigmoid_sign": ("oracle_bf16_round(1.0 / (1.0 + exp(-y)))", "oracle_bf16_round(1.0 / (1.0 + exp(y)))"),
    "bwd_dsilu_missing_term": ("d * U * (s * (1.0 + G * (1.0 - s)))", "d * U * s"),
    "bwd_up_grad_from_dG": ("su += j->dU[(int64_t)m * j->N + n] * hk;", "su += j->dG[(int64_t)m * j->N + n] * hk;"),
    "hf_product_on_unrounded_up": ("o = oracle_bf16_round(oracle_bf16_to_double(sb) * oracle_bf16_to_double(ub));",
                                   "o = oracle_bf16_round(oracle_bf16_to_double(sb) * U);"),
    "norm_stat_on_unrounded_sum": ("            const double sv = oracle_bf16_to_double(sr[k]);\n            ss += sv * sv;",
                                   "            const double sv = oracle_bf16_to_double(xr[k]) + oracle_bf16_to_double(rr[k]);\n"
                                   "            ss += sv * sv;"),
    "bwd_dU_uses_dsilu": ("j->dU[(int64_t)m * j->N + n] = d * oracle_silu(G);",
                          "j->dU[(int64_t)m * j->N + n] = d * (s * (1.0 + G * (1.0 - s)));"),
    "bwd_grad_w_first_row_only": ("const double hk = oracle_bf16_to_double(j->h[(int64_t)m * j->ldh + k]);",
                                  "const double hk = oracle_bf16_to_double(j->h[(int64_t)0 * j->ldh + k]);"),
    "bwd_grad_h_drops_up_term": ("                acc += j->dU[(int64_t)m * j->N + n] * "
                                 "oracle_bf16_to_double(j->up_w[(int64_t)n * j->ld_up + k]);\n", ""),
    "bwd_grad_h_gate_reads_up": ("acc += j->dG[(int64_t)m * j->N + n] * oracle_bf16_to_double(j->gate_w[(int64_t)n * j->ld_gate + k]);",
                                 "acc += j->dG[(int64_t)m * j->N + n] * oracle_bf16_to_double(j->up_w[(int64_t)n * j->ld_up + k]);"),
    "gdn_decay_sign": ("g[(int64_t)t * H + j] = -exp((double)A_log[j])", "g[(int64_t)t * H + j] = exp((double)A_log[j])"),
    "gdn_x_not_binary32": ("const float x = (float)oracle_bf16_to_double(a[(int64_t)t * lda + j]) + dt_bias[j];",
                           "const double x = oracle_bf16_to_double(a[(int64_t)t * lda + j]) + (double)dt_bias[j];"),
}


def quick_pins(lib) -> list:
    """Returns the names of the pins that fail for ``lib``."""
    fails = []
    # rounding: random doubles over the whole range, plus ties
    rng = np.random.default_rng(5)
    vals = np.ldexp(rng.random(400) + 1.0, rng.integers(-140, 130, 400)) * rng.choice([-1, 1], 400)
    ties = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2.0 ** -134, 3 * 2.0 ** -134]
    for v in list(vals) + ties:
        want = rne_bf16(Fraction(float(v)))
        if want == 0 and v < 0:
            want = 0x8000
        if lib.oracle_bf16_round(float(v)) != want:
            fails.append("round")
            break
    # SiLU closed forms
    for x in (-3.0, 0.5, 2.0):
        if abs(lib.oracle_silu(x) - float(silu_exact(Fraction(x)))) > 1e-15:
            fails.append("silu")
            break
    # exact GLU on small integers and on N(0,1) draws, both modes
    for mode in ("fused", "hf"):
        for (M, N, K), kind in [((2, 5, 8), "int"), ((3, 6, 7), "normal"), ((2, 24, 8), "normal")]:
            if kind == "int":
                h = gi.small_int_bf16((M, K), seed=1 + M)
                gw = gi.small_int_bf16((N, K), seed=2 + N)
                uw = gi.small_int_bf16((N, K), seed=3 + K, lo=-3, hi=3)
            else:
                h = gi.bits(gi.normal_bf16((M, K), 1.0, 0, "mut-h", N))
                gw = gi.bits(gi.normal_bf16((N, K), 0.5, 0, "mut-g", N))
                uw = gi.bits(gi.normal_bf16((N, K), 0.5, 0, "mut-u", N))
            out = oracle.glu_gemv(h, gw, uw, mode, lib=lib)
            want, _, _ = glu_exact(h, gw, uw, mode)
            nz = (want & 0x7FFF) != 0
            if not (np.array_equal(out[nz], want[nz]) and np.all((out[~nz] & 0x7FFF) == 0)):
                fails.append(f"glu_{mode}_{kind}")
    # norm: high precision, and the cancelled residual
    x = gi.bits(gi.normal_bf16((2, 48), 1.0, 0, "mut-x"))
    r = gi.bits(gi.normal_bf16((2, 48), 1.0, 0, "mut-r"))
    w = gi.bits(gi.normal_bf16((48,), 0.1, 0, "mut-w"))
    s, hh = oracle.add_rmsnorm(x, r, w, 1e-6, lib=lib)
    for m in range(2):
        ws, wh = rmsnorm_exact_row(x[m], r[m], w, EPS32)
        if list(s[m]) != ws or list(hh[m]) != wh:
            fails.append("norm")
            break
    s0, h0 = oracle.add_rmsnorm(x, x ^ np.uint16(0x8000), w, 1e-6, lib=lib)
    if not (np.all(s0 == 0) and np.all(h0 == 0)):
        fails.append("norm_cancelled")
    # backward: against fp64 autograd of the composite
    bh = gi.bits(gi.normal_bf16((2, 12), 1.0, 0, "mut-bh"))
    bg = gi.bits(gi.normal_bf16((9, 12), 0.3, 0, "mut-bg"))
    bu = gi.bits(gi.normal_bf16((9, 12), 0.3, 0, "mut-bu"))
    bd = gi.bits(gi.normal_bf16((2, 9), 1.0, 0, "mut-bd"))
    got = oracle.glu_backward(bh, bg, bu, bd, lib=lib)
    f64 = lambda a: torch.from_numpy((a.astype(np.uint32) << 16).view(np.float32).astype(np.float64))  # noqa: E731
    ht, gt, ut = (f64(a).requires_grad_(True) for a in (bh, bg, bu))
    ref = torch.autograd.grad(torch.nn.functional.silu(ht @ gt.T) * (ht @ ut.T), (ht, gt, ut), grad_outputs=f64(bd))
    if any(np.abs(x - r.numpy()).max() > 1e-12 * np.abs(r.numpy()).max() for x, r in zip(got, ref)):
        fails.append("backward")
    # gdn_gates: g against binary64 on x = fp32(a + dt_bias), a huge x, beta exact
    rng = np.random.default_rng(8)
    ga = gi.bits(torch.tensor(np.append(rng.normal(0, 3, 31), 1000.0), dtype=torch.float32).to(torch.bfloat16))[None, :]
    gb_ = gi.bits(torch.tensor(rng.normal(0, 3, 32), dtype=torch.float32).to(torch.bfloat16))[None, :]
    A_log = rng.normal(0, 1, 32).astype(np.float32)
    dt = rng.normal(0, 1, 32).astype(np.float32)
    gg, bb = oracle.gdn_gates(ga, gb_, A_log, dt, lib=lib)
    xa = (((ga.astype(np.uint32) << 16).view(np.float32)) + dt[None, :]).astype(np.float32).astype(np.float64)
    want = -np.exp(A_log.astype(np.float64)) * np.where(xa > 0, xa + np.log1p(np.exp(-np.abs(xa))),
                                                        np.log1p(np.exp(np.minimum(xa, 0))))
    if not np.all(np.abs(gg - want) <= 1e-13 * np.abs(want)):
        fails.append("gdn_g")
    yb = (gb_.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for j in range(32):
        if bb[0, j] != rne_bf16(Fraction(1) / (1 + Fraction(math.exp(-float(yb[0, j]))))):
            # exp in binary64 is within 1 ulp; only a tie-close value could differ
            if abs(oracle.bf16_to_float(int(bb[0, j])) - 1 / (1 + math.exp(-yb[0, j]))) > 2 ** -9:
                fails.append("gdn_beta")
                break
    # silu_mul, both modes, against exact rounding (gate half first)
    g = gi.bits(gi.normal_bf16((64,), 2.0, 0, "mut-sg"))
    u = gi.bits(gi.normal_bf16((64,), 2.0, 0, "mut-su"))
    for mode in ("fused", "hf"):
        got = oracle.silu_mul(np.concatenate([g, u])[None, :], mode, lib=lib)[0]
        for i in range(64):
            gv, uv = bf16_bits_to_fraction(int(g[i])), bf16_bits_to_fraction(int(u[i]))
            sv = silu_exact(gv) if mode == "fused" else bf16_bits_to_fraction(rne_bf16(silu_exact(gv)))
            want = rne_bf16(sv * uv)
            if got[i] != want and not ((got[i] & 0x7FFF) == 0 and (want & 0x7FFF) == 0):
                fails.append(f"silu_mul_{mode}")
                break
    return fails


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mut")


def _build_variant(workdir, name, old=None, new=None):
    src = open(oracle.SRC).read()
    if old is not None:
        assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
        src = src.replace(old, new)
    d = os.path.join(str(workdir), name)
    os.makedirs(d, exist_ok=True)
    cpath = os.path.join(d, "m.c")
    with open(cpath, "w") as f:
        f.write(src)
    so = oracle.build(src=cpath, out=os.path.join(d, "libm.so"))
    return oracle.load(path=so)


def test_unmodified_oracle_passes_quick_pins(workdir):
    lib = _build_variant(workdir, "clean")
    assert quick_pins(lib) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(workdir, name):
    old, new = MUTATIONS[name]
    lib = _build_variant(workdir, name, old, new)
    assert quick_pins(lib), f"mutation {name} went unnoticed"
