"""The parity bar between the CUDA path and the oracle.

Stated bar: |delta| <= 1 bf16 ULP of the oracle on >= 99.9% of outputs, and
max relative error <= 1e-2 elsewhere.

Readings used here:
  * ULP distance: the two bf16 patterns mapped to ordered integers
    (sign-magnitude -> two's complement), with +0 and -0 the same point.
  * Relative error of an output outside 1 ULP: |gpu - ref| / max(|ref|, tau),
    where tau bounds what fp32 accumulation alone can move the output.  The
    kernels sum each dot product as 32 strided lane sums of ceil(K/32) terms
    (exact bf16 x bf16 products, one rounding per FMA) followed by a 5-level
    butterfly, so |g - G| <= gamma * Ag with gamma = (ceil(K/32) + 5) * 2^-24
    (the classical depth bound) and Ag the oracle's sum of |h*w| (likewise u):
        dg = gamma*Ag,  du = gamma*Au,
        tau = |SiLU'(G)*U|*dg + |SiLU(G)|*du  (HF mode adds 2^-8*|G| to dg
              and 2^-8*|U| to du for the bf16 roundings of g and u).
    An output with |ref| < tau sits where u or SiLU(g)*u cancels.
  * The stated bar is enforced literally: at least 99.9% of outputs lie
    within 1 ULP of the oracle's own result (STRICT_FLOOR), for every op
    and both modes.
  * "Elsewhere" (the at most 0.1% outside 1 ULP): relative error floored at
    tau must be <= 1e-2, unless the output is explained by the fp32 error
    box: it lies within 1 ULP of the range the mode's chain takes over
    g in [G - dg, G + dg], u in [U - du, U + du] (interval arithmetic over
    the monotone pieces, SiLU's minimum near g = -1.2785 included).  Such
    outputs are counted as "alt_rounding" and bounded: alt_rounding / n <=
    ALT_MAX_FRAC.  Two readings produce them:
      - HF mode rounds g and u to bf16 before SiLU: where the exact sum lies
        within dg (du) of a bf16 midpoint both neighbours are correct, and
        SiLU's log-slope (about 4 at g = -5) can turn one flip of gb into a
        few output ULPs;
      - an output so cancelled (|ref| < tau) that fp32 accumulation alone
        can move it by its own size ("ill_conditioned").
    Measured on the GPU: about 1e-4 of outputs in HF mode and 5e-5 in
    FUSED mode (outlier-weight workloads), hence the bound 5e-4.
  * Non-finite outputs must match exactly.
"""
from __future__ import annotations

import numpy as np

ULP_FRAC_REQUIRED = 0.999
MAX_REL_ELSEWHERE = 1e-2


def bf16_bits_to_f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ordered(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.uint16).astype(np.int64)
    mag = a & 0x7FFF
    return np.where(a & 0x8000, -mag, mag)


def ulp_distance(a, b) -> np.ndarray:
    return np.abs(ordered(a) - ordered(b))


def _silu(x):
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def _dsilu(x):
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-x))
    return s * (1.0 + x * (1.0 - s))


def accumulation_gamma(K: int, diag=None) -> float:
    """Relative bound of the kernels' fp32 dot products: the CUDA-core kernels
    sum at depth ceil(K/32)+5 with one rounding (2^-24) per step; the
    tensor-core kernel chains K/16 MMAs whose fp32 accumulation is not
    specified to round to nearest, bounded as depth K/16 + 16 with unit 2^-23
    (diag["acc"] == "mma")."""
    if diag is not None and diag.get("acc") == "mma":
        return (-(-K // 16) + 16) * 2.0 ** -23
    return (-(-K // 32) + 5) * 2.0 ** -24


def conditioning_floor(diag, K: int, mode: str) -> np.ndarray:
    G, U, Ag, Au = diag["G"], diag["U"], diag["Ag"], diag["Au"]
    gamma = accumulation_gamma(K, diag)
    dg, du = gamma * Ag, gamma * Au
    if mode == "hf":
        dg = dg + 2.0 ** -8 * np.abs(G)
        du = du + 2.0 ** -8 * np.abs(U)
    return np.abs(_dsilu(G) * U) * dg + np.abs(_silu(G)) * du


def _bf16_bits(x) -> np.ndarray:
    """float64 -> bf16 bits (via float32; used for candidate values only)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


SILU_ARGMIN = -1.2784645427610738


def _silu_range(lo, hi):
    """[min, max] of SiLU over [lo, hi] (decreasing, then increasing)."""
    a, b = _silu(lo), _silu(hi)
    inside = (lo <= SILU_ARGMIN) & (SILU_ARGMIN <= hi)
    mn = np.where(inside, _silu(np.full_like(lo, SILU_ARGMIN)), np.minimum(a, b))
    return mn, np.maximum(a, b)


def _product_range(alo, ahi, blo, bhi):
    c = np.stack([alo * blo, alo * bhi, ahi * blo, ahi * bhi])
    return c.min(0), c.max(0)


def alternative_ok(gpu_bits, diag, K: int, mode: str, idx) -> np.ndarray:
    """For the flat indices idx: does the GPU output lie within 1 ULP of the
    range the mode's chain takes with g, u anywhere in their fp32 error box?"""
    g = np.asarray(gpu_bits).reshape(-1)[idx]
    G = diag["G"].reshape(-1)[idx]
    U = diag["U"].reshape(-1)[idx]
    gamma = accumulation_gamma(K, diag)
    dG = gamma * diag["Ag"].reshape(-1)[idx]
    dU = gamma * diag["Au"].reshape(-1)[idx]
    f, b = bf16_bits_to_f64, _bf16_bits
    if mode == "hf":
        # rounding is monotone: the reachable gb, ub are the roundings of the ends
        glo, ghi = f(b(G - dG)), f(b(G + dG))
        smin, smax = _silu_range(glo, ghi)
        slo, shi = f(b(smin)), f(b(smax))
        ulo, uhi = f(b(U - dU)), f(b(U + dU))
        lo, hi = _product_range(slo, shi, ulo, uhi)
    else:
        smin, smax = _silu_range(G - dG, G + dG)
        lo, hi = _product_range(smin, smax, U - dU, U + dU)
    lob, hib = b(lo), b(hi)
    gv = f(g)
    return ((gv >= f(lob)) & (gv <= f(hib))) | (ulp_distance(g, lob) <= 1) | (ulp_distance(g, hib) <= 1)


def compare(gpu_bits, ref_bits, tau=None, diag=None, K=None, mode=None) -> dict:
    gpu_bits = np.asarray(gpu_bits, dtype=np.uint16)
    ref_bits = np.asarray(ref_bits, dtype=np.uint16)
    assert gpu_bits.shape == ref_bits.shape, (gpu_bits.shape, ref_bits.shape)
    n = gpu_bits.size
    g = bf16_bits_to_f64(gpu_bits)
    r = bf16_bits_to_f64(ref_bits)
    fin_r, fin_g = np.isfinite(r), np.isfinite(g)
    nonfinite_mismatch = int(np.sum((~fin_r | ~fin_g) & (gpu_bits != ref_bits)))
    d = ulp_distance(gpu_bits, ref_bits)
    within = (d <= 1) & fin_r & fin_g
    strict = float(np.mean(within | (~fin_r & (gpu_bits == ref_bits)))) if n else 1.0
    floor = np.abs(r) if tau is None else np.maximum(np.abs(r), np.asarray(tau))
    with np.errstate(divide="ignore", invalid="ignore"):
        raw = np.where(floor > 0, np.abs(g - r) / floor, np.where(g == r, 0.0, np.inf))
    rel = np.where(within | ~fin_r, 0.0, raw)
    rel = np.where(np.isnan(rel), np.inf, rel)
    alt = 0
    if diag is not None and np.any(rel > MAX_REL_ELSEWHERE):
        idx = np.flatnonzero((rel > MAX_REL_ELSEWHERE).reshape(-1))
        okf = alternative_ok(gpu_bits, diag, K, mode, idx)
        flat = rel.reshape(-1).copy()
        flat[idx[okf]] = 0.0
        alt = int(okf.sum())
        rel = flat.reshape(rel.shape)
    outside = ~within & fin_r
    ill = 0 if tau is None else int(np.sum(outside & (np.abs(r) < np.asarray(tau))))
    return {
        "n": n,
        "exact_frac": float(np.mean(d == 0)) if n else 1.0,
        "within_1ulp_of_oracle": strict,   # the stated bar: >= 0.999
        "outside_1ulp": int(np.sum(outside)),
        "max_ulp": int(d.max()) if n else 0,
        "max_rel_elsewhere": float(rel.max()) if n else 0.0,   # outputs no reading explains
        "ill_conditioned": ill,
        "alt_rounding": alt,
        "nonfinite_mismatch": nonfinite_mismatch,
    }


STRICT_FLOOR = 0.999    # 1 ULP of the oracle's own result on >= 99.9% of outputs
ALT_MAX_FRAC = 5e-4     # outputs accepted through the fp32 error box (HF flips, cancellation)


def passes(stats: dict) -> bool:
    n = max(1, stats["n"])
    return (stats["within_1ulp_of_oracle"] >= STRICT_FLOOR
            and stats["max_rel_elsewhere"] <= MAX_REL_ELSEWHERE
            and stats["alt_rounding"] <= ALT_MAX_FRAC * n
            and stats["nonfinite_mismatch"] == 0)


# Every comparison assert_parity makes is kept here with its label; the test
# session writes them out (tests/conftest.py) so the statistics behind each
# "pass" can be read afterwards.
RECORDS = []
CURRENT_TEST = [""]


def assert_parity(gpu_bits, ref_bits, tau=None, what="", diag=None, K=None, mode=None):
    st = compare(gpu_bits, ref_bits, tau, diag, K, mode)
    RECORDS.append({"test": CURRENT_TEST[0], "what": what, **st, "pass": passes(st)})
    assert passes(st), f"parity failed {what}: {st}"
    return st


# ---------------------------------------------------------------------------
# the backward (glu_backward)
# ---------------------------------------------------------------------------
#
# Each gradient is an fp32 sum rounded once to bf16, and the same bar
# applies: 1 ULP of the oracle on >= 99.9%, relative error <= 1e-2
# elsewhere, floored at what fp32 alone can move the output.  The floors:
#   * g, u carry the forward's accumulation error eg = gamma*Ag, eu = gamma*Au
#     (tensor-core bound, the looser of the two kernels');
#   * dG = d*u*SiLU'(g) moves by |d|*(|SiLU'(G)|*eu + |U|*max|SiLU''|*eg)
#     with max|SiLU''| = 1/2 (at 0), plus its own fp32 evaluation, bounded
#     by 16 * 2^-24 relative (expf, two divisions, three products);
#     dU = d*SiLU(g) by |d|*max|SiLU'|*eg (max|SiLU'| < 1.1) plus the same;
#   * grad_h = sum over 2N products (any order: depth <= 2N + 64), grad_W
#     = sum over M products (depth M + 1), each with the dG, dU error above
#     carried through |W| or |h|;
#   * on the tensor cores (glu_bwd_mma_kernel) dG and dU enter exactly, as
#     three bf16 terms, so grad_h sums 6N exact products and grad_W 3M, in
#     the MMA's fp32 adds, bounded here as truncating (2^-23 each).  The
#     floors take the looser of the two kernels' bounds.

BWD_EVAL_REL = 16 * 2.0 ** -24
SILU_D1_MAX = 1.1
SILU_D2_MAX = 0.5


def backward_floors(h, gate, up, dout, G, U, Ag, Au, K):
    """(tau_h [M,K], tau_gate [N,K], tau_up [N,K]) from fp64 operands (h, gate,
    up, dout as values) and the forward's diagnostics G, U, Ag, Au [M,N]."""
    gamma = accumulation_gamma(K, {"acc": "mma"})
    eg, eu = gamma * Ag, gamma * Au
    ad = np.abs(dout)
    ds = _dsilu(G)
    dG = dout * U * ds
    dU = dout * _silu(G)
    edG = ad * (np.abs(ds) * eu + np.abs(U) * SILU_D2_MAX * eg) + BWD_EVAL_REL * np.abs(dG)
    edU = ad * SILU_D1_MAX * eg + BWD_EVAL_REL * np.abs(dU)
    M, N = G.shape
    ag, au, ah = np.abs(gate), np.abs(up), np.abs(h)
    g2n = (6 * N + 64) * 2.0 ** -23
    tau_h = edG @ ag + edU @ au + g2n * (np.abs(dG) @ ag + np.abs(dU) @ au)
    gm = (3 * M + 2) * 2.0 ** -23
    tau_gate = edG.T @ ah + gm * (np.abs(dG).T @ ah)
    tau_up = edU.T @ ah + gm * (np.abs(dU).T @ ah)
    return tau_h, tau_gate, tau_up
