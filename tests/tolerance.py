"""The parity bar between the CUDA path and the oracle.

Stated bar: |delta| <= 1 bf16 ULP of the oracle on >= 99.9% of outputs, and
max relative error <= 1e-2 elsewhere.

Readings used here:
  * ULP distance: the two bf16 patterns mapped to ordered integers
    (sign-magnitude -> two's complement), with +0 and -0 the same point.
  * Relative error of an output outside 1 ULP: |gpu - ref| / max(|ref|, tau),
    where tau bounds what fp32 accumulation alone can move the output.  With
    gamma = K * 2^-24 (the classical bound on a K-term fp32 sum) and the
    oracle's sums of |h*w| (Ag, Au):
        dg = gamma*Ag,  du = gamma*Au,
        tau = |SiLU'(G)*U|*dg + |SiLU(G)|*du  (HF mode adds 2^-8*|G| to dg
              and 2^-8*|U| to du for the bf16 roundings of g and u).
    An output with |ref| < tau sits where u or SiLU(g)*u cancels; any fp32
    summation order may legitimately land anywhere inside tau of it.
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


def conditioning_floor(diag, K: int, mode: str) -> np.ndarray:
    G, U, Ag, Au = diag["G"], diag["U"], diag["Ag"], diag["Au"]
    gamma = K * 2.0 ** -24
    dg, du = gamma * Ag, gamma * Au
    if mode == "hf":
        dg = dg + 2.0 ** -8 * np.abs(G)
        du = du + 2.0 ** -8 * np.abs(U)
    return np.abs(_dsilu(G) * U) * dg + np.abs(_silu(G)) * du


def compare(gpu_bits, ref_bits, tau=None) -> dict:
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
    frac = float(np.mean(within | (~fin_r & (gpu_bits == ref_bits)))) if n else 1.0
    floor = np.abs(r) if tau is None else np.maximum(np.abs(r), np.asarray(tau))
    with np.errstate(divide="ignore", invalid="ignore"):
        raw = np.where(floor > 0, np.abs(g - r) / floor, np.where(g == r, 0.0, np.inf))
    rel = np.where(within | ~fin_r, 0.0, raw)
    rel = np.where(np.isnan(rel), np.inf, rel)
    ill = 0 if tau is None else int(np.sum(~within & fin_r & (np.abs(r) < np.asarray(tau))))
    return {
        "n": n,
        "exact_frac": float(np.mean(d == 0)) if n else 1.0,
        "within_1ulp_frac": frac,
        "max_ulp": int(d.max()) if n else 0,
        "max_rel_elsewhere": float(rel.max()) if n else 0.0,
        "ill_conditioned": ill,
        "nonfinite_mismatch": nonfinite_mismatch,
    }


def passes(stats: dict) -> bool:
    return (stats["within_1ulp_frac"] >= ULP_FRAC_REQUIRED
            and stats["max_rel_elsewhere"] <= MAX_REL_ELSEWHERE
            and stats["nonfinite_mismatch"] == 0)


def assert_parity(gpu_bits, ref_bits, tau=None, what=""):
    st = compare(gpu_bits, ref_bits, tau)
    assert passes(st), f"parity failed {what}: {st}"
    return st
