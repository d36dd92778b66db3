"""Seeded synthetic inputs for the GLU GEMV workloads.

This module is the one piece shared by the CUDA path's harness and the
oracle's tests.  It holds none of the method's arithmetic: it only draws
random numbers, rounds them to bf16 (the storage type of every operand) and
describes the workloads' shapes.

Recipe (all draws on the CPU, so the bytes do not depend on the GPU):
  * each tensor has its own ``torch.Generator`` seeded with
    ``derive_seed(seed, workload, name, index)`` (SHA-256 of the tuple,
    63 bits), so any layer can be regenerated alone;
  * values are ``torch.randn(float32) * std`` rounded to bf16 (round to
    nearest even, torch's float32 -> bfloat16 conversion);
  * "outlier" weights (large-shape sweep): per matrix, round(0.005*N) rows and
    round(0.005*K) columns are picked with ``randperm`` from the same
    generator after the normal draw, and every entry in a picked row or
    column is multiplied by 50 once before rounding (~0.995% of entries).

The pages' model is Qwen3.5-4B-Base (hidden 2560, intermediate 9728); the
other shapes are common decoder MLP sizes.  No dataset is involved.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional, Sequence

import numpy as np
import torch


def derive_seed(seed: int, *names) -> int:
    key = repr((int(seed),) + tuple(names)).encode()
    return int.from_bytes(hashlib.sha256(key).digest()[:8], "little") & ((1 << 63) - 1)


def normal_bf16(shape: Sequence[int], std: float, seed: int, *names) -> torch.Tensor:
    """bf16 CPU tensor of N(0, std^2) draws."""
    g = torch.Generator().manual_seed(derive_seed(seed, *names))
    return (torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def outlier_weight_bf16(N: int, K: int, std: float, seed: int, *names,
                        frac_rows: float = 0.005, frac_cols: float = 0.005,
                        factor: float = 50.0) -> torch.Tensor:
    """N(0, std^2) weights with whole rows and columns scaled by ``factor``."""
    g = torch.Generator().manual_seed(derive_seed(seed, *names))
    w = torch.randn((N, K), generator=g, dtype=torch.float32) * std
    nr, nc = int(round(frac_rows * N)), int(round(frac_cols * K))
    rows = torch.randperm(N, generator=g)[:nr]
    cols = torch.randperm(K, generator=g)[:nc]
    scale = torch.ones((N, K), dtype=torch.float32)
    scale[rows, :] = factor
    scale[:, cols] = factor
    return (w * scale).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor, as a C-contiguous uint16 array."""
    if t.dtype != torch.bfloat16:
        raise TypeError(t.dtype)
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def from_bits(a: np.ndarray) -> torch.Tensor:
    """bf16 CPU tensor from raw bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)


def splitmix64(state: int):
    """SplitMix64 (Steele, Lea, Flood 2014): yields 64-bit words."""
    mask = (1 << 64) - 1
    while True:
        state = (state + 0x9E3779B97F4A7C15) & mask
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        yield z ^ (z >> 31)


def small_int_bf16(shape: Sequence[int], seed: int, lo: int = -8, hi: int = 8) -> np.ndarray:
    """Platform-independent small-integer bf16 bits (for tiny fixtures).

    Integers in [lo, hi] are exact in bf16 and their products and sums are
    exact in binary64, so expected dot products are known exactly.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    gen = splitmix64(seed)
    vals = np.array([lo + (next(gen) % (hi - lo + 1)) for _ in range(n)], dtype=np.float32)
    return bits(torch.from_numpy(vals.reshape(shape)).to(torch.bfloat16))


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    op: str                      # "glu_gemv", "add_rmsnorm_glu", "glu_backward", "silu_mul" or "gdn_gates"
    Ms: tuple                    # batch rows exercised
    K: int
    N: int
    modes: tuple                 # "fused" and/or "hf"
    layers: int                  # independent weight pairs cycled for cold L2
    w_std: float
    h_std: float = 1.0
    outliers: bool = False
    norm_w_std: float = 0.1
    eps: float = 1e-6
    seed: int = 0

    def weight_bytes(self) -> int:
        return 0 if self.op in ("silu_mul", "gdn_gates") else 2 * self.N * self.K * 2

    def input_bytes(self, M: int) -> int:
        """Per call: both weights for the GEMV paths; x [M, 2N] for silu_mul;
        a, b [M, N] for gdn_gates (M tokens, N heads)."""
        if self.op in ("silu_mul", "gdn_gates"):
            return M * 2 * self.N * 2
        return self.weight_bytes()

    def algorithmic_bytes(self, M: int) -> int:
        """Bytes a call must move at least once: both weights, inputs, outputs."""
        b = self.weight_bytes() + M * self.N * 2
        if self.op == "silu_mul":     # x [M, 2N] read, out [M, N] written
            b += M * 2 * self.N * 2
        elif self.op == "gdn_gates":  # a, b read (bf16); g (fp32), beta (bf16) written; A_log, dt_bias read
            return M * self.N * (2 + 2 + 4 + 2) + 2 * self.N * 4
        elif self.op == "glu_gemv":
            b += M * self.K * 2
        elif self.op == "glu_backward":   # weights read and their gradients written; h, dout read; grad_h written
            return 2 * self.weight_bytes() + 2 * M * self.K * 2 + M * self.N * 2
        else:  # x, residual read; residual written; norm_w read
            b += 3 * M * self.K * 2 + self.K * 2
        return b


WORKLOADS = {
    w.name: w for w in [
        # single-rounding mode, one small layer (the oracle runs in well under 1 s)
        Workload("gemv_k1024_n3072", "glu_gemv", (1,), 1024, 3072, ("fused",), 1, 0.02),
        # the headline: Qwen3.5-4B MLP gate/up at batch 1, HF-boundary rounding
        Workload("gemv_k2560_n9728", "glu_gemv", (1,), 2560, 9728, ("hf",), 32, 1 / math.sqrt(2560)),
        # batched decode, both modes
        Workload("gemv_k2560_n9728_batched", "glu_gemv", (1, 2, 4, 8), 2560, 9728, ("fused", "hf"), 32,
                 1 / math.sqrt(2560)),
        # batched decode at 32 and 64 rows (one pass over the weights on the
        # tcgen05 kernel; row blocks of 16 where it does not apply), HF-boundary
        # rounding
        Workload("gemv_k2560_n9728_wide", "glu_gemv", (32, 64), 2560, 9728, ("hf",), 32, 1 / math.sqrt(2560)),
        # the backward of the K=2560, N=9728 layer (gradients of h and both weights)
        Workload("bwd_k2560_n9728", "glu_backward", (1, 8), 2560, 9728, ("fused",), 16, 1 / math.sqrt(2560)),
        # fused residual-add + zero-centred RMSNorm prologue
        Workload("norm_gemv_k2560_n9728", "add_rmsnorm_glu", (1, 4, 8), 2560, 9728, ("hf",), 32,
                 1 / math.sqrt(2560)),
        # large shapes with outlier rows/columns
        Workload("gemv_k4096_n11008", "glu_gemv", (1, 8, 16), 4096, 11008, ("fused", "hf"), 24, 1 / 64.0,
                 outliers=True),
        Workload("gemv_k4096_n14336", "glu_gemv", (1, 8, 16), 4096, 14336, ("fused", "hf"), 24, 1 / 64.0,
                 outliers=True),
        # the standalone epilogue on a prefill batch (halves layout [M, 2N]):
        # 4096 tokens of the Qwen3.5-4B MLP; two inputs of 159 MB cycled for cold L2
        Workload("silu_mul_m4096_n9728", "silu_mul", (4096,), 0, 9728, ("hf", "fused"), 2, 0.0),
        # the gated-delta-net gates beside the GLU: 262144 tokens x 32 heads, four
        # cycled inputs (134 MB of a, b) for cold L2; no rounding mode applies
        Workload("gdn_gates_t262144_h32", "gdn_gates", (262144,), 0, 32, ("hf",), 4, 0.0),
    ]
}

HEADLINE = "gemv_k2560_n9728"


def layer_weights(w: Workload, layer: int, seed: Optional[int] = None):
    """(gate_w, up_w) bf16 CPU tensors [N, K] of one layer."""
    s = w.seed if seed is None else seed
    if w.outliers:
        g = outlier_weight_bf16(w.N, w.K, w.w_std, s, w.name, "gate_w", layer)
        u = outlier_weight_bf16(w.N, w.K, w.w_std, s, w.name, "up_w", layer)
    else:
        g = normal_bf16((w.N, w.K), w.w_std, s, w.name, "gate_w", layer)
        u = normal_bf16((w.N, w.K), w.w_std, s, w.name, "up_w", layer)
    return g, u


def hidden(w: Workload, M: int, seed: Optional[int] = None) -> torch.Tensor:
    """h [M, K] bf16 CPU tensor (glu_gemv input)."""
    return normal_bf16((M, w.K), w.h_std, w.seed if seed is None else seed, w.name, "h", M)


def upstream(w: Workload, M: int, seed: Optional[int] = None) -> torch.Tensor:
    """dout [M, N] bf16 CPU tensor ~ N(0, 1): the upstream gradient of glu_backward."""
    return normal_bf16((M, w.N), 1.0, w.seed if seed is None else seed, w.name, "dout", M)


def projections(w: Workload, M: int, layer: int = 0, seed: Optional[int] = None) -> torch.Tensor:
    """x [M, 2N] bf16 CPU tensor for silu_mul: the gate and up projections of
    M tokens side by side, N(0, h_std) (projections of a unit-variance hidden
    state through N(0, 1/sqrt(K)) weights)."""
    return normal_bf16((M, 2 * w.N), w.h_std, w.seed if seed is None else seed, w.name, "x", layer)


def gdn_inputs(w: Workload, T: int, layer: int = 0, seed: Optional[int] = None):
    """(a, b) bf16 [T, H] CPU tensors ~ N(0, 3) and (A_log, dt_bias) float32 [H]
    ~ N(0, 1) for gdn_gates: T tokens, H = w.N heads."""
    s = w.seed if seed is None else seed
    a = normal_bf16((T, w.N), 3.0, s, w.name, "a", layer)
    b = normal_bf16((T, w.N), 3.0, s, w.name, "b", layer)
    A_log = normal_bf16((w.N,), 1.0, s, w.name, "A_log").float()
    dt_bias = normal_bf16((w.N,), 1.0, s, w.name, "dt_bias").float()
    return a, b, A_log, dt_bias


def norm_inputs(w: Workload, M: int, seed: Optional[int] = None):
    """(x, residual, norm_w) bf16 CPU tensors for add_rmsnorm_glu."""
    s = w.seed if seed is None else seed
    x = normal_bf16((M, w.K), 1.0, s, w.name, "x", M)
    r = normal_bf16((M, w.K), 1.0, s, w.name, "residual", M)
    nw = normal_bf16((w.K,), w.norm_w_std, s, w.name, "norm_w")
    return x, r, nw
