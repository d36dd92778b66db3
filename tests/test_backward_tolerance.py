"""The backward's parity bar (tolerance.backward_floors) on the CPU.

A plain float32 implementation of the backward -- fp32 products and sums
(BLAS sgemm), SiLU and SiLU' in fp32, one rounding to bf16 at the end -- is a
correct result within fp32's accuracy, so it must pass the bar against the
fp64 oracle; the same implementation with one plausible mistake planted
(a dropped term, a swapped gradient, SiLU for SiLU') must fail it.  This
pins the bar from both sides before any GPU result is held against it."""
import numpy as np
import pytest
import torch

import glu_inputs as gi
import oracle
import tolerance as tol


def _f64(bits):
    return tol.bf16_bits_to_f64(bits)


def _bits_from_f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _case(M, N, K, seed):
    h = gi.bits(gi.normal_bf16((M, K), 1.0, seed, "bt-h"))
    g = gi.bits(gi.normal_bf16((N, K), K ** -0.5, seed, "bt-g"))
    u = gi.bits(gi.normal_bf16((N, K), K ** -0.5, seed, "bt-u"))
    d = gi.bits(gi.normal_bf16((M, N), 1.0, seed, "bt-d"))
    return h, g, u, d


def _reference(h, g, u, d):
    gh, gg, gu = oracle.glu_backward(h, g, u, d)
    _, diag = oracle.glu_gemv(h, g, u, "fused", diagnostics=True)
    K = h.shape[1]
    floors = tol.backward_floors(_f64(h), _f64(g), _f64(u), _f64(d), diag["G"], diag["U"], diag["Ag"], diag["Au"], K)
    refs = tuple(oracle.bf16_round_array(x) for x in (gh, gg, gu))
    return refs, floors


def _float32_backward(h, g, u, d, mistake=None):
    h32, g32, u32, d32 = (_f64(a).astype(np.float32) for a in (h, g, u, d))
    G = h32 @ g32.T
    U = h32 @ u32.T
    with np.errstate(over="ignore"):
        t = np.exp(-np.abs(G))
    one = np.float32(1.0)
    sig = np.where(G >= 0, one, t) / (one + t)
    rest = np.where(G >= 0, t, one) / (one + t)
    silu = G * sig
    dsilu = sig * (one + G * rest)
    if mistake == "dsilu_is_sigmoid":
        dsilu = sig
    if mistake == "dU_uses_dsilu":
        silu = dsilu
    dG = (d32 * U) * dsilu
    dU = d32 * silu
    grad_h = dG @ g32 + dU @ u32
    if mistake == "grad_h_drops_up":
        grad_h = dG @ g32
    if mistake == "grad_h_sign":
        grad_h = dG @ g32 - dU @ u32
    grad_gate = dG.T @ h32
    grad_up = dU.T @ h32
    if mistake == "grads_swapped":
        grad_gate, grad_up = grad_up, grad_gate
    return tuple(_bits_from_f32(x) for x in (grad_h, grad_gate, grad_up))


@pytest.mark.parametrize("M,N,K,seed", [(1, 700, 520, 1), (4, 700, 520, 2), (16, 2048, 1024, 3)])
def test_float32_backward_meets_the_bar(M, N, K, seed):
    h, g, u, d = _case(M, N, K, seed)
    refs, floors = _reference(h, g, u, d)
    got = _float32_backward(h, g, u, d)
    for name, a, r, tau in zip(("grad_h", "grad_gate", "grad_up"), got, refs, floors):
        tol.assert_parity(a, r, tau, f"float32 {name} M={M}")


@pytest.mark.parametrize("mistake", ["dsilu_is_sigmoid", "dU_uses_dsilu", "grad_h_drops_up", "grad_h_sign",
                                     "grads_swapped"])
def test_planted_mistakes_fail_the_bar(mistake):
    h, g, u, d = _case(4, 700, 520, 2)
    refs, floors = _reference(h, g, u, d)
    got = _float32_backward(h, g, u, d, mistake)
    results = [tol.passes(tol.compare(a, r, tau)) for a, r, tau in zip(got, refs, floors)]
    assert not all(results), f"{mistake} passed the bar"


def test_bf16_round_array_is_the_scalar_rounding():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-45, 40, 2000),
                        [0.0, -0.0, np.inf, -np.inf, np.nan, 3.3895e38, 3.4e38, 1e-40, -9.2e-41]])
    assert np.array_equal(oracle.bf16_round_array(x), np.array([oracle.bf16_round(v) for v in x], dtype=np.uint16))


def _fma32(a, b, c):
    """fp32 fused multiply-add, elementwise: the product of two fp32 values is
    exact in binary64 and the sum is rounded once to fp32 (a second rounding
    in binary64 first can differ only at exact fp32 ties, far rarer than the
    bar's allowance)."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _kernel_order_backward(h, g, u, d):
    """glu_backward's sums in the kernels' order (csrc/glu_backward.cuh): dG,
    dU from fp32 g, u; grad_h per 512-column block and row split as two
    alternating-row FMA chains (dG*Wg then dU*Wu per row) added half 0 +
    half 1, then the splits summed in order; grad_W as an FMA chain over
    m = 0, 1, ...  g and u themselves come from an fp32 GEMM (their own
    order is the forward's, checked by the forward's bar)."""
    h32, g32, u32, d32 = (_f64(a).astype(np.float32) for a in (h, g, u, d))
    M, K = h32.shape
    N = g32.shape[0]
    G, U = h32 @ g32.T, h32 @ u32.T
    with np.errstate(over="ignore"):
        t = np.exp(-np.abs(G))
    one = np.float32(1.0)
    sig = np.where(G >= 0, one, t) / (one + t)
    rest = np.where(G >= 0, t, one) / (one + t)
    silu, dsilu = G * sig, sig * (one + G * rest)
    dG, dU = ((d32 * U) * dsilu).astype(np.float32), (d32 * silu).astype(np.float32)
    nsplit = max(1, min(48, N // 256))
    part = np.zeros((nsplit, M, K), dtype=np.float32)
    for b in range(nsplit):
        n0, n1 = N * b // nsplit, N * (b + 1) // nsplit
        halves = []
        for half in (0, 1):
            acc = np.zeros((M, K), dtype=np.float32)
            for n in range(n0 + half, n1, 2):
                acc = _fma32(dG[:, n:n + 1], g32[n][None, :], acc)
                acc = _fma32(dU[:, n:n + 1], u32[n][None, :], acc)
            halves.append(acc)
        part[b] = halves[0] + halves[1]
    grad_h = part[0].copy()
    for b in range(1, nsplit):
        grad_h = (grad_h + part[b]).astype(np.float32)
    sg = np.zeros((N, K), dtype=np.float32)
    su = np.zeros((N, K), dtype=np.float32)
    for m in range(M):
        sg = _fma32(dG[m][:, None], h32[m][None, :], sg)
        su = _fma32(dU[m][:, None], h32[m][None, :], su)
    return tuple(_bits_from_f32(x) for x in (grad_h, sg, su))


@pytest.mark.parametrize("M,N,K,seed", [(1, 1300, 600, 4), (16, 2048, 1024, 5)])
def test_kernel_order_backward_meets_the_bar(M, N, K, seed):
    """The kernels' own summation order (row splits of 256+ rows, alternating
    rows per half, in-order split sums) passes the bar."""
    h, g, u, d = _case(M, N, K, seed)
    refs, floors = _reference(h, g, u, d)
    got = _kernel_order_backward(h, g, u, d)
    for name, a, r, tau in zip(("grad_h", "grad_gate", "grad_up"), got, refs, floors):
        tol.assert_parity(a, r, tau, f"kernel order {name} M={M}")
