"""GPU parity of glu_backward (grad_h, grad_gate, grad_up) against the fp64
oracle, through the C ABI, with the bar of tolerance.backward_floors; the
autograd Function built on it; determinism and the degenerate shapes."""
import numpy as np
import pytest
import torch

import glu_inputs as gi
import oracle
import tolerance as tol

pytestmark = pytest.mark.gpu

mb = pytest.importorskip("memory_bound_glu_gb300")
DEV = torch.device("cuda:0")
BACKWARD = 8   # mbglu_last_variant() after glu_backward


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _inputs(M, N, K, seed, tag="bw"):
    h = gi.normal_bf16((M, K), 1.0, seed, f"{tag}-h")
    g = gi.normal_bf16((N, K), K ** -0.5, seed, f"{tag}-g")
    u = gi.normal_bf16((N, K), K ** -0.5, seed, f"{tag}-u")
    d = gi.normal_bf16((M, N), 1.0, seed, f"{tag}-d")
    return h, g, u, d


def _check(got, h, g, u, d, what, rows=None):
    """got: (grad_h, grad_gate, grad_up) bf16 CPU tensors (None to skip); rows:
    the feature rows of grad_gate / grad_up to compare (all by default)."""
    hb, gb, ub, db = (gi.bits(t) for t in (h, g, u, d))
    gh, gg, gu = oracle.glu_backward(hb, gb, ub, db)
    _, diag = oracle.glu_gemv(hb, gb, ub, "fused", diagnostics=True)
    f = tol.bf16_bits_to_f64
    taus = tol.backward_floors(f(hb), f(gb), f(ub), f(db), diag["G"], diag["U"], diag["Ag"], diag["Au"], h.shape[1])
    sel = slice(None) if rows is None else rows
    stats = {}
    for name, a, ref, tau, r in zip(("grad_h", "grad_gate", "grad_up"), got, (gh, gg, gu), taus,
                                    (slice(None), sel, sel)):
        if a is None:
            continue
        stats[name] = tol.assert_parity(gi.bits(a)[r], oracle.bf16_round_array(ref[r]), tau[r], f"{what} {name}")
    return stats


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 13, 16])
def test_backward_every_batch_tile(M):
    """Ragged N and K (the row splits, the 512-column blocks and the 8-column
    stores all end mid-way); the first step runs on the kernel the forward
    takes at this batch."""
    N, K = 1337, 1288
    h, g, u, d = _inputs(M, N, K, M)
    got = mb.glu_backward(h.to(DEV), g.to(DEV), u.to(DEV), d.to(DEV))
    torch.cuda.synchronize()
    assert mb.last_variant() == BACKWARD
    assert mb.last_backward_path() == (2 if M <= 2 else 3 if M <= 16 else 1)
    _check(tuple(t.cpu() for t in got), h, g, u, d, f"M={M}")
    assert mb.read_device_error() == 0


@pytest.mark.parametrize("M,N,K", [
    (3, 17, 8),        # one column box, 8 columns in it; shares of 8-9 rows (one partial block)
    (6, 1000, 192),    # K a multiple of 64, not of 128: the last slice's second box lies past K
    (7, 2049, 1032),   # a box with 8 columns in it; partial top blocks
    (8, 40, 4096),     # 32 slices in several column groups; every share one partial block
    (4, 9728, 2560),   # the headline layer at batch 4
    (16, 2049, 1032),  # batch 16: two batch tiles, three terms each
    (11, 9728, 2560),  # batch 11 on the headline layer (rows 11..15 of the tile zero)
])
def test_backward_tensor_core_pass(M, N, K):
    """The one-pass step on the tensor cores (dG, dU as three bf16 terms):
    ragged column slices and row blocks, against the oracle."""
    h, g, u, d = _inputs(M, N, K, 100 + M, "bwtc")
    got = mb.glu_backward(h.to(DEV), g.to(DEV), u.to(DEV), d.to(DEV))
    torch.cuda.synchronize()
    assert mb.last_backward_path() == 3
    rows = None if N <= 2049 else np.sort(np.random.default_rng(M).choice(N, 600, replace=False))
    _check(tuple(t.cpu() for t in got), h, g, u, d, f"tensor-core pass M={M} N={N} K={K}", rows=rows)
    assert mb.read_device_error() == 0


@pytest.mark.parametrize("M", [17, 32, 64])
def test_backward_wide_batch(M):
    """Batches above one pass: dG, dU per 16-row block, grad_h per pass of 8
    rows, the weight gradients summed over all M rows at once."""
    N, K = 1500, 1024
    h, g, u, d = _inputs(M, N, K, M, "bwwide")
    got = mb.glu_backward(h.to(DEV), g.to(DEV), u.to(DEV), d.to(DEV))
    torch.cuda.synchronize()
    assert mb.last_variant() == BACKWARD
    _check(tuple(t.cpu() for t in got), h, g, u, d, f"M={M}")
    assert mb.read_device_error() == 0


def test_backward_autograd_at_batch_32():
    """DualWeightGlu runs wherever its forward does: batch 32 (row blocks)."""
    M, N, K = 32, 700, 512
    h0, g0, u0, d0 = (t.to(DEV) for t in _inputs(M, N, K, 5, "bwa32"))
    h = h0.clone().requires_grad_(True)
    g = g0.clone().requires_grad_(True)
    u = u0.clone().requires_grad_(True)
    out = mb.DualWeightGlu.apply(h, g, u)
    out.backward(d0)
    torch.cuda.synchronize()
    _check((h.grad.cpu(), g.grad.cpu(), u.grad.cpu()), h0.cpu(), g0.cpu(), u0.cpu(), d0.cpu(), "autograd M=32")


@pytest.mark.parametrize("N,K", [(1, 8), (7, 64), (256, 520), (3000, 2560), (513, 4100), (300, 8192), (200, 9216)])
def test_backward_shapes(N, K):
    M = 4
    h, g, u, d = _inputs(M, N, K, N, "bws")
    got = mb.glu_backward(h.to(DEV), g.to(DEV), u.to(DEV), d.to(DEV))
    torch.cuda.synchronize()
    _check(tuple(t.cpu() for t in got), h, g, u, d, f"N={N} K={K}")


def test_backward_strided_and_subsets():
    """Operands and gradients as views into wider buffers (odd strides take
    the element-wise loads and stores), and each subset of the outputs."""
    M, N, K = 5, 999, 1030
    hb = gi.normal_bf16((M, K + 9), 1.0, 3, "bwt-h")
    gb = gi.normal_bf16((N, K + 3), K ** -0.5, 3, "bwt-g")
    ub = gi.normal_bf16((N, K + 16), K ** -0.5, 3, "bwt-u")
    db = gi.normal_bf16((M, N + 5), 1.0, 3, "bwt-d")
    h, g, u, d = hb[:, 1:1 + K], gb[:, :K], ub[:, 8:8 + K], db[:, :N]
    hd, gd, ud, dd = hb.to(DEV)[:, 1:1 + K], gb.to(DEV)[:, :K], ub.to(DEV)[:, 8:8 + K], db.to(DEV)[:, :N]
    oh = torch.full((M, K + 24), float("nan"), dtype=torch.bfloat16, device=DEV)
    og = torch.full((N, K + 8), float("nan"), dtype=torch.bfloat16, device=DEV)
    ou = torch.full((N, K + 1), float("nan"), dtype=torch.bfloat16, device=DEV)
    mb.glu_backward(hd, gd, ud, dd, grad_h=oh[:, :K], grad_gate=og[:, 8:], grad_up=ou[:, :K])
    torch.cuda.synchronize()
    assert mb.last_backward_path() == 1   # K % 8 != 0: the separate kernels
    assert torch.isnan(oh[:, K:].float()).all() and torch.isnan(og[:, :8].float()).all()
    assert torch.isnan(ou[:, K:].float()).all()
    full = (oh[:, :K].cpu(), og[:, 8:].cpu(), ou[:, :K].cpu())
    _check(full, h.contiguous(), g.contiguous(), u.contiguous(), d.contiguous(), "strided")
    only_h = mb.glu_backward(hd, gd, ud, dd, want_w=False)
    only_w = mb.glu_backward(hd, gd, ud, dd, want_h=False)
    torch.cuda.synchronize()
    assert only_h[1] is None and only_w[0] is None
    assert torch.equal(only_h[0].cpu().view(torch.int16), full[0].view(torch.int16))
    assert torch.equal(only_w[1].cpu().view(torch.int16), full[1].view(torch.int16))
    assert torch.equal(only_w[2].cpu().view(torch.int16), full[2].view(torch.int16))


def test_backward_deterministic():
    M, N, K = 8, 3001, 2560
    h, g, u, d = (t.to(DEV) for t in _inputs(M, N, K, 9, "bwd"))
    a = mb.glu_backward(h, g, u, d)
    b = mb.glu_backward(h, g, u, d)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_backward_degenerate_shapes():
    K = 64
    h = torch.zeros((0, K), dtype=torch.bfloat16, device=DEV)
    g = gi.normal_bf16((10, K), 0.1, 1, "bwz-g").to(DEV)
    gg = torch.full((10, K), 3.0, dtype=torch.bfloat16, device=DEV)
    gu = torch.full((10, K), 3.0, dtype=torch.bfloat16, device=DEV)
    mb.glu_backward(h, g, g, torch.zeros((0, 10), dtype=torch.bfloat16, device=DEV), grad_gate=gg, grad_up=gu,
                    want_h=False)                                   # M == 0: the weight gradients are 0
    gh = torch.full((3, K), 3.0, dtype=torch.bfloat16, device=DEV)
    mb.glu_backward(torch.ones((3, K), dtype=torch.bfloat16, device=DEV), g[:0], g[:0],
                    torch.zeros((3, 0), dtype=torch.bfloat16, device=DEV), grad_h=gh, want_w=False)   # N == 0
    torch.cuda.synchronize()
    assert (gi.bits(gg.cpu()) == 0).all() and (gi.bits(gu.cpu()) == 0).all() and (gi.bits(gh.cpu()) == 0).all()
    with pytest.raises(mb.MbgluError):
        mb.glu_backward(torch.zeros((65, K), dtype=torch.bfloat16, device=DEV), g, g,
                        torch.zeros((65, 10), dtype=torch.bfloat16, device=DEV))


def test_autograd_function_matches_glu_backward():
    """DualWeightGlu: forward is glu_gemv (FUSED), backward returns
    glu_backward's gradients to h and to both weights."""
    M, N, K = 4, 1000, 1024
    h0, g0, u0, d0 = (t.to(DEV) for t in _inputs(M, N, K, 11, "bwa"))
    h = h0.clone().requires_grad_(True)
    g = g0.clone().requires_grad_(True)
    u = u0.clone().requires_grad_(True)
    out = mb.DualWeightGlu.apply(h, g, u)
    assert torch.equal(out.detach().view(torch.int16), mb.glu_gemv(h0, g0, u0, mode="fused").view(torch.int16))
    out.backward(d0)
    ref = mb.glu_backward(h0, g0, u0, d0)
    torch.cuda.synchronize()
    for a, b in zip((h.grad, g.grad, u.grad), ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
