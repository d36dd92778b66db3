"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar (tolerance.py): |delta| <= 1 bf16 ULP on >= 99.9% of outputs, relative
error <= 1e-2 elsewhere (floored at the fp32-accumulation conditioning
bound); the updated residual of add_rmsnorm_glu must match bit for bit (one
correctly rounded addition).  Every workload is checked at its full size on
a sampled layer, plus small shapes that span several tiles and ragged tails,
strided and unaligned operands, and the degenerate cases.
"""
import functools

import numpy as np
import pytest
import torch

import glu_inputs as gi
import oracle
import tolerance as tol

pytestmark = pytest.mark.gpu

mb = pytest.importorskip("memory_bound_glu_gb300")
DEV = torch.device("cuda:0")


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(autouse=True)
def _gpu():
    _need_gpu()
    yield


def oracle_glu(h, g, u, mode):
    out, diag = oracle.glu_gemv(gi.bits(h), gi.bits(g), gi.bits(u), mode, diagnostics=True)
    return out, (tol.conditioning_floor(diag, h.shape[1], mode), diag, h.shape[1], mode)


def parity(got, ref, tau_info, what=""):
    tau, diag, K, mode = tau_info
    if mb.last_variant() in (4, 7, 9, 10):   # tensor-core accumulation bound (7: row blocks, mostly; 9: tcgen05)
        diag["acc"] = "mma"
        tau = tol.conditioning_floor(diag, K, mode)
    return tol.assert_parity(got, ref, tau, what, diag=diag, K=K, mode=mode)


def run_gpu(h, g, u, mode, **kw):
    out = mb.glu_gemv(h.to(DEV), g.to(DEV), u.to(DEV), mode=mode, **kw)
    torch.cuda.synchronize()
    return gi.bits(out.cpu())


FAST = (1, 4, 10)   # the streaming kernels: CUDA-core FMA, tensor core, tensor core with h in registers
SLICE = 10          # mbglu_last_variant(): the K-slice tensor-core kernel


def tc_variant(M, K):
    """The kernel a tensor-core batch (M >= 3, aligned operands, K % 16 == 0)
    takes: the K-slice kernel where its plan fits (K up to 4608 at M <= 8, up to
    2560 at M = 9..16), else the kernel with h in shared memory."""
    fits = 256 <= K and (K <= 4608 if M <= 8 else K <= 2560)
    return SLICE if fits else 4


def check(h, g, u, mode, what="", variant=None):
    got = run_gpu(h, g, u, mode)
    if variant == 1:
        assert mb.last_variant() in FAST
    elif variant is not None:
        assert mb.last_variant() == variant
    ref, tau = oracle_glu(h, g, u, mode)
    return parity(got, ref, tau, what)


# ---------------------------------------------------------------------------
# small shapes: tiles, tails, every batch size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["fused", "hf"])
@pytest.mark.parametrize("M", list(range(1, 17)))
def test_every_batch_size(M, mode):
    N, K = 1337, 1024 + 256 + 8   # ragged N over 152 CTAs, K with a short last chunk
    h = gi.normal_bf16((M, K), 1.0, M, "bs-h")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "bs-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "bs-u")
    check(h, g, u, mode, f"M={M}", variant=1)


@pytest.mark.parametrize("N,K", [(1, 8), (7, 64), (152, 256), (153, 2048), (4096, 2056), (300, 4104),
                                 (2000, 5120), (513, 8192)])
def test_shapes_fast_path(N, K):
    M = 3
    h = gi.normal_bf16((M, K), 1.0, N, "sh-h")
    g = gi.normal_bf16((N, K), K ** -0.5, N, "sh-g")
    u = gi.normal_bf16((N, K), K ** -0.5, N, "sh-u")
    check(h, g, u, "hf", f"N={N} K={K}", variant=1)


@pytest.mark.parametrize("K", [1, 7, 9, 1001])
def test_ragged_k_uses_generic_kernel(K):
    M, N = 2, 517
    h = gi.normal_bf16((M, K), 1.0, K, "rk-h")
    g = gi.normal_bf16((N, K), K ** -0.5, K, "rk-g")
    u = gi.normal_bf16((N, K), K ** -0.5, K, "rk-u")
    for mode in ("fused", "hf"):
        check(h, g, u, mode, f"K={K}", variant=2)


def test_large_m16_k_uses_generic_when_h_does_not_fit():
    M, N, K = 16, 300, 16384
    h = gi.normal_bf16((M, K), 1.0, 1, "bigk-h")
    g = gi.normal_bf16((N, K), K ** -0.5, 1, "bigk-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 1, "bigk-u")
    check(h, g, u, "fused", "M=16 K=16384", variant=2)


@pytest.mark.parametrize("M,N,K", [(16, 700, 4096), (13, 1337, 4096), (16, 153, 6144), (9, 700, 8192),
                                   (16, 300, 8192), (8, 1000, 6144)])
@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_tensor_core_k_phases(M, N, K, mode):
    """M*K too large to keep h whole beside a deep ring: the tensor-core kernel
    stages h through shared memory in two K-phases and carries every group's
    accumulators across the boundary (the last two shapes did not fit the
    tensor-core kernel at all with h whole).  Batch 8 at K = 6144 lies past
    the K-slice kernel's reach and runs here too."""
    h = gi.normal_bf16((M, K), 1.0, M, "kp-h")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "kp-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "kp-u")
    check(h, g, u, mode, f"M={M} N={N} K={K}", variant=tc_variant(M, K))


@pytest.mark.parametrize("K", [4096, 6144])
def test_k_phases_deterministic_and_row_permutation_bitwise(K):
    """With K-phases, as with one phase, a row's bits do not depend on where
    the row falls (how the CTA's units are cut between warps and phases): batch
    16 on the kernel with h in shared memory, in two K-phases at K = 4096 and
    at K = 6144."""
    M, N = 16, 1500
    h = gi.normal_bf16((M, K), 1.0, 7, "kpp-h").to(DEV)
    g = gi.normal_bf16((N, K), K ** -0.5, 7, "kpp-g").to(DEV)
    u = gi.normal_bf16((N, K), K ** -0.5, 7, "kpp-u").to(DEV)
    a = mb.glu_gemv(h, g, u, mode="hf")
    assert mb.last_variant() == tc_variant(M, K)
    b = mb.glu_gemv(h, g, u, mode="hf")
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(1)).to(DEV)
    c = mb.glu_gemv(h, g[perm], u[perm], mode="hf")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a[:, perm].view(torch.int16), c.view(torch.int16))
    assert mb.read_device_error() == 0


def test_strided_views_fast_and_generic():
    """Row strides are honoured: operands sliced out of wider buffers."""
    M, N, K = 4, 999, 1536
    hb = gi.normal_bf16((M, K + 40), 1.0, 2, "st-h")
    gb = gi.normal_bf16((N, K + 64), K ** -0.5, 2, "st-g")
    ub = gi.normal_bf16((N, K + 16), K ** -0.5, 2, "st-u")
    h, g, u = hb[:, 8:8 + K], gb[:, :K], ub[:, 16:16 + K]
    ref, tau = oracle_glu(h.contiguous(), g.contiguous(), u.contiguous(), "hf")
    hd, gd, ud = hb.to(DEV)[:, 8:8 + K], gb.to(DEV)[:, :K], ub.to(DEV)[:, 16:16 + K]
    outb = torch.full((M, N + 24), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = outb[:, 24:]
    mb.glu_gemv(hd, gd, ud, out=out, mode="hf")
    torch.cuda.synchronize()
    assert mb.last_variant() in FAST
    parity(gi.bits(out.cpu()), ref, tau, "strided")
    assert torch.isnan(outb[:, :24].float()).all(), "wrote outside out"
    # an odd element offset breaks 16-byte alignment of the weights: generic kernel
    g2 = gb.to(DEV)[:, 1:1 + K]
    ref2, tau2 = oracle_glu(h.contiguous(), gb[:, 1:1 + K].contiguous(), u.contiguous(), "fused")
    o2 = mb.glu_gemv(hd, g2, ud, mode="fused")
    torch.cuda.synchronize()
    assert mb.last_variant() == 2
    parity(gi.bits(o2.cpu()), ref2, tau2, "unaligned")


@pytest.mark.parametrize("K,ld_pad,h_off,expect", [(2560, 0, 0, SLICE), (2560, 64, 8, SLICE), (4096, 8, 1, 1),
                                                    (1024, 0, 3, SLICE), (5120, 0, 0, 1), (2568, 0, 0, SLICE),
                                                    (3584, 0, 2, 1)])
def test_batch_one_paths(K, ld_pad, h_off, expect):
    """M = 1: strided weight rows, an h that is not 16-byte aligned; up to
    K = 3072 the K-slice kernel (h in registers, one segment per warp), above
    it the CUDA-core streaming kernel (h in registers up to K = 4096, in shared
    memory beyond)."""
    N = 2111
    hb = gi.normal_bf16((1, K + 8), 1.0, K, "m1-h")
    gb = gi.normal_bf16((N, K + ld_pad), K ** -0.5, K, "m1-g")
    ub = gi.normal_bf16((N, K + ld_pad), K ** -0.5, K, "m1-u")
    h, g, u = hb[:, h_off:h_off + K], gb[:, :K], ub[:, :K]
    ref, tau = oracle_glu(h.contiguous(), g.contiguous(), u.contiguous(), "hf")
    out = mb.glu_gemv(hb.to(DEV)[:, h_off:h_off + K], gb.to(DEV)[:, :K], ub.to(DEV)[:, :K], mode="hf")
    torch.cuda.synchronize()
    assert mb.last_variant() == expect
    parity(gi.bits(out.cpu()), ref, tau, f"M=1 K={K}")


@pytest.mark.parametrize("M", [3, 4, 5, 8, 9, 12, 16])
@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_tensor_core_kernel(M, mode):
    """Batch >= 3 on the tensor cores: ragged N (partial last 8-row group),
    several K-segments, on the K-slice kernel (h in registers; 16-row tiles at
    batch 9..16)."""
    N, K = 1339, 2560
    h = gi.normal_bf16((M, K), 1.0, M, "tc-h")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "tc-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "tc-u")
    check(h, g, u, mode, f"tc M={M}", variant=tc_variant(M, 2560))


@pytest.mark.parametrize("K,ld_pad,h_off", [(1024, 8, 8), (4096, 0, 0), (2576, 16, 1), (1040, 0, 0)])
def test_tensor_core_kernel_strides_and_k(K, ld_pad, h_off):
    M, N = 8, 611
    hb = gi.normal_bf16((M, K + 8), 1.0, K, "tcs-h")
    gb = gi.normal_bf16((N, K + ld_pad), K ** -0.5, K, "tcs-g")
    ub = gi.normal_bf16((N, K + ld_pad), K ** -0.5, K, "tcs-u")
    h, g, u = hb[:, h_off:h_off + K], gb[:, :K], ub[:, :K]
    ref, tau = oracle_glu(h.contiguous(), g.contiguous(), u.contiguous(), "hf")
    out = mb.glu_gemv(hb.to(DEV)[:, h_off:h_off + K], gb.to(DEV)[:, :K], ub.to(DEV)[:, :K], mode="hf")
    torch.cuda.synchronize()
    assert mb.last_variant() == SLICE
    parity(gi.bits(out.cpu()), ref, tau, f"tc K={K}")


def test_guard_band_untouched():
    M, N, K = 5, 2049, 1024
    h = gi.normal_bf16((M, K), 1.0, 3, "gd-h")
    g = gi.normal_bf16((N, K), K ** -0.5, 3, "gd-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 3, "gd-u")
    buf = torch.full((M + 2, N + 64), -7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[1:1 + M, 32:32 + N]
    mb.glu_gemv(h.to(DEV), g.to(DEV), u.to(DEV), out=out, mode="fused")
    torch.cuda.synchronize()
    b = buf.float().cpu()
    mask = torch.ones_like(b, dtype=torch.bool)
    mask[1:1 + M, 32:32 + N] = False
    assert (b[mask] == -7.0).all()
    ref, tau = oracle_glu(h, g, u, "fused")
    parity(gi.bits(out.cpu()), ref, tau, "guard")


def test_degenerate_sizes():
    K = 64
    h = gi.normal_bf16((2, K), 1.0, 4, "dg-h").to(DEV)
    w = gi.normal_bf16((10, K), 0.1, 4, "dg-w").to(DEV)
    # N == 0 and M == 0: no-op
    o = torch.empty((2, 0), dtype=torch.bfloat16, device=DEV)
    mb.glu_gemv(h, w[:0], w[:0], out=o)
    assert mb.last_variant() == 0
    o = torch.full((0, 10), 1.0, dtype=torch.bfloat16, device=DEV)
    mb.glu_gemv(h[:0], w, w, out=o)
    # K == 0: +0 everywhere
    o = torch.full((2, 10), 3.0, dtype=torch.bfloat16, device=DEV)
    mb.glu_gemv(h[:, :0], w[:, :0], w[:, :0], out=o, mode="hf")
    torch.cuda.synchronize()
    assert mb.last_variant() == 3
    assert (gi.bits(o.cpu()) == 0).all()
    with pytest.raises(mb.MbgluError):
        mb.glu_gemv(torch.zeros((mb.MAX_M + 1, K), dtype=torch.bfloat16, device=DEV), w, w)


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_closed_forms_on_gpu(mode):
    K, N = 256, 300
    h = gi.normal_bf16((4, K), 1.0, 5, "cf-h")
    z = torch.zeros((N, K), dtype=torch.bfloat16)
    assert (run_gpu(h, z, z, mode) == 0).all()            # zero weights -> +0
    eye = torch.eye(K, dtype=torch.bfloat16)
    got = run_gpu(h, eye, eye, mode)                       # identity rows: SiLU(h_i)*h_i
    ref = oracle.glu_gemv(gi.bits(h), gi.bits(eye), gi.bits(eye), mode)
    assert np.array_equal(tol.ordered(got), tol.ordered(ref))


@pytest.mark.parametrize("mode", ["fused", "hf"])
def test_silu_exhaustive_over_bf16_gate_values_on_gpu(mode):
    """h = e_0, W_gate[:,0] = every finite bf16, W_up[:,0] = 1: out = bf16(SiLU(g))
    for every g, including the far negative tail where e^-g overflows fp32."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = pats[(pats & 0x7FFF) < 0x7F80]
    N, K = g.size, 8
    gw = np.zeros((N, K), dtype=np.uint16)
    gw[:, 0] = g
    uw = np.zeros((N, K), dtype=np.uint16)
    uw[:, 0] = 0x3F80
    h = np.zeros((1, K), dtype=np.uint16)
    h[0, 0] = 0x3F80
    got = run_gpu(gi.from_bits(h), gi.from_bits(gw), gi.from_bits(uw), mode)
    assert mb.last_variant() in FAST
    ref = oracle.glu_gemv(h, gw, uw, mode)
    d = tol.ulp_distance(got, ref)
    assert d.max() <= 1, (g[d.argmax()], got[0, d.argmax()], ref[0, d.argmax()])
    assert np.mean(d == 0) > 0.999


def test_deterministic_and_row_permutation_bitwise():
    M, N, K = 8, 3000, 2560
    h = gi.normal_bf16((M, K), 1.0, 6, "dp-h").to(DEV)
    g = gi.normal_bf16((N, K), K ** -0.5, 6, "dp-g").to(DEV)
    u = gi.normal_bf16((N, K), K ** -0.5, 6, "dp-u").to(DEV)
    a = mb.glu_gemv(h, g, u, mode="hf")
    b = mb.glu_gemv(h, g, u, mode="hf")
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(0)).to(DEV)
    c = mb.glu_gemv(h, g[perm], u[perm], mode="hf")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a[:, perm].view(torch.int16), c.view(torch.int16))


@pytest.mark.parametrize("policy", [0, 1, 2])
def test_launch_policies_give_identical_results(policy):
    """Serial, programmatic dependent launch and weight prefetch before the
    dependency wait: bitwise the same outputs, also back to back in a graph."""
    M, N, K = 4, 3001, 2560
    h = gi.normal_bf16((M, K), 1.0, 11, "pol-h").to(DEV)
    gs = [gi.normal_bf16((N, K), K ** -0.5, 11, "pol-g", i).to(DEV) for i in range(3)]
    us = [gi.normal_bf16((N, K), K ** -0.5, 11, "pol-u", i).to(DEV) for i in range(3)]
    x = gi.normal_bf16((M, K), 1.0, 11, "pol-x").to(DEV)
    r0 = gi.normal_bf16((M, K), 1.0, 11, "pol-r").to(DEV)
    w = gi.normal_bf16((K,), 0.1, 11, "pol-w").to(DEV)

    def run():
        outs = [mb.glu_gemv(h, gs[i], us[i], mode="hf") for i in range(3)]
        r = r0.clone()
        outs += [mb.add_rmsnorm_glu(x, r, w, 1e-6, gs[i], us[i], mode="fused") for i in range(3)]
        torch.cuda.synchronize()
        return [o.view(torch.int16).cpu() for o in outs] + [r.view(torch.int16).cpu()]

    old = mb.get_launch_policy()
    try:
        mb.set_launch_policy(0)
        ref = run()
        mb.set_launch_policy(policy)
        got = run()
    finally:
        mb.set_launch_policy(old)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


def test_swap_gate_and_up_matches_oracle_swap():
    M, N, K = 2, 777, 1024
    h = gi.normal_bf16((M, K), 1.0, 7, "sw-h")
    g = gi.normal_bf16((N, K), K ** -0.5, 7, "sw-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 7, "sw-u")
    check(h, u, g, "fused", "swapped")


def test_in_place_weight_update_is_seen():
    """No state derived from the weights: an in-place update shows at once."""
    M, N, K = 1, 2000, 2048
    h = gi.normal_bf16((M, K), 1.0, 8, "ip-h")
    g = gi.normal_bf16((N, K), K ** -0.5, 8, "ip-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 8, "ip-u")
    hd, gd, ud = h.to(DEV), g.to(DEV), u.to(DEV)
    mb.glu_gemv(hd, gd, ud, mode="hf")
    g2 = gi.normal_bf16((N, K), K ** -0.5, 9, "ip-g")
    gd.copy_(g2.to(DEV))
    out = mb.glu_gemv(hd, gd, ud, mode="hf")
    torch.cuda.synchronize()
    ref, tau = oracle_glu(h, g2, u, "hf")
    parity(gi.bits(out.cpu()), ref, tau, "after in-place update")


def test_cuda_graph_replay_matches_eager():
    M, N, K = 4, 4000, 2560
    h = gi.normal_bf16((M, K), 1.0, 10, "cg-h").to(DEV)
    g = gi.normal_bf16((N, K), K ** -0.5, 10, "cg-g").to(DEV)
    u = gi.normal_bf16((N, K), K ** -0.5, 10, "cg-u").to(DEV)
    x = gi.normal_bf16((M, K), 1.0, 10, "cg-x").to(DEV)
    r0 = gi.normal_bf16((M, K), 1.0, 10, "cg-r").to(DEV)
    w = gi.normal_bf16((K,), 0.1, 10, "cg-w").to(DEV)
    eager = mb.glu_gemv(h, g, u, mode="fused")
    r_e = r0.clone()
    eager2 = mb.add_rmsnorm_glu(x, r_e, w, 1e-6, g, u, mode="hf")
    out = torch.empty_like(eager)
    out2 = torch.empty_like(eager2)
    r_g = r0.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            mb.glu_gemv(h, g, u, out=out, mode="fused")
            mb.add_rmsnorm_glu(x, r_g, w, 1e-6, g, u, out=out2, mode="hf")
    r_g.copy_(r0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert torch.equal(out2.view(torch.int16), eager2.view(torch.int16))
    assert torch.equal(r_g.view(torch.int16), r_e.view(torch.int16))


# ---------------------------------------------------------------------------
# add_rmsnorm_glu
# ---------------------------------------------------------------------------

def check_norm(x, r, w, g, u, mode, eps=1e-6, what="", variant=None, ws=None):
    rd = r.to(DEV)
    out = mb.add_rmsnorm_glu(x.to(DEV), rd, w.to(DEV), eps, g.to(DEV), u.to(DEV), mode=mode, workspace=ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert int(ws.sum()) == 0, "workspace not returned to zero"
    if variant == 1:
        assert mb.last_variant() in FAST
    elif variant is not None:
        assert mb.last_variant() == variant
    ref, res, hn = oracle.add_rmsnorm_glu(gi.bits(x), gi.bits(r), gi.bits(w), eps, gi.bits(g), gi.bits(u), mode)
    assert np.array_equal(gi.bits(rd.cpu()), res), f"residual {what}"
    # the kernels' h is the correctly rounded one (the oracle's hn), so the
    # GEMV part carries only its own fp32 accumulation
    _, diag = oracle.glu_gemv(hn, gi.bits(g), gi.bits(u), mode, diagnostics=True)
    K = x.shape[1]
    return parity(gi.bits(out.cpu()), ref, (tol.conditioning_floor(diag, K, mode), diag, K, mode), what)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 13, 16])
def test_add_rmsnorm_glu_small(M):
    N, K = 1500, 2048
    x = gi.normal_bf16((M, K), 1.0, M, "an-x")
    r = gi.normal_bf16((M, K), 1.0, M, "an-r")
    w = gi.normal_bf16((K,), 0.1, M, "an-w")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "an-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "an-u")
    for mode in ("hf", "fused"):
        check_norm(x, r, w, g, u, mode, what=f"M={M} {mode}", variant=1)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 13, 16])
@pytest.mark.parametrize("mode", ["hf", "fused"])
def test_add_rmsnorm_glu_single_kernel(M, mode):
    """The workspace entry point: one kernel, residual written back by the
    last CTA, the workspace left at zero."""
    N, K = 1500, 2048
    x = gi.normal_bf16((M, K), 1.0, M, "ws-x")
    r = gi.normal_bf16((M, K), 1.0, M, "ws-r")
    w = gi.normal_bf16((K,), 0.1, M, "ws-w")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "ws-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "ws-u")
    ws = mb.new_workspace(DEV)
    check_norm(x, r, w, g, u, mode, what=f"ws M={M} {mode}", variant=1, ws=ws)


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("single", [False, True])
def test_add_rmsnorm_glu_strided_weights_and_out(M, single):
    """Weights and out as row-strided views (add_rmsnorm_glu_strided): the same
    bytes reach the same arithmetic, so the bits equal the contiguous call's;
    a stride that is not a multiple of 8 elements runs the generic kernel and
    is checked against the oracle."""
    N, K = 1500, 2048
    x = gi.normal_bf16((M, K), 1.0, M, "st-x").to(DEV)
    r = gi.normal_bf16((M, K), 1.0, M, "st-r")
    w = gi.normal_bf16((K,), 0.1, M, "st-w").to(DEV)
    g = gi.normal_bf16((N, K), K ** -0.5, M, "st-g").to(DEV)
    u = gi.normal_bf16((N, K), K ** -0.5, M, "st-u").to(DEV)
    ws = (lambda: mb.new_workspace(DEV)) if single else (lambda: None)
    r_ref = r.to(DEV)
    ref = mb.add_rmsnorm_glu(x, r_ref, w, 1e-6, g, u, mode="hf", workspace=ws())
    variant = mb.last_variant()
    gw = torch.zeros((N, K + 64), dtype=torch.bfloat16, device=DEV)
    uw = torch.zeros((N, K + 8), dtype=torch.bfloat16, device=DEV)
    gw[:, :K], uw[:, :K] = g, u
    out_w = torch.full((M, N + 16), float("nan"), dtype=torch.bfloat16, device=DEV)
    r_st = r.to(DEV)
    mb.add_rmsnorm_glu(x, r_st, w, 1e-6, gw[:, :K], uw[:, :K], out=out_w[:, :N], mode="hf", workspace=ws())
    torch.cuda.synchronize()
    assert mb.last_variant() == variant
    assert torch.equal(r_st.view(torch.int16), r_ref.view(torch.int16))
    assert torch.equal(out_w[:, :N].view(torch.int16), ref.view(torch.int16))
    assert torch.isnan(out_w[:, N:].float()).all()
    # an odd stride: the generic kernel, against the oracle
    go = torch.zeros((N, K + 3), dtype=torch.bfloat16, device=DEV)
    go[:, :K] = g
    r_odd = r.to(DEV)
    out_odd = mb.add_rmsnorm_glu(x, r_odd, w, 1e-6, go[:, :K], u, mode="hf", workspace=ws())
    torch.cuda.synchronize()
    assert mb.last_variant() == 2
    assert torch.equal(r_odd.view(torch.int16), r_ref.view(torch.int16))
    ref_o, _, hn = oracle.add_rmsnorm_glu(gi.bits(x.cpu()), gi.bits(r), gi.bits(w.cpu()), 1e-6, gi.bits(g.cpu()),
                                          gi.bits(u.cpu()), "hf")
    _, diag = oracle.glu_gemv(hn, gi.bits(g.cpu()), gi.bits(u.cpu()), "hf", diagnostics=True)
    tol.assert_parity(gi.bits(out_odd.cpu()), ref_o, tol.conditioning_floor(diag, K, "hf"), "odd stride",
                      diag=diag, K=K, mode="hf")


def test_add_rmsnorm_glu_single_kernel_back_to_back_and_graph():
    """Consecutive calls on one stream share a workspace (also replayed in a
    CUDA graph), each reading the residual the previous one wrote."""
    M, N, K = 4, 2000, 2560
    x = [gi.normal_bf16((M, K), 1.0, i, "bb-x").to(DEV) for i in range(3)]
    r0 = gi.normal_bf16((M, K), 1.0, 0, "bb-r").to(DEV)
    w = gi.normal_bf16((K,), 0.1, 0, "bb-w").to(DEV)
    gs = [gi.normal_bf16((N, K), K ** -0.5, i, "bb-g").to(DEV) for i in range(3)]
    us = [gi.normal_bf16((N, K), K ** -0.5, i, "bb-u").to(DEV) for i in range(3)]
    ws = mb.new_workspace(DEV)

    def chain(res, use_ws):
        return [mb.add_rmsnorm_glu(x[i], res, w, 1e-6, gs[i], us[i], mode="hf", workspace=ws if use_ws else None)
                for i in range(3)]

    r_ref = r0.clone()
    ref = chain(r_ref, False)
    r_ws = r0.clone()
    got = chain(r_ws, True)
    torch.cuda.synchronize()
    assert int(ws.sum()) == 0
    assert torch.equal(r_ws.view(torch.int16), r_ref.view(torch.int16))
    for a, b in zip(ref, got):
        d = tol.ulp_distance(gi.bits(a.cpu()), gi.bits(b.cpu()))
        assert np.mean(d == 0) > 0.999 and d.max() <= 4
    # the same chain captured once and replayed twice
    r_g = r0.clone()
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for i in range(3):
                mb.add_rmsnorm_glu(x[i], r_g, w, 1e-6, gs[i], us[i], out=outs[i], mode="hf", workspace=ws)
    for _ in range(2):
        r_g.copy_(r0)
        graph.replay()
    torch.cuda.synchronize()
    assert int(ws.sum()) == 0
    assert torch.equal(r_g.view(torch.int16), r_ref.view(torch.int16))
    for a, b in zip(got, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_add_rmsnorm_glu_single_kernel_falls_back():
    """K % 8 != 0: the two-kernel path runs and the workspace is not touched."""
    M, N, K = 2, 300, 1004
    x = gi.normal_bf16((M, K), 1.0, 5, "fb-x")
    r = gi.normal_bf16((M, K), 1.0, 5, "fb-r")
    w = gi.normal_bf16((K,), 0.1, 5, "fb-w")
    g = gi.normal_bf16((N, K), K ** -0.5, 5, "fb-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 5, "fb-u")
    ws = mb.new_workspace(DEV)
    ws[17] = 5                     # a marker the fallback must leave alone
    rd = r.to(DEV)
    out = mb.add_rmsnorm_glu(x.to(DEV), rd, w.to(DEV), 1e-6, g.to(DEV), u.to(DEV), mode="hf", workspace=ws)
    torch.cuda.synchronize()
    assert mb.last_variant() == 2 and int(ws[17]) == 5 and int(ws.sum()) == 5
    ref, res, _ = oracle.add_rmsnorm_glu(gi.bits(x), gi.bits(r), gi.bits(w), 1e-6, gi.bits(g), gi.bits(u), "hf")
    assert np.array_equal(gi.bits(rd.cpu()), res)


def test_add_rmsnorm_glu_generic_and_edge_cases():
    M, N, K = 3, 400, 1000 + 4   # K % 8 != 0 -> generic kernel with the norm in smem
    x = gi.normal_bf16((M, K), 1.0, 1, "ae-x")
    r = gi.normal_bf16((M, K), 1.0, 1, "ae-r")
    w = gi.normal_bf16((K,), 0.1, 1, "ae-w")
    g = gi.normal_bf16((N, K), K ** -0.5, 1, "ae-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 1, "ae-u")
    check_norm(x, r, w, g, u, "hf", what="generic", variant=2)
    # x = -residual: s = 0, h = 0, out = +0
    K2 = 512
    x2 = gi.normal_bf16((2, K2), 1.0, 2, "ae-x2")
    g2 = gi.normal_bf16((N, K2), 0.05, 2, "ae-g2")
    rd = (-x2).to(DEV)
    out = mb.add_rmsnorm_glu(x2.to(DEV), rd, torch.zeros(K2, dtype=torch.bfloat16, device=DEV), 1e-6,
                             g2.to(DEV), g2.to(DEV), mode="hf")
    torch.cuda.synchronize()
    assert (gi.bits(rd.cpu()) & 0x7FFF == 0).all()
    assert (gi.bits(out.cpu()) & 0x7FFF == 0).all()
    # residual == x is allowed: s = bf16(2x)
    xd = x2.to(DEV)
    mb.add_rmsnorm_glu(xd, xd, torch.zeros(K2, dtype=torch.bfloat16, device=DEV), 1e-6, g2.to(DEV),
                       g2.to(DEV), mode="hf")
    torch.cuda.synchronize()
    assert torch.equal(xd.cpu(), (x2.float() * 2).to(torch.bfloat16))


# ---------------------------------------------------------------------------
# every workload at full size, one sampled layer
# ---------------------------------------------------------------------------

@functools.lru_cache(maxsize=1)
def _layer(name, layer):
    return gi.layer_weights(gi.WORKLOADS[name], layer)


# every workload at every batch in BOTH modes (the bar holds for each mode,
# whichever mode the workload is timed in)
FULL_CASES = [(w.name, M, mode) for w in gi.WORKLOADS.values() if w.op in ("glu_gemv", "add_rmsnorm_glu")
              for M in w.Ms for mode in ("fused", "hf")]


@pytest.mark.parametrize("name,M,mode", FULL_CASES)
def test_full_size_workload(name, M, mode):
    w = gi.WORKLOADS[name]
    layer = w.layers - 1          # the last layer of the cycled set
    g, u = _layer(name, layer)
    if w.op == "glu_gemv":
        h = gi.hidden(w, M)
        st = check(h, g, u, mode, f"{name} M={M} {mode}", variant=1 if M <= mb.BLOCK_M else 9)
    else:
        x, r, nw = gi.norm_inputs(w, M)
        st = check_norm(x, r, nw, g, u, mode, eps=w.eps, what=f"{name} M={M}", variant=1)
        check_norm(x, r, nw, g, u, mode, eps=w.eps, what=f"{name} M={M} single kernel", variant=1,
                   ws=mb.new_workspace(DEV))
    assert st["exact_frac"] > 0.9


def test_device_error_word_is_clear():
    assert mb.read_device_error() == 0
