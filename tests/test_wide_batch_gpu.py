"""GPU parity of batches above 16 rows (M = 17..64, decode at batch 32 and
64): glu_gemv runs them in one pass on the tcgen05 kernel where its operands
allow tensor copies, otherwise -- and the add_rmsnorm_glu entry points
always -- as row blocks of 16, the remainder last, each block one call of
the M <= 16 kernels.

Checked against the fp64 oracle with the bar every other batch size meets
(tolerance.py), with the tensor-core accumulation bound (blocks of 3 or more
rows run on the tensor cores); each block's bits are also compared with a
call on the same rows alone, since a row's result does not depend on the
rows beside it.  Full size: the K = 2560, N = 9728 layer at M = 64, on a
sample of output features the oracle computes one by one.
"""
import ctypes

import numpy as np
import pytest
import torch

import glu_inputs as gi
import oracle
import tolerance as tol

pytestmark = pytest.mark.gpu

mb = pytest.importorskip("memory_bound_glu_gb300")
DEV = torch.device("cuda:0")
ROW_BLOCKS = 7   # mbglu_last_variant(): a batch above 16 rows as row blocks
TCGEN05 = 9      # mbglu_last_variant(): the batch in one pass on the tcgen05 kernel


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _gemv_parity(got_bits, h, g, u, mode, what):
    ref, diag = oracle.glu_gemv(gi.bits(h), gi.bits(g), gi.bits(u), mode, diagnostics=True)
    diag["acc"] = "mma"       # the looser of the two kernels' accumulation bounds
    K = h.shape[1]
    return tol.assert_parity(got_bits, ref, tol.conditioning_floor(diag, K, mode), what, diag=diag, K=K, mode=mode)


def test_tcgen05_one_tile_one_chunk():
    """The smallest case first: one 128-row tile, one 64-wide K chunk, batch
    17 padded to 32 -- one stage, eight MMAs, no K split.  Distinct values
    per row and column, so a transposed or misplaced operand cannot pass."""
    M, N, K = 17, 128, 64
    h = gi.normal_bf16((M, K), 1.0, 1, "tc1-h")
    g = gi.normal_bf16((N, K), K ** -0.5, 1, "tc1-g")
    u = gi.normal_bf16((N, K), K ** -0.5, 1, "tc1-u")
    out = mb.glu_gemv(h.to(DEV), g.to(DEV), u.to(DEV), mode="fused")
    torch.cuda.synchronize()
    assert mb.last_variant() == TCGEN05
    assert mb.read_device_error() == 0
    _gemv_parity(gi.bits(out.cpu()), h, g, u, "fused", "one tile")


@pytest.mark.parametrize("m0,k0", [(0, 0), (5, 17), (16, 40), (3, 63)])
def test_tcgen05_one_hot_mapping(m0, k0):
    """One tile, one chunk, structured: h = e(m0, k0) (a single 1), gate_w[n][k0]
    = distinct values v_n, up_w[n][k0] = 1, zeros elsewhere.  Then g[m][n] =
    v_n for m = m0 and 0 otherwise, u likewise 1 or 0, and out[m0][n] =
    SiLU(v_n), every other output +0.  On a mismatch the message says where
    the values landed (a transposed, shifted or swizzled operand shows as a
    pattern)."""
    M, N, K = 17, 128, 64
    h = torch.zeros((M, K), dtype=torch.bfloat16)
    h[m0, k0] = 1.0
    v = (torch.arange(N, dtype=torch.float32) / 32.0 - 2.0).to(torch.bfloat16)   # -2 .. 1.97, exact in bf16
    g = torch.zeros((N, K), dtype=torch.bfloat16)
    g[:, k0] = v
    u = torch.zeros((N, K), dtype=torch.bfloat16)
    u[:, k0] = 1.0
    out = mb.glu_gemv(h.to(DEV), g.to(DEV), u.to(DEV), mode="fused").float().cpu()
    assert mb.last_variant() == TCGEN05
    assert mb.read_device_error() == 0
    ref = oracle.glu_gemv(gi.bits(h), gi.bits(g), gi.bits(u), "fused")
    got = gi.bits(out.to(torch.bfloat16))
    bad = np.argwhere(got != ref)
    nz = np.argwhere(out.numpy() != 0)
    assert bad.size == 0, (f"{len(bad)} outputs differ; first {bad[:8].tolist()}; nonzero outputs at rows "
                           f"{sorted(set(nz[:, 0].tolist()))[:8]}, {len(nz)} in all (expected row {m0}, {N})")


@pytest.mark.parametrize("mode", ["fused", "hf"])
@pytest.mark.parametrize("M", [17, 18, 24, 32, 33, 40, 48, 63, 64])
@pytest.mark.parametrize("path", ["tcgen05", "row blocks"])
def test_glu_gemv_batch_17_to_64(M, mode, path):
    """Ragged N (a partial last 128-row tile; partial 8-row groups) and a K
    that ends inside a 64-wide chunk.  Aligned operands take the tcgen05
    kernel in one pass; h with a row stride that is not a multiple of 8
    elements takes the row blocks (remainders of 1 and 2 rows on the
    CUDA-core kernel, the others on the mma.sync kernel)."""
    N, K = 1337, 1288
    h = gi.normal_bf16((M, K), 1.0, M, "wb-h")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "wb-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "wb-u")
    hd = h.to(DEV)
    if path == "row blocks":
        hw = torch.zeros((M, K + 1), dtype=torch.bfloat16, device=DEV)
        hw[:, :K] = hd
        hd = hw[:, :K]
    out = mb.glu_gemv(hd, g.to(DEV), u.to(DEV), mode=mode)
    torch.cuda.synchronize()
    assert mb.last_variant() == (TCGEN05 if path == "tcgen05" else ROW_BLOCKS)
    _gemv_parity(gi.bits(out.cpu()), h, g, u, mode, f"M={M} {mode} {path}")
    assert mb.read_device_error() == 0


def test_row_blocks_equal_calls_on_each_block():
    """M = 50: blocks of 16, 16, 16 and 2 rows, bit for bit the calls on those
    rows alone."""
    M, N, K = 50, 2001, 2560
    hw = torch.zeros((M, K + 3), dtype=torch.bfloat16, device=DEV)   # an odd row stride: row blocks
    hw[:, :K] = gi.normal_bf16((M, K), 1.0, 3, "wbe-h").to(DEV)
    h = hw[:, :K]
    g = gi.normal_bf16((N, K), K ** -0.5, 3, "wbe-g").to(DEV)
    u = gi.normal_bf16((N, K), K ** -0.5, 3, "wbe-u").to(DEV)
    whole = mb.glu_gemv(h, g, u, mode="hf")
    assert mb.last_variant() == ROW_BLOCKS
    parts = [mb.glu_gemv(h[m0:m0 + 16], g, u, mode="hf") for m0 in range(0, M, 16)]
    torch.cuda.synchronize()
    assert torch.equal(whole.view(torch.int16), torch.cat(parts).view(torch.int16))
    assert mb.read_device_error() == 0


def test_row_blocks_strided_operands_and_guard_band():
    """h, the weights and out as views into wider buffers: the block offsets
    follow the row strides, and nothing outside out is written."""
    M, N, K = 37, 999, 1536
    hb = gi.normal_bf16((M, K + 40), 1.0, 4, "wbs-h")
    gb = gi.normal_bf16((N, K + 64), K ** -0.5, 4, "wbs-g")
    ub = gi.normal_bf16((N, K + 16), K ** -0.5, 4, "wbs-u")
    h, g, u = hb[:, 8:8 + K], gb[:, :K], ub[:, 16:16 + K]
    buf = torch.full((M + 2, N + 48), -7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[1:1 + M, 24:24 + N]
    mb.glu_gemv(hb.to(DEV)[:, 8:8 + K], gb.to(DEV)[:, :K], ub.to(DEV)[:, 16:16 + K], out=out, mode="hf")
    torch.cuda.synchronize()
    assert mb.last_variant() == TCGEN05   # every row stride a multiple of 8 elements
    mask = torch.ones(buf.shape, dtype=torch.bool)
    mask[1:1 + M, 24:24 + N] = False
    assert (buf.float().cpu()[mask] == -7.0).all(), "wrote outside out"
    _gemv_parity(gi.bits(out.cpu()), h.contiguous(), g.contiguous(), u.contiguous(), "hf", "strided")


def test_row_blocks_degenerate_sizes():
    K, N = 64, 10
    w = gi.normal_bf16((N, K), 0.1, 5, "wbd-w").to(DEV)
    o = torch.full((40, N), 3.0, dtype=torch.bfloat16, device=DEV)
    mb.glu_gemv(torch.zeros((40, 0), dtype=torch.bfloat16, device=DEV), w[:, :0], w[:, :0], out=o)   # K == 0
    torch.cuda.synchronize()
    assert mb.last_variant() == ROW_BLOCKS
    assert (gi.bits(o.cpu()) == 0).all()
    o = torch.empty((40, 0), dtype=torch.bfloat16, device=DEV)
    mb.glu_gemv(torch.zeros((40, K), dtype=torch.bfloat16, device=DEV), w[:0], w[:0], out=o)          # N == 0
    assert mb.last_variant() == 0
    with pytest.raises(mb.MbgluError):
        mb.glu_gemv(torch.zeros((mb.MAX_M + 1, K), dtype=torch.bfloat16, device=DEV), w, w)


def _noalloc(x, residual, norm_w, eps, gate_w, up_w, out, mode):
    M, K = x.shape
    st = mb.lib().add_rmsnorm_glu_noalloc(x.data_ptr(), residual.data_ptr(), norm_w.data_ptr(), float(eps),
                                          gate_w.data_ptr(), up_w.data_ptr(), out.data_ptr(), M, gate_w.shape[0], K,
                                          mb.MODE_HF if mode == "hf" else mb.MODE_FUSED,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise mb.MbgluError(st, "add_rmsnorm_glu_noalloc")


@pytest.mark.parametrize("M", [17, 40, 64])
@pytest.mark.parametrize("path", ["two kernels", "workspace", "noalloc", "strided"])
def test_add_rmsnorm_glu_row_blocks(M, path):
    """The residual update is bitwise the oracle's; out is within the bar.  The
    blocks of one call share the workspace (and the library's scratch), which
    each completed block leaves zero."""
    N, K, mode = 1500, 2048, ("hf" if M % 2 == 0 else "fused")
    x = gi.normal_bf16((M, K), 1.0, M, "wbn-x")
    r = gi.normal_bf16((M, K), 1.0, M, "wbn-r")
    w = gi.normal_bf16((K,), 0.1, M, "wbn-w")
    g = gi.normal_bf16((N, K), K ** -0.5, M, "wbn-g")
    u = gi.normal_bf16((N, K), K ** -0.5, M, "wbn-u")
    xd, rd, wd, gd, ud = (t.to(DEV) for t in (x, r, w, g, u))
    ws = None
    if path == "two kernels":
        out = mb.add_rmsnorm_glu(xd, rd, wd, 1e-6, gd, ud, mode=mode)
    elif path == "workspace":
        ws = mb.new_workspace(DEV)
        out = mb.add_rmsnorm_glu(xd, rd, wd, 1e-6, gd, ud, mode=mode, workspace=ws)
    elif path == "noalloc":
        out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        _noalloc(xd, rd, wd, 1e-6, gd, ud, out, mode)
    else:
        gw = torch.zeros((N, K + 64), dtype=torch.bfloat16, device=DEV)
        uw = torch.zeros((N, K + 8), dtype=torch.bfloat16, device=DEV)
        gw[:, :K], uw[:, :K] = gd, ud
        ob = torch.full((M, N + 16), float("nan"), dtype=torch.bfloat16, device=DEV)
        ws = mb.new_workspace(DEV)
        out = ob[:, :N]
        mb.add_rmsnorm_glu(xd, rd, wd, 1e-6, gw[:, :K], uw[:, :K], out=out, mode=mode, workspace=ws)
    torch.cuda.synchronize()
    assert mb.last_variant() == ROW_BLOCKS
    if ws is not None:
        assert int(ws.sum()) == 0, "workspace not returned to zero"
    if path == "strided":
        assert torch.isnan(ob[:, N:].float()).all(), "wrote outside out"
    ref, res, hn = oracle.add_rmsnorm_glu(gi.bits(x), gi.bits(r), gi.bits(w), 1e-6, gi.bits(g), gi.bits(u), mode)
    assert np.array_equal(gi.bits(rd.cpu()), res), "residual"
    _, diag = oracle.glu_gemv(hn, gi.bits(g), gi.bits(u), mode, diagnostics=True)
    diag["acc"] = "mma"
    tol.assert_parity(gi.bits(out.cpu()), ref, tol.conditioning_floor(diag, K, mode), f"{path} M={M}",
                      diag=diag, K=K, mode=mode)
    assert mb.read_device_error() == 0


def test_full_size_batch_64():
    """The K = 2560, N = 9728 layer (the headline shape) at batch 64, both
    modes, on the tcgen05 kernel (76 tiles, K split over CTA pairs): every
    output on the GPU, 1024 sampled features against the oracle."""
    w = gi.WORKLOADS["gemv_k2560_n9728"]
    g, u = gi.layer_weights(w, w.layers - 1)
    h = gi.hidden(w, 64)
    feats = np.sort(np.random.default_rng(64).choice(w.N, 1024, replace=False))
    gd, ud, hd = g.to(DEV), u.to(DEV), h.to(DEV)
    for mode in ("hf", "fused"):
        out = mb.glu_gemv(hd, gd, ud, mode=mode)
        torch.cuda.synchronize()
        assert mb.last_variant() == TCGEN05
        st = _gemv_parity(gi.bits(out.cpu())[:, feats], h, g[feats], u[feats], mode, f"M=64 {mode}, sampled")
        assert st["exact_frac"] > 0.9
    assert mb.read_device_error() == 0
