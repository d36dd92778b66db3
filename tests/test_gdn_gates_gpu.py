"""GPU parity of gdn_gates (the gated-delta-net decay and write gates)
against the fp64 oracle, through the C ABI.

g is fp32: the kernel's fp32 softplus, exp and product sit a few fp32 ulps
from the oracle's exact value on the same binary32 x = a + dt_bias, so the bar
for g is |dg| <= 2e-6 |g| + 1e-36 (the absolute term covers x below ~ -87,
where e^x is subnormal in fp32).  beta is bf16: the GEMV's bar (tolerance.py).
"""
import numpy as np
import pytest
import torch

import glu_inputs as gi
import oracle
import tolerance as tol

pytestmark = pytest.mark.gpu

mb = pytest.importorskip("memory_bound_glu_gb300")
DEV = torch.device("cuda:0")
GDN_GATES = 6   # mbglu_last_variant() after a gdn_gates launch


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def check(a, b, A_log, dt_bias, what=""):
    g, beta = mb.gdn_gates(a, b, A_log, dt_bias)
    torch.cuda.synchronize()
    assert mb.last_variant() == GDN_GATES
    g_ref, beta_ref = oracle.gdn_gates(gi.bits(a.cpu()), gi.bits(b.cpu()), A_log.cpu().numpy(), dt_bias.cpu().numpy())
    gd = g.double().cpu().numpy()
    err = np.abs(gd - g_ref) - (2e-6 * np.abs(g_ref) + 1e-36)
    assert np.isfinite(gd).all() and err.max() <= 0, (what, np.unravel_index(err.argmax(), err.shape))
    tol.assert_parity(gi.bits(beta.cpu()), beta_ref, what=f"beta {what}")
    return g, beta


@pytest.mark.parametrize("T,H", [(1, 32), (7, 48), (300, 16), (1000, 3)])
def test_gdn_gates_shapes_and_strided_inputs(T, H):
    """a and b as column blocks of one [T, 2H + 8] projection output."""
    proj = gi.normal_bf16((T, 2 * H + 8), 3.0, T, "gg-proj", H).to(DEV)
    a, b = proj[:, :H], proj[:, H:2 * H]
    A_log = gi.normal_bf16((H,), 1.0, T, "gg-A", H).float().to(DEV)
    dt_bias = gi.normal_bf16((H,), 1.0, T, "gg-dt", H).float().to(DEV)
    check(a, b, A_log, dt_bias, f"T={T} H={H}")


def test_gdn_gates_every_bf16_input():
    """a and b run over every finite bf16 (A_log = 0, dt_bias = 0: g = -softplus(a)),
    including both tails where the naive softplus overflows or underflows."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = pats[(pats & 0x7FFF) < 0x7F80]
    H = 64
    T = v.size // H
    x = gi.from_bits(v[:T * H].reshape(T, H)).to(DEV)
    zeros = torch.zeros(H, dtype=torch.float32, device=DEV)
    check(x, x, zeros, zeros, "exhaustive")


def test_gdn_gates_extremes_and_noop():
    big = torch.tensor([[3.3895e38, -3.3895e38, 1000.0, -1000.0]], dtype=torch.bfloat16, device=DEV)
    z = torch.zeros(4, dtype=torch.float32, device=DEV)
    g, beta = check(big, big, z, z, "extremes")
    assert torch.isfinite(g).all() and g[0, 1].item() == 0.0 and beta[0, 0].item() == 1.0 and beta[0, 1].item() == 0.0
    e = torch.zeros((0, 8), dtype=torch.bfloat16, device=DEV)
    g0, b0 = mb.gdn_gates(e, e, torch.zeros(8, device=DEV), torch.zeros(8, device=DEV))
    assert g0.shape == (0, 8) and mb.last_variant() == 0


def test_gdn_gates_paths_agree_bitwise():
    """The three layouts -- 16-byte chunks of 8 heads, the same chunks element
    by element (rows offset by one element), and one element per thread (more
    heads than the per-CTA table holds) -- run the same arithmetic per
    element: identical bits, and the last against the oracle."""
    T, H = 257, 40
    a = gi.normal_bf16((T, H), 3.0, 1, "gp-a").to(DEV)
    b = gi.normal_bf16((T, H), 3.0, 1, "gp-b").to(DEV)
    A_log = gi.normal_bf16((H,), 1.0, 1, "gp-A").float().to(DEV)
    dt = gi.normal_bf16((H,), 1.0, 1, "gp-dt").float().to(DEV)
    g_vec, beta_vec = mb.gdn_gates(a, b, A_log, dt)
    buf = torch.zeros((2, T * H + 1), dtype=torch.bfloat16, device=DEV)
    buf[0, 1:], buf[1, 1:] = a.reshape(-1), b.reshape(-1)
    a1, b1 = buf[0, 1:].view(T, H), buf[1, 1:].view(T, H)          # 2-byte aligned rows only
    g_el, beta_el = mb.gdn_gates(a1, b1, A_log, dt)
    torch.cuda.synchronize()
    assert torch.equal(g_vec.view(torch.int32), g_el.view(torch.int32))
    assert torch.equal(beta_vec.view(torch.int16), beta_el.view(torch.int16))
    Hw = 4104                                                        # above the per-CTA table: one element per thread
    aw = gi.normal_bf16((3, Hw), 3.0, 2, "gp-aw").to(DEV)
    Aw = gi.normal_bf16((Hw,), 1.0, 2, "gp-Aw").float().to(DEV)
    dw = gi.normal_bf16((Hw,), 1.0, 2, "gp-dw").float().to(DEV)
    check(aw, aw, Aw, dw, "H=4104")
