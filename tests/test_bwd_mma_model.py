"""CPU model of the backward's second step on the tensor cores
(glu_bwd_mma_kernel in csrc/glu_backward.cuh): its plan (plan_bwd_mma in
csrc/mbglu_api.cu, restated here) and every shared-memory address, fragment
and store of the kernel, replayed lane by lane with the PTX ISA's fragment
layouts for ldmatrix (with and without .trans) and mma.sync m16n8k16 /
m16n8k8 .row.col, and with the 128-byte swizzle of a tensor copy.

Values travel in float64 and are never rounded, so the replay must give the
plain sums
    grad_W[n][k]     = sum_m dG[m][n] h[m][k]
    part[s][m][k]    = sum_{n in share s} dG[m][n] Wg[n][k] + dU[m][n] Wu[n][k]
to float64 rounding, because the three bf16 terms hi + mid + lo hold each
fp32 dG, dU exactly (checked here too); a wrong index, swizzle, fragment
mapping or row mask anywhere changes them.  The replay also checks that
every gradient element and every grad_h partial is stored exactly once
(the weight gradients as 16-byte pieces on 16-byte boundaries),
that every shared-memory access stays inside its own region, and that each
tensor copy lands on a 1024-byte boundary with x a multiple of 8 elements."""
import numpy as np
import pytest

from frag_model import C4, G4, LANE, MI, RI, Smem, bf16_rn, mma

SMEM_OPTIN = 232448        # GB300: max dynamic shared memory per block (opt-in)
BOX = 16 * 128             # one 64-column x 16-row box of bf16, bytes
MAX_PARTS = 256

def bwd_mma_warps(NB):
    return 8 if NB >= 4 else 12


def plan(M, N, K, sms, NB=2, warps=0):
    if M > 8 or K % 8:
        return None
    wtot = -(-K // (64 * NB))
    wmax = warps if warps > 0 else bwd_mma_warps(NB)
    wmin = warps if warps > 0 else 1
    stage = 2 * NB * BOX
    best, best_score = None, -1
    for w in range(wmax, wmin - 1, -1):
        cg = -(-wtot // w)
        W = -(-wtot // cg)
        if W != w:
            continue
        shares = max(1, min((N + 15) // 16, sms // cg, MAX_PARTS))
        rows_cta = -(-N // shares)
        rows_pad = -(-rows_cta // 16) * 16
        off_mn = 512
        off_nm = off_mn + 96 * (rows_pad + 8)
        off_ring = (off_nm + 96 * rows_pad + 1023) & ~1023
        room = SMEM_OPTIN - 1024 - off_ring
        if room <= 0:
            continue
        S = min(4, room // (W * stage), 64 // W)
        if S < 2:
            continue
        score = 16 * W + S
        if score > best_score:
            best_score = score
            best = dict(NB=NB, cg=cg, warps=W, shares=shares, rows_cta=rows_cta, rows_pad=rows_pad, S=S,
                        off_mn=off_mn, off_nm=off_nm, off_ring=off_ring, stage=stage,
                        smem=off_ring + W * S * stage + 1024)
    return best


def split3(x):
    """x = hi + mid + lo in bf16 terms, each difference taken in fp32."""
    x = x.astype(np.float32)
    hi = bf16_rn(x)
    r = (x - hi).astype(np.float32)
    mid = bf16_rn(r)
    lo = bf16_rn((r - mid).astype(np.float32))
    return [t.astype(np.float64) for t in (hi, mid, lo)]


def replay(M, N, K, sms, NB=2, warps=0, seed=0):
    p = plan(M, N, K, sms, NB, warps)
    assert p is not None
    W, S, cg, G = p["warps"], p["S"], p["cg"], p["shares"]
    rp, rs = p["rows_pad"], p["rows_pad"] + 8
    stage, kmat = p["stage"], NB * BOX
    assert p["smem"] <= SMEM_OPTIN and W * S <= 64 and W <= bwd_mma_warps(NB)
    assert p["off_nm"] >= p["off_mn"] + 96 * rs
    assert p["off_ring"] >= p["off_nm"] + 96 * rp and p["off_ring"] % 1024 == 0 and stage % 1024 == 0
    rng = np.random.default_rng(seed)
    q = lambda *shape: bf16_rn(rng.standard_normal(shape).astype(np.float32)).astype(np.float64)
    h, Wg, Wu = q(M, K), q(N, K), q(N, K)
    dG = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    dU = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    tg, tu = split3(dG), split3(dU)
    assert np.array_equal(tg[0] + tg[1] + tg[2], dG.astype(np.float64))
    assert np.array_equal(tu[0] + tu[1] + tu[2], dU.astype(np.float64))

    grad_g = np.full((N, K), np.nan)
    grad_u = np.full((N, K), np.nan)
    n_g = np.zeros((N, K), int)
    n_u = np.zeros((N, K), int)
    part = np.full((G, M, K), np.nan)
    n_part = np.zeros((G, M, K), int)
    avail = p["smem"] - 1024            # what lies past the aligned base in the worst case
    R_MN = (p["off_mn"], p["off_mn"] + 96 * rs)
    R_NM = (p["off_nm"], p["off_nm"] + 96 * rp)

    for bid in range(G * cg):
        share, cgrp = divmod(bid, cg)
        n0, n1 = N * share // G, N * (share + 1) // G
        rows = n1 - n0
        nblk = -(-rows // 16)
        assert rows <= p["rows_cta"] <= rp
        mem = Smem(avail)
        # dG, dU staged as three bf16 terms in both layouts, zero past the share and M
        for m in range(8):
            for r in range(rp):
                ok = m < M and r < rows
                for mat, terms in ((0, tg), (1, tu)):
                    for e in range(3):
                        v = terms[e][m, n0 + r] if ok else 0.0
                        mem.v[p["off_mn"] // 2 + ((mat * 3 + e) * 8 + m) * rs + r] = v   # [matrix][term][8][rs]
                        mem.v[p["off_nm"] // 2 + (mat * rp + r) * 24 + 8 * e + m] = v    # [matrix][rp][24]
        for warp in range(W):
            x0 = (cgrp * W + warp) * 64 * NB
            if x0 >= K:
                continue
            ring = p["off_ring"] + warp * S * stage
            R_RING = (ring, ring + S * stage)
            assert ring + S * stage <= avail

            def fill(j):
                y = n0 + 16 * (nblk - 1 - j)
                st = j % S
                for mat, Wm in ((0, Wg), (1, Wu)):
                    for i in range(NB):
                        dst = ring + st * stage + mat * kmat + i * BOX
                        x = x0 + 64 * i
                        assert dst % 1024 == 0 and x % 8 == 0 and 0 <= y < N
                        for r in range(16):
                            for c in range(64):
                                v = Wm[y + r, x + c] if (y + r < N and x + c < K) else 0.0
                                off = dst + r * 128 + (((c >> 3) ^ (r & 7)) << 4) + (c & 7) * 2
                                assert R_RING[0] <= off < R_RING[1]
                                mem.v[off // 2] = v

            # h fragments: (h[2c][k], h[2c+1][k]), k the weight column of MMA
            # column g in tile t = 4p + t'
            hb = np.zeros((8 * NB, 32, 2))
            for t in range(8 * NB):
                k = x0 + 32 * (t >> 2) + 8 * (G4 >> 1) + 2 * (t & 3) + (G4 & 1)
                for e in range(2):
                    m = 2 * C4 + e
                    ok = (k < K) & (m < M)
                    hb[t, :, e] = np.where(ok, h[np.minimum(m, M - 1), np.minimum(k, K - 1)], 0.0)
            for j in range(min(S, nblk)):
                fill(j)
            acc = np.zeros((4 * NB, 32, 4))
            for j in range(nblk):
                st = j % S
                nb0 = 16 * (nblk - 1 - j)
                nr = min(16, rows - nb0)
                sg = ring + st * stage
                su = sg + kmat
                off = (((MI >> 1) * 8 + RI) * rs + nb0 + 8 * (MI & 1)) * 2
                off8 = ((16 + RI) * rs + nb0 + 8 * (MI & 1)) * 2
                bg = mem.ldsm(p["off_mn"] + off, R_MN)
                bg8 = mem.ldsm(p["off_mn"] + off8, R_MN, x=2)
                bu = mem.ldsm(p["off_mn"] + 48 * rs + off, R_MN)
                bu8 = mem.ldsm(p["off_mn"] + 48 * rs + off8, R_MN, x=2)
                n = nb0 + RI + 8 * (MI & 1)
                off = n * 48 + ((MI >> 1) << 4)
                off8 = n * 48 + 32
                ag = mem.ldsm(p["off_nm"] + off, R_NM)
                ag8 = mem.ldsm(p["off_nm"] + off8, R_NM, x=2)
                au = mem.ldsm(p["off_nm"] + 48 * rp + off, R_NM)
                au8 = mem.ldsm(p["off_nm"] + 48 * rp + off8, R_NM, x=2)
                for i in range(NB):
                    for q4 in range(4):
                        nn = RI + 8 * (MI >> 1)
                        chunk = 2 * q4 + (MI & 1)
                        off = i * BOX + nn * 128 + ((chunk ^ RI) << 4)
                        a = mem.ldsm(sg + off, (sg, sg + kmat), trans=True)
                        mma(acc[4 * i + q4], a, bg[:, 0], bg[:, 1])
                        mma(acc[4 * i + q4], a, bg[:, 2], bg[:, 3])
                        mma(acc[4 * i + q4], a, bg8[:, 0], bg8[:, 1])
                        a = mem.ldsm(su + off, (su, su + kmat), trans=True)
                        mma(acc[4 * i + q4], a, bu[:, 0], bu[:, 1])
                        mma(acc[4 * i + q4], a, bu[:, 2], bu[:, 3])
                        mma(acc[4 * i + q4], a, bu8[:, 0], bu8[:, 1])
                    col = x0 + 64 * i
                    for af, af8, grad, cnt in ((ag, ag8, grad_g, n_g), (au, au8, grad_u, n_u)):
                        d = np.zeros((8, 32, 4))
                        for t in range(8):
                            mma(d[t], af, hb[8 * i + t], hb[8 * i + t])
                            mma(d[t], af8, hb[8 * i + t])
                        for pp in range(2):
                            # lane (g, c): rows g and g + 8, columns 32 pp + 8 c .. + 7
                            for ln in range(32):
                                g, c = ln >> 2, ln & 3
                                cc = 32 * pp + 8 * c
                                if cc >= K - col:
                                    continue
                                for rr, e0 in ((g, 0), (g + 8, 2)):
                                    if rr < nr:
                                        v = np.array([d[4 * pp + tt, ln, e0 + e] for tt in range(4) for e in range(2)])
                                        gr, gc = n0 + nb0 + rr, col + cc
                                        assert n0 <= gr < n1 and gc + 8 <= K and gc % 8 == 0
                                        grad[gr, gc:gc + 8] = v
                                        cnt[gr, gc:gc + 8] += 1
                if j + S < nblk:
                    fill(j + S)
            for gq in range(4 * NB):
                k = x0 + 16 * gq + G4
                for t in range(32):
                    for e, (dm, dk) in enumerate(((0, 0), (1, 0), (0, 8), (1, 8))):
                        m, kk = 2 * C4[t] + dm, k[t] + dk
                        if m < M and kk < K:
                            part[share, m, kk] = acc[gq, t, e]
                            n_part[share, m, kk] += 1

    assert np.all(n_g == 1) and np.all(n_u == 1), "each weight-gradient element stored exactly once"
    assert np.all(n_part == 1), "each grad_h partial stored exactly once"
    dg, du = dG.astype(np.float64), dU.astype(np.float64)
    ge, ue = dg.T @ h, du.T @ h
    np.testing.assert_allclose(grad_g, ge, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(grad_u, ue, rtol=1e-12, atol=1e-12)
    for s in range(G):
        n0, n1 = N * s // G, N * (s + 1) // G
        pe = dg[:, n0:n1] @ Wg[n0:n1] + du[:, n0:n1] @ Wu[n0:n1]
        np.testing.assert_allclose(part[s], pe, rtol=1e-12, atol=1e-12)
    return p


@pytest.mark.parametrize("M,N,K,sms,NB", [
    (3, 100, 1000, 6, 2),     # K tail inside a box, a partial top block per share
    (8, 64, 512, 4, 2),       # whole blocks
    (5, 37, 264, 3, 2),       # slices past K, shares of 12-13 rows
    (2, 33, 3200, 8, 2),      # several column groups per share
    (8, 300, 136, 5, 2),      # two warps, shares of 60 rows (4 blocks through 2+ stages)
])
def test_replay_matches_plain_sums(M, N, K, sms, NB):
    replay(M, N, K, sms, NB)


def test_plan_on_gb300_shapes():
    """The plan for the workloads' shapes fits the SM's shared memory with at
    least two stages, one CTA per SM."""
    for K, N in ((2560, 9728), (4096, 11008), (4096, 14336), (1024, 3072), (8192, 1000), (768, 1000)):
        for NB in (2,):
            p = plan(8, N, K, 152, NB)
            assert p is not None, (K, N, NB)
            assert p["S"] >= 2 and p["shares"] * p["cg"] <= 152 and p["smem"] <= SMEM_OPTIN
            assert p["warps"] * p["cg"] * 64 * NB >= K
