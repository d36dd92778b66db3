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

def bwd_mma_warps(NB, MB=8):
    return 8 if MB > 8 else 8 if NB >= 4 else 12


def pitch(MB):
    return 56 if MB > 8 else 24


def plan(M, N, K, sms, NB=2, warps=0):
    if M > 16 or K % 8:
        return None
    MB = 16 if M > 8 else 8
    P = pitch(MB)
    parts_cap = max(MAX_PARTS * min(M, 8), 48 * M) // M
    wtot = -(-K // (64 * NB))
    wmax = min(warps if warps > 0 else bwd_mma_warps(NB, MB), bwd_mma_warps(NB, MB))
    wmin = warps if warps > 0 else 1
    stage = 2 * NB * BOX
    best, best_score = None, -1
    for w in range(wmax, wmin - 1, -1):
        cg = -(-wtot // w)
        W = -(-wtot // cg)
        if W != w:
            continue
        shares = max(1, min((N + 15) // 16, sms // cg, parts_cap))
        rows_cta = -(-N // shares)
        rows_pad = -(-rows_cta // 16) * 16
        off_nm = 512
        off_ring = (off_nm + 4 * P * rows_pad + 1023) & ~1023
        room = SMEM_OPTIN - 1024 - off_ring
        if room <= 0:
            continue
        S = min(4, room // (W * stage), 64 // W)
        if S < 2:
            continue
        score = 16 * W + S
        if score > best_score:
            best_score = score
            best = dict(NB=NB, MB=MB, cg=cg, warps=W, shares=shares, rows_cta=rows_cta, rows_pad=rows_pad, S=S,
                        off_nm=off_nm, off_ring=off_ring, stage=stage, smem=off_ring + W * S * stage + 1024)
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
    W, S, cg, G, MB = p["warps"], p["S"], p["cg"], p["shares"], p["MB"]
    NT, P = MB // 8, pitch(MB)
    NC = 3 * NT
    rp = p["rows_pad"]
    mat_bytes = rp * P * 2
    stage, kmat = p["stage"], NB * BOX
    assert p["smem"] <= SMEM_OPTIN and W * S <= 64 and W <= bwd_mma_warps(NB, MB)
    assert p["off_ring"] >= p["off_nm"] + 2 * mat_bytes and p["off_ring"] % 1024 == 0 and stage % 1024 == 0
    assert (P * 2 // 16) % 2 == 1, "a staged row is an odd number of 16-byte units (no bank conflict)"
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
    R_NM = (p["off_nm"], p["off_nm"] + 2 * mat_bytes)

    for bid in range(G * cg):
        share, cgrp = divmod(bid, cg)
        n0, n1 = N * share // G, N * (share + 1) // G
        rows = n1 - n0
        nblk = -(-rows // 16)
        assert rows <= p["rows_cta"] <= rp
        mem = Smem(avail)
        # dG, dU staged as three bf16 terms: [matrix][rp][P], row n = hi m0.., mid m0.., lo m0..
        for m in range(MB):
            for r in range(rp):
                ok = m < M and r < rows
                for mat, terms in ((0, tg), (1, tu)):
                    for e in range(3):
                        v = terms[e][m, n0 + r] if ok else 0.0
                        mem.v[p["off_nm"] // 2 + (mat * rp + r) * P + e * MB + m] = v
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

            # h fragments: (h[2c + 8 half][k], h[2c + 1 + 8 half][k]), k the weight
            # column of MMA column g in tile t = 4p + t'
            hb = np.zeros((8 * NB, 2, 32, 2))
            for t in range(8 * NB):
                k = x0 + 32 * (t >> 2) + 8 * (G4 >> 1) + 2 * (t & 3) + (G4 & 1)
                for half in range(NT):
                    for e in range(2):
                        m = 2 * C4 + e + 8 * half
                        ok = (k < K) & (m < M)
                        hb[t, half, :, e] = np.where(ok, h[np.minimum(m, M - 1), np.minimum(k, K - 1)], 0.0)
            for j in range(min(S, nblk)):
                fill(j)
            acc = np.zeros((NT, 4 * NB, 32, 4))
            for j in range(nblk):
                st = j % S
                nb0 = 16 * (nblk - 1 - j)
                nr = min(16, rows - nb0)
                sg = ring + st * stage
                su = sg + kmat
                # grad_h's B: per (term, batch tile) chunk, rows 0-7 then 8-15, transposed
                bh = np.zeros((2, NC, 2, 32, 2))
                for mat in range(2):
                    for c0 in range(0, NC, 2):
                        ch = np.minimum(c0 + (MI >> 1), NC - 1)
                        addr = p["off_nm"] + mat * mat_bytes + (nb0 + 8 * (MI & 1) + RI) * P * 2 + ch * 16
                        r = mem.ldsm(addr, R_NM, trans=True)
                        bh[mat, c0] = r[:, 0:2].transpose(1, 0, 2)
                        if c0 + 1 < NC:
                            bh[mat, c0 + 1] = r[:, 2:4].transpose(1, 0, 2)
                for i in range(NB):
                    for mat, sb in ((0, sg), (1, su)):
                        for q4 in range(4):
                            nn = RI + 8 * (MI >> 1)
                            chunk = 2 * q4 + (MI & 1)
                            a = mem.ldsm(sb + i * BOX + nn * 128 + ((chunk ^ RI) << 4), (sb, sb + kmat), trans=True)
                            for c in range(NC):
                                mma(acc[c % NT, 4 * i + q4], a, bh[mat, c, 0], bh[mat, c, 1])
                if j + S < nblk:
                    fill(j + S)
                # grad_W's A
                n = nb0 + RI + 8 * (MI & 1)
                aws = []
                for mat in range(2):
                    row = p["off_nm"] + mat * mat_bytes + n * P * 2
                    if MB > 8:
                        aws.append([mem.ldsm(row + ((2 * e + (MI >> 1)) << 4), R_NM) for e in range(3)])
                    else:
                        aws.append([mem.ldsm(row + ((MI >> 1) << 4), R_NM), mem.ldsm(row + 32, R_NM, x=2)])
                for i in range(NB):
                    col = x0 + 64 * i
                    for aw, grad, cnt in ((aws[0], grad_g, n_g), (aws[1], grad_u, n_u)):
                        d = np.zeros((8, 32, 4))
                        for t in range(8):
                            if MB > 8:
                                for e in range(3):
                                    mma(d[t], aw[e], hb[8 * i + t, 0], hb[8 * i + t, 1])
                            else:
                                mma(d[t], aw[0], hb[8 * i + t, 0], hb[8 * i + t, 0])
                                mma(d[t], aw[1], hb[8 * i + t, 0])
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
            for mt in range(NT):
                for gq in range(4 * NB):
                    k = x0 + 16 * gq + G4
                    for t in range(32):
                        for e, (dm, dk) in enumerate(((0, 0), (1, 0), (0, 8), (1, 8))):
                            m, kk = 8 * mt + 2 * C4[t] + dm, k[t] + dk
                            if m < M and kk < K:
                                part[share, m, kk] = acc[mt, gq, t, e]
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
    (16, 100, 1000, 6, 2),    # batch 16: two batch tiles, three terms per tile
    (11, 37, 264, 3, 2),      # batch 11 (rows 11..15 zero), slices past K
])
def test_replay_matches_plain_sums(M, N, K, sms, NB):
    replay(M, N, K, sms, NB)


def test_plan_on_gb300_shapes():
    """The plan for the workloads' shapes fits the SM's shared memory with at
    least two stages, one CTA per SM."""
    for K, N in ((2560, 9728), (4096, 11008), (4096, 14336), (1024, 3072), (8192, 1000), (768, 1000)):
        for NB in (2,):
            p = plan(16 if K < 8192 else 8, N, K, 152, NB)
            assert p is not None, (K, N, NB)
            assert p["S"] >= 2 and p["shares"] * p["cg"] <= 152 and p["smem"] <= SMEM_OPTIN
            assert p["warps"] * p["cg"] * 64 * NB >= K
