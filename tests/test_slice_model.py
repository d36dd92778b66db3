"""CPU model of the K-slice tensor-core GEMV (glu_slice_kernel in
csrc/glu_slice.cuh): its plan (plan_slice in csrc/mbglu_api.cu, restated
here) and the kernel's shared-memory addresses, fragments, unit order and
stores, replayed lane by lane with the PTX fragment layouts of ldmatrix and
mma.sync m16n8k16 (tests/frag_model.py) and the 128-byte swizzle of a tensor
copy.

Values travel in float64 and are never rounded, so the replay must give the
plain dot products g[m][n] = sum_k h[m][k] Wg[n][k] (u likewise) to float64
rounding: a wrong index, swizzle, fragment mapping, row mask or unit order
anywhere changes them.  The replay also checks that every output is stored
exactly once and only by the CTA owning its row, that each ring stage is
read only after the copy of the unit it holds, that every shared-memory
access stays inside its region and that each tensor copy lands on a
1024-byte boundary with x a multiple of 8 elements."""
import numpy as np
import pytest

from frag_model import C4, G4, MI, RI, Smem, bf16_rn, mma

SMEM_OPTIN = 232448        # GB300: max dynamic shared memory per block (opt-in)
SMS = 152
SEG = 256                  # columns per segment
BOX = 8 * 128              # one 64-column x 8-row box of bf16, bytes
STAGE = 2 * 4 * BOX        # both matrices, 8 KB
SLOTS = 4
SLOT_BYTES = 4 * 32 * 4


def max_warps(spw, mb=8):
    return 10 if mb > 8 else 12 if spw <= 1 else 8 if spw == 2 else 6


def slots(mb):
    return 2 if mb > 8 else 4


def slot_bytes(mb):
    return (8 if mb > 8 else 4) * 32 * 4


def layout(c, M=0, K=0, norm=False):
    """Shared-memory layout and ring depth of one candidate (slice_layout).
    norm: h_s[M][K + 8] shares the slots' region; norm_w [K] and the
    statistic's partials (2 floats per thread) follow at off_s."""
    W = c["warps"]
    region = slots(c["mb"]) * W * slot_bytes(c["mb"])
    if norm:
        region = max(region, M * (K + 8) * 2)
    c["off_s"] = (1024 + region + 127) & ~127
    end = c["off_s"]
    if norm:
        end = c["off_s"] + ((2 * K + 127) & ~127) + 2 * 32 * (W + 1) * 4
    c["off_ring"] = (end + 1023) & ~1023
    room = SMEM_OPTIN - 1024 - 256 - c["off_ring"]
    if room <= 0:
        return False
    c["stages"] = min(6, room // (W * STAGE), 64 // W)
    c["smem"] = c["off_ring"] + W * c["stages"] * STAGE + 1024
    return c["stages"] >= 2


def plan(M, N, K, sms=SMS, spw_only=0, mma_min_m=3, norm=False):
    if M < 1 or M > 16 or K < SEG or K % 8 or N < 1 or (norm and M < mma_min_m):
        return None
    nseg = -(-K // SEG)
    if M > 8:
        if norm:
            return None
        c = dict(spw=1, mb=16, warps=nseg)
        if nseg > max_warps(1, 16) or not layout(c):
            return None
        c["grid"] = max(1, min(sms, (N + 7) // 8))
        return c
    for spw in ((1,) if M < mma_min_m else (1, 2, 3)):
        if spw_only and spw != spw_only:
            continue
        W = -(-nseg // spw)
        if W > max_warps(spw) or (W - 1) * spw >= nseg:
            continue
        c = dict(spw=spw, mb=8, warps=W)
        if not layout(c, M, K, norm):
            continue
        c["grid"] = max(1, min(sms, (N + 7) // 8))
        return c
    return None


def replay(M, N, K, sms=SMS, spw_only=0, seed=0):
    p = plan(M, N, K, sms, spw_only)
    assert p is not None
    W, S, spw, mb = p["warps"], p["stages"], p["spw"], p["mb"]
    NP, NA = (8, 4) if mb > 8 else (4, 2)
    assert p["smem"] <= SMEM_OPTIN and W * S <= 64 and W <= max_warps(spw, mb)
    assert p["off_s"] >= 1024 + slots(mb) * W * slot_bytes(mb) and p["off_ring"] % 1024 == 0
    assert 64 + 2 * slots(mb) <= 72   # barrier words [512, 576)
    rng = np.random.default_rng(seed)
    q = lambda *shape: bf16_rn(rng.standard_normal(shape).astype(np.float32)).astype(np.float64)
    h, Wg, Wu = q(M, K), q(N, K), q(N, K)
    G = p["grid"]
    out_g = np.full((M, N), np.nan)
    out_u = np.full((M, N), np.nan)
    n_out = np.zeros((M, N), int)
    avail = p["smem"] - 1024
    for share in range(G):
        r0, r1 = N * share // G, N * (share + 1) // G
        ngroups = -(-(r1 - r0) // 8)
        sums = np.zeros((ngroups, NP, 32))
        if True:
            mem = Smem(avail)
            for g in range(ngroups):
                slot = np.full((W, NP, 32), np.nan)
                for warp in range(W):
                    x0 = warp * spw * SEG
                    nseg = max(0, min(spw, -(-(K - x0) // SEG)))
                    assert nseg >= 1, "every compute warp has a segment"
                    ring = p["off_ring"] + warp * S * STAGE
                    assert ring + S * STAGE <= avail
                    # h fragments of this warp's columns: rows g and g + 8
                    ha = np.zeros((16 * spw, 4, 32, 2))
                    for j in range(16 * spw):
                        for e in range(2):
                            k = x0 + 16 * j + 8 * e + 2 * C4
                            for rr in range(mb // 8):
                                row = G4 + 8 * rr
                                for t in range(2):
                                    ok = (row < M) & (k + t < K)
                                    ha[j, 2 * e + rr, :, t] = np.where(
                                        ok, h[np.minimum(row, M - 1), np.minimum(k + t, K - 1)], 0.0)
                    part = np.zeros((32, NP))
                    for s in range(nseg):
                        u = g * nseg + s
                        st = u % S
                        y, x = r0 + 8 * g, x0 + s * SEG
                        assert 0 <= y < N
                        for mat, Wm in ((0, Wg), (1, Wu)):
                            for i in range(4):
                                dst = ring + st * STAGE + (4 * mat + i) * BOX
                                assert dst % 1024 == 0 and (x + 64 * i) % 8 == 0
                                for r in range(8):
                                    for c in range(64):
                                        v = Wm[y + r, x + 64 * i + c] if (y + r < N and x + 64 * i + c < K) else 0.0
                                        mem.v[(dst + r * 128 + (((c >> 3) ^ r) << 4) + (c & 7) * 2) // 2] = v
                        sb = ring + st * STAGE
                        dg = np.zeros((32, 4))
                        du = np.zeros((32, 4))
                        for j in range(16):
                            ch = 2 * j + (MI & 1)
                            addr = sb + (MI >> 1) * 4 * BOX + (ch >> 3) * BOX + RI * 128 + (((ch & 7) ^ RI) << 4)
                            bfr = mem.ldsm(addr, (sb, sb + STAGE))
                            a = ha[16 * s + j].transpose(1, 0, 2)   # [lane][a0..a3][2]
                            mma(dg, a, bfr[:, 0], bfr[:, 1])
                            mma(du, a, bfr[:, 2], bfr[:, 3])
                        if mb == 8:
                            assert np.all(dg[:, 2:] == 0) and np.all(du[:, 2:] == 0)
                        part += np.concatenate([dg[:, :NP // 2], du[:, :NP // 2]], axis=1)
                    slot[warp] = part.T
                # the epilogue warp: the warps' partials in order
                acc = slot[0].copy()
                for w in range(1, W):
                    acc += slot[w]
                sums[g] = acc
        for g in range(ngroups):
            acc = sums[g]
            for ln in range(32):
                m, n = ln >> 2, r0 + 8 * g + 2 * (ln & 3)
                for hh in range(mb // 8):
                    mm = m + 8 * hh
                    if mm >= M:
                        continue
                    for dn in range(2):
                        if n + dn < r1:
                            out_g[mm, n + dn] = acc[2 * hh + dn, ln]
                            out_u[mm, n + dn] = acc[NP // 2 + 2 * hh + dn, ln]
                            n_out[mm, n + dn] += 1
    assert np.all(n_out == 1), "each output stored exactly once"
    np.testing.assert_allclose(out_g, h @ Wg.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out_u, h @ Wu.T, rtol=1e-12, atol=1e-12)
    return p


@pytest.mark.parametrize("M,N,K,sms,spw", [
    (3, 50, 256, 4, 0),        # one segment, one warp; partial last groups
    (1, 100, 2568, 5, 0),      # batch 1 (rows 1..7 of A zero); 11 warps, the last with 8 columns
    (8, 37, 1000, 3, 0),       # a segment past K in part; shares of 12-13 rows
    (5, 64, 1288, 2, 2),       # two segments per warp, the last warp with one
    (8, 20, 2560, 3, 3),       # three per warp, ragged; shares under one group
    (4, 9, 4096, 1, 0),        # 16 segments, one CTA, one partial group
    (16, 40, 2560, 4, 0),      # batch 16, 10 warps, one CTA per share
    (11, 30, 1288, 3, 0),      # batch 11 (rows 11..15 zero), a segment past K
])
def test_replay_matches_plain_dot_products(M, N, K, sms, spw):
    replay(M, N, K, sms, spw)


def test_plan_on_the_workloads():
    """The workloads' shapes get a plan with at least two stages per warp and
    one CTA per SM; K past the register budget of the h fragments gets none."""
    for K in (1024, 2560, 4096):
        for M in (3, 4, 8):
            p = plan(M, 9728, K)
            assert p is not None and p["stages"] >= 2 and p["smem"] <= SMEM_OPTIN and p["grid"] == SMS
            assert p["warps"] * p["spw"] * SEG >= K
    assert plan(8, 9728, 8192) is None and plan(17, 9728, 2560) is None and plan(8, 9728, 200) is None
    # batch 9-16: one segment per warp, up to 10 warps
    assert plan(16, 9728, 2560)["warps"] == 10 and plan(16, 9728, 2560)["stages"] >= 2
    assert plan(16, 14336, 4096) is None and plan(9, 9728, 2568) is None
    # batch 1-2: one segment per warp only (K <= 12 * 256)
    assert plan(1, 9728, 2560)["spw"] == 1 and plan(2, 9728, 3072)["spw"] == 1
    assert plan(1, 9728, 4096) is None and plan(2, 11008, 3080) is None


PRO_BAR = 784              # the prologue copies' mbarrier (kProBarOffset)
STATIC_SMEM = 256          # the kernel's static shared memory (inv_s and alignment)


@pytest.mark.parametrize("M", [3, 4, 5, 8])
def test_norm_variant_layout(M):
    """The add_rmsnorm_glu variant's shared memory, for every K the plan
    takes: the barriers, the prologue barrier, h_s[M][K + 8] (which the slots
    reuse after a barrier), norm_w and the statistic's partials at off_s, and
    the 1024-byte aligned ring are disjoint and inside the allocation; every
    bulk copy of the prologue starts and ends on 16-byte boundaries."""
    taken = 0
    for K in range(256, 4608 + 1, 8):
        p = plan(M, 9728, K, norm=True)
        if p is None:
            continue
        taken += 1
        W, S, nslot = p["warps"], p["stages"], slots(p["mb"])
        threads = 32 * (W + 1)
        assert 8 * W * S <= 512 and 512 + 16 * nslot <= PRO_BAR and PRO_BAR + 8 <= 1024
        hs_end = 1024 + M * (K + 8) * 2
        assert hs_end <= p["off_s"] and 1024 + nslot * W * slot_bytes(p["mb"]) <= p["off_s"]
        parts = p["off_s"] + ((2 * K + 127) & ~127)
        assert parts + 2 * threads * 4 <= p["off_ring"] and p["off_ring"] % 1024 == 0
        # the kernel rounds its base up to 1024 bytes: at most 1023 of the allocation
        assert p["off_ring"] + W * S * STAGE + 1023 <= p["smem"]
        assert p["smem"] + STATIC_SMEM <= SMEM_OPTIN and S >= 2
        # residual rows land row by row at the padded pitch, norm_w in one copy
        for r in range(M):
            assert (1024 + r * (K + 8) * 2) % 16 == 0 and (2 * K) % 16 == 0
        assert p["off_s"] % 16 == 0
    assert taken > 0
    # the K2560 shape of the norm workload: 10 compute warps, 2 stages
    p = plan(M, 9728, 2560, norm=True)
    assert p["warps"] == 10 and p["stages"] == 2 and p["spw"] == 1


@pytest.mark.parametrize("K", [256, 1024, 2560, 2568, 4096])
def test_norm_fragment_loads_and_bank_groups(K):
    """The compute warps read their A fragments from h_s at a row pitch of
    K + 8: lane (g, c) reads 4 bytes of row g at column k0 + 2 c.  With
    K % 16 == 0 the 32 lanes hit 32 different banks; at K % 16 == 8 the pitch
    puts two rows on each bank (the kernel is still correct, only slower)."""
    words = [(g * (K + 8) * 2 + 4 * c) // 4 for g in range(8) for c in range(4)]
    banks = {w % 32 for w in words}
    if K % 16 == 0:
        assert len(banks) == 32
    else:
        assert len(banks) == 16
