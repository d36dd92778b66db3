"""CPU model of the backward's fused second step (glu_bwd_hw_kernel): its
plan (plan_bwd_hw in csrc/mbglu_api.cu, restated here) and the kernel's
index arithmetic, replayed for many shapes.  Checks that every weight-
gradient element is written exactly once, that every grad_h partial column
is written by exactly one lane per row share, that each warp's ring, the
barriers and the staged dG/dU stay inside shared memory, and that every
tensor copy starts on a 16-byte boundary (x a multiple of 8 elements)."""
import pytest

SMEM_OPTIN = 232448        # GB300: max dynamic shared memory per block (opt-in)
SMS = 152
SLICE = 256


def batch_tile(M):
    return 1 if M <= 1 else 2 if M <= 2 else 4 if M <= 4 else 8 if M <= 8 else 16


def hw_warps(MB):
    return 10 if MB >= 8 else 14 if MB >= 4 else 16


def plan(M, N, K):
    if M > 8 or K % 8:
        return None
    MB = batch_tile(M)
    wtot = -(-K // SLICE)
    wmax = hw_warps(MB)
    cg = -(-wtot // wmax)
    warps = -(-wtot // cg)
    shares = max(1, min(N, SMS // cg))
    rows_cta = -(-N // shares)
    dgu = 2 * MB * rows_cta * 4
    off_ring = (256 + dgu + 127) & ~127
    room = SMEM_OPTIN - off_ring
    for Rmax in (8, 4, 2):
        R = min(Rmax, rows_cta)
        stage = 2 * R * SLICE * 2
        S = min(8, room // (warps * stage), 32 // warps)
        if S >= 2:
            smem = off_ring + warps * S * stage
            return dict(MB=MB, cg=cg, warps=warps, shares=shares, rows_cta=rows_cta, R=R, S=S, off_ring=off_ring,
                        stage=stage, smem=smem)
    return None


def replay(M, N, K):
    p = plan(M, N, K)
    assert p is not None
    assert p["smem"] <= SMEM_OPTIN and p["warps"] * p["S"] * 8 <= 256 and p["warps"] <= hw_warps(p["MB"])
    assert p["off_ring"] % 128 == 0 and p["stage"] % 1024 == 0
    written = {}
    part_cols = {}
    G = p["shares"]
    for bid in range(G * p["cg"]):
        share, cgrp = divmod(bid, p["cg"])
        n0, n1 = N * share // G, N * (share + 1) // G
        rows = n1 - n0
        assert rows <= p["rows_cta"] and 2 * p["MB"] * p["rows_cta"] * 4 + 256 <= p["off_ring"]
        nblk = -(-rows // p["R"])
        for warp in range(p["warps"]):
            x0 = (cgrp * p["warps"] + warp) * SLICE
            assert x0 % 8 == 0
            ring0 = p["off_ring"] + warp * p["S"] * p["stage"]
            assert ring0 + p["S"] * p["stage"] <= p["smem"]
            if x0 >= K:
                continue
            for j in range(nblk):
                hi = n1 - j * p["R"]
                lo = max(n0, hi - p["R"])
                assert lo < hi and lo >= n0 and hi - lo <= p["R"]
                for lane in range(32):
                    col = x0 + 8 * lane
                    if col >= K:
                        continue
                    for i in range(hi - lo):
                        key = (lo + i, col)
                        assert key not in written, key
                        written[key] = True
            for lane in range(32):
                col = x0 + 8 * lane
                if col < K:
                    k = (share, col)
                    assert k not in part_cols
                    part_cols[k] = True
    assert len(written) == N * (K // 8)
    assert len(part_cols) == G * (K // 8)
    return p


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 8), (7, 64), (300, 264), (1337, 1288), (3000, 2560), (9728, 2560),
                                 (513, 4104), (2000, 4096), (700, 8192), (11008, 4096)])
def test_every_gradient_element_written_once(M, N, K):
    replay(M, N, K)


def test_headline_plan():
    p = plan(8, 9728, 2560)
    assert (p["cg"], p["warps"], p["shares"], p["R"], p["S"]) == (1, 10, 152, 8, 2)
    p = plan(1, 9728, 2560)
    assert p["warps"] == 10 and p["S"] >= 2
