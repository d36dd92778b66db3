"""Lane-level model of the PTX operations the tensor-core kernels use, for
the CPU replays of their index arithmetic: ldmatrix .x4 / .x2 (with and
without .trans), mma.sync m16n8k16 / m16n8k8 .row.col fragment layouts, and
shared memory as float64 slots (one per bf16) whose every access names the
region it must stay in.  Test infrastructure: it models data movement only."""
import numpy as np

LANE = np.arange(32)
G4, C4 = LANE >> 2, LANE & 3     # mma: group id, thread in group
MI, RI = LANE >> 3, LANE & 7     # ldmatrix / stmatrix: matrix, row of the lane's address


def bf16_rn(x):
    """float32 -> the nearest bf16 (ties to even), as float32 (finite x)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32)


class Smem:
    """Shared memory as float64 slots, one per bf16 (byte offset // 2) from the
    kernel's 1024-byte aligned base; every access names its region."""

    def __init__(self, nbytes):
        self.nbytes = nbytes
        self.v = np.full(nbytes // 2, np.nan)

    def rows16(self, addrs, region):
        lo, hi = region
        addrs = np.asarray(addrs)
        assert np.all(addrs % 16 == 0), "matrix rows are 16-byte aligned"
        assert np.all(addrs >= lo) and np.all(addrs + 16 <= hi), (addrs.min(), addrs.max(), region)
        assert hi <= self.nbytes
        return (addrs // 2)[:, None] + np.arange(8)[None, :]   # [lanes][8] slots

    def ldsm(self, addrs, region, trans=False, x=4):
        """ldmatrix .x4 / .x2: lanes 8i..8i+7 address the rows of matrix i; lane t
        gets, per matrix, (row t/4, columns 2(t%4), +1), or the transpose's."""
        addrs = np.asarray(addrs)[:8 * x]
        vals = self.v[self.rows16(addrs, region)].reshape(x, 8, 8)   # [matrix][row][col]
        assert not np.any(np.isnan(vals)), "read of unwritten shared memory"
        if trans:
            vals = vals.transpose(0, 2, 1)
        out = np.empty((32, x, 2))
        for e in range(2):
            out[:, :, e] = vals[:, G4, 2 * C4 + e].T
        return out


def mma(d, a, b0, b1=None):
    """mma.sync .row.col, d [32][4] += A x B from fragments: m16n8k16 (a: 4
    registers, b0 and b1) or m16n8k8 (a: 2 registers, b0 only)."""
    kk = 16 if a.shape[1] == 4 else 8
    A = np.zeros((16, kk))
    B = np.zeros((kk, 8))
    D = np.zeros((16, 8))
    for e in range(2):
        A[G4, 2 * C4 + e] = a[:, 0, e]
        A[G4 + 8, 2 * C4 + e] = a[:, 1, e]
        B[2 * C4 + e, G4] = b0[:, e]
        if kk == 16:
            A[G4, 2 * C4 + 8 + e] = a[:, 2, e]
            A[G4 + 8, 2 * C4 + 8 + e] = a[:, 3, e]
            B[2 * C4 + 8 + e, G4] = b1[:, e]
        D[G4, 2 * C4 + e] = d[:, e]
        D[G4 + 8, 2 * C4 + e] = d[:, 2 + e]
    D = D + A @ B
    for e in range(2):
        d[:, e] = D[G4, 2 * C4 + e]
        d[:, 2 + e] = D[G4 + 8, 2 * C4 + e]
