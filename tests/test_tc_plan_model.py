"""A CPU model of the tcgen05 GEMV's plan and addressing (csrc/glu_tc.cuh and
plan_tc in csrc/mbglu_api.cu), restated from their rules, checked for every
batch 1..64 over a grid of N and K before the kernel runs on a GPU:

  * shared memory: header + alignment slack + stages fit the opt-in limit,
    and every swizzled tile (gate, up, h of each stage) starts on a 1024-byte
    boundary once the base is aligned;
  * the K split: each CTA of a pair gets at least one 64-wide chunk, and rank
    0's stages can hold rank 1's partial sums (2 Np x 128 fp32);
  * tensor memory: g's columns [0, Np) and u's [C/2, C/2 + Np) lie inside the
    C allocated columns (a power of two, 32..512), and do not overlap;
  * tensor copies: every x coordinate is a multiple of 64 elements (128 bytes)
    and inside K, every tile's first row inside N, the h box (Np rows) within
    the 256-row box limit;
  * the MMA shape: M = 128, N = Np a multiple of 16 in 16..256."""
import itertools

import pytest

SMS, OPTIN = 152, 232448               # GB300: SMs, max dynamic + static shared memory per block
BOX, BOXES = 64, 2                     # K per tensor copy (128 bytes, the swizzle row); copies per matrix and stage
ROWS, CHUNK, HEADER, SLACK, MAX_STAGES = 128, BOX * BOXES, 1024, 1024, 8
WBOX = ROWS * BOX * 2                  # one matrix's box
WBYTES = WBOX * BOXES                  # one matrix's stage


def plan(M, N, K):
    Np = (M + 15) // 16 * 16
    nchunk = -(-K // CHUNK)
    ntiles = -(-N // ROWS)
    sbytes = 2 * WBYTES + Np * 128 * BOXES
    stages = min(MAX_STAGES, (OPTIN - HEADER - SLACK) // sbytes)
    if stages < 2:
        return None

    def span(ks):
        return -(-(ntiles * ks) // SMS) / ks

    ks = 1
    for k in range(2, 5):
        fits = (k - 1) * ROWS * (2 * Np + 4) * 4 <= OPTIN - HEADER - SLACK
        if nchunk >= 2 * k and fits and span(k) < span(ks):
            ks = k
    parts = (ks - 1) * ROWS * (2 * Np + 4) * 4    # rank 0's stage memory also takes the partial sums
    return dict(Np=Np, nchunk=nchunk, ntiles=ntiles, ks=ks, stages=stages, sbytes=sbytes,
                smem=HEADER + SLACK + max(stages * sbytes, parts))


@pytest.mark.parametrize("M", list(range(1, 65)))
def test_tc_plan_and_addressing(M):
    for N, K in itertools.product([1, 127, 128, 1337, 9728, 11008, 14336, 19456], [8, 64, 72, 1288, 2560, 4096, 8192]):
        p = plan(M, N, K)
        assert p is not None
        Np, S, sb, ks = p["Np"], p["stages"], p["sbytes"], p["ks"]
        assert Np % 16 == 0 and 16 <= Np <= 256 and Np <= 256          # MMA N; h box rows
        assert p["smem"] <= OPTIN and 2 <= S <= MAX_STAGES
        for base_off in (0, 16, 1008):                                   # where the runtime puts the dynamic base
            base = base_off + ((1024 - base_off % 1024) % 1024)
            assert base % 1024 == 0 and base - base_off + HEADER + S * sb <= p["smem"]
            for s in range(S):
                offs = [b * WBOX for b in range(BOXES)] + [WBYTES + b * WBOX for b in range(BOXES)] + \
                       [2 * WBYTES + b * Np * 128 for b in range(BOXES)]
                for off in offs:                                          # every box a swizzled tile
                    assert (base + HEADER + s * sb + off) % 1024 == 0
                assert 2 * WBYTES + BOXES * Np * 128 == sb
        ncols = 64 if 2 * Np <= 64 else 128
        ucol = ncols // 2
        assert ncols & (ncols - 1) == 0 and 32 <= ncols <= 512
        assert Np <= ucol and ucol + Np <= ncols                          # g and u apart, inside the allocation
        for rank in range(ks):
            c0 = p["nchunk"] * rank // ks
            nch = p["nchunk"] * (rank + 1) // ks - c0
            assert nch >= 1
            for i in (0, nch - 1):
                x = (c0 + i) * CHUNK
                assert x % 64 == 0 and x < K
                for b in range(BOXES):                                    # later boxes may lie past K: zeros
                    assert (x + b * BOX) % 64 == 0
        if ks > 1:
            room = p["smem"] - HEADER - SLACK                               # rank 0's stage memory, allocated
            pitch = 2 * Np + 4                                            # [128 rows][2 Np + 4] fp32 per rank
            assert (pitch * 4) % 16 == 0 and (pitch * 4) % 128 == 16      # 16-byte rows, banks apart
            for r in range(1, ks):                                        # each partial slot inside it
                assert (r - 1) * ROWS * pitch * 4 + ROWS * pitch * 4 <= room
        for tile in (0, p["ntiles"] - 1):
            assert tile * ROWS < N
        assert p["ntiles"] * ks <= 2 ** 31 - 1


def test_tc_split_choice():
    """The split that shortens the longest per-SM queue: 76 tiles (N = 9728)
    pair up into 152 CTAs; 86 tiles (N = 11008) split 3 ways into 258 CTAs,
    2 waves of a third of K (0.67 of a tile, against 1.0 unsplit); 112 tiles
    (N = 14336) split 4 ways into 448 CTAs, 3 waves of a quarter (0.75)."""
    assert plan(64, 9728, 2560)["ks"] == 2
    assert plan(32, 11008, 4096)["ks"] == 3
    assert plan(64, 14336, 4096)["ks"] == 4
    assert plan(17, 128, 64)["ks"] == 1                      # one chunk: no split


def _sw128_offset(addr):
    """The 128-byte swizzle on a shared-memory byte address: the 16-byte chunk
    index (bits 4-6) XOR the row within the 1024-byte atom (bits 7-9)."""
    return addr ^ (((addr >> 7) & 7) << 4)


@pytest.mark.parametrize("rows", [16, 32, 48, 64, 128])
def test_sw128_descriptor_walk_reads_the_tma_tile(rows):
    """A tensor copy with 128-byte swizzling places element (r, c) of a
    [rows][64] bf16 box at swizzle(base + r * 128 + 2c) (base 1024-aligned:
    rows of 128 bytes, 8-row atoms of 1024).  The MMA reads row r, K step kk
    (16 elements) through the descriptor: start address base + 32 kk, 8-row
    groups SBO = 1024 bytes apart, 16-byte units j = 0, 1, the same swizzle
    on the address.  Every element it reads must be (r, 16 kk + 8 j + e)."""
    base = 3 * 1024
    smem = {}
    for r in range(rows):
        for c in range(64):
            smem[_sw128_offset(base + r * 128 + 2 * c)] = (r, c)
    assert len(smem) == rows * 64                                      # a bijection onto the tile's bytes
    sbo = 1024
    for kk in range(4):
        start = base + 32 * kk
        for r in range(rows):
            for j in range(2):
                for e in range(8):
                    a = start + (r >> 3) * sbo + (r & 7) * 128 + 16 * j + 2 * e
                    assert smem[_sw128_offset(a)] == (r, 16 * kk + 8 * j + e)
