"""CPU model of gdn_gates' work split (the host's choice in csrc/mbglu_api.cu
and gdn_gates_chunk_kernel in csrc/glu_kernels.cuh), restated here.

The chunk kernel gives thread i the item (t, j0) = (i // hc, 8 (i % hc)) with
hc = ceil(H / 8), grid-striding in 32-bit unsigned indices.  The model checks,
for the shapes the host sends to it, that every (token, head) is computed
exactly once, that no index wraps, that the per-head table fits its shared
arrays, and that the 16-byte path only ever touches 16-byte aligned
addresses."""
import pytest

SMS = 152
MAX_HEADS = 4096            # kGdnMaxHeads


def host_choice(T, H, lda, ldb, ldg, ldbeta, align=(0, 0, 0, 0)):
    chunks = T * ((H + 7) // 8)
    by_chunk = H <= MAX_HEADS and chunks < (1 << 31)
    vec = H % 8 == 0 and all(a % 16 == 0 for a in align) and lda % 8 == 0 and ldb % 8 == 0 and \
        ldg % 4 == 0 and ldbeta % 8 == 0
    work = chunks if by_chunk else T * H
    grid = max(1, min(SMS * 8, (work + 255) // 256))
    return by_chunk, vec, grid


def chunk_items(T, H, grid, block=256):
    hc = (H + 7) // 8
    items = T * hc
    stride = grid * block
    assert stride < (1 << 32) and items - 1 + stride < (1 << 32), "a 32-bit index would wrap"
    for tid in range(grid * block):
        i = tid
        while i < items:
            t, j0 = i // hc, (i % hc) * 8
            yield t, j0
            i += stride


@pytest.mark.parametrize("T,H", [(1, 1), (3, 7), (5, 8), (17, 32), (33, 40), (2, 4096), (1000, 13)])
def test_every_token_and_head_once(T, H):
    by_chunk, vec, grid = host_choice(T, H, H, H, H, H)
    assert by_chunk
    seen = {}
    for t, j0 in chunk_items(T, H, grid):
        n = min(8, H - j0)
        assert n >= 1 and j0 + n <= H <= MAX_HEADS
        for e in range(n):
            seen[(t, j0 + e)] = seen.get((t, j0 + e), 0) + 1
    assert seen == {(t, j): 1 for t in range(T) for j in range(H)}


@pytest.mark.parametrize("T,H,lda,ldb,ldg,ldbeta", [(64, 32, 32, 32, 32, 32), (40, 16, 24, 40, 20, 16),
                                                    (9, 8, 8, 64, 8, 8)])
def test_vector_path_addresses_are_16_byte_aligned(T, H, lda, ldb, ldg, ldbeta):
    by_chunk, vec, grid = host_choice(T, H, lda, ldb, ldg, ldbeta)
    assert by_chunk and vec
    for t, j0 in chunk_items(T, H, grid):
        assert (2 * (t * lda + j0)) % 16 == 0 and (2 * (t * ldb + j0)) % 16 == 0
        assert (4 * (t * ldg + j0)) % 16 == 0 and (4 * (t * ldg + j0 + 4)) % 16 == 0
        assert (2 * (t * ldbeta + j0)) % 16 == 0 and j0 + 8 <= H


def test_the_host_falls_back_where_the_chunk_kernel_cannot_go():
    assert not host_choice(10, 4097, 4097, 4097, 4097, 4097)[0]      # heads past the shared table
    assert not host_choice(1 << 28, 64, 64, 64, 64, 64)[0]           # 2^31 items
    assert not host_choice(5, 8, 9, 8, 8, 8)[1]                      # an odd row stride: no 16-byte path
    assert not host_choice(5, 12, 16, 16, 16, 16)[1]                 # H % 8 != 0
    # the benchmark's shape: 262144 tokens x 32 heads, one CTA wave of 8 per SM
    by_chunk, vec, grid = host_choice(262144, 32, 32, 32, 32, 32)
    assert by_chunk and vec and grid == SMS * 8
