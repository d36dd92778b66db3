"""CPU model of the norm prologue's work split (row_map, x_prefetch_rows and
add_rows_in_place in csrc/glu_kernels.cuh), restated here.

Thread t of a block of B threads owns row m = t // P (P = B // M threads per
row; threads past M P own nothing) and the row's 16-byte chunks c0 + i P
(c0 = t - m P).  x arrives in batches of NX chunks per thread: the first
before the residual copy is awaited, the rest inside the add loop.  The model
checks that every chunk of every row is added exactly once, by a thread of
its row, in ascending order within that thread, and that this order is the
same for NX = 8 and NX = 16.  A thread's double-float sum of squares, and so
the statistic and h, therefore do not depend on the batch size.  It also
checks that the shapes the K-slice and streaming kernels take at K = 2560
need a single batch (one round trip for x) at NX = 8."""
import pytest


def visits(M, K, B, NX):
    """Per thread: the (row, chunk) pairs in the order they are added, and
    the number of x batches it loads."""
    P = B // M
    nch = K // 8
    out = []
    for t in range(B):
        m = t // P
        c0 = t - m * P
        active = m < M
        seq, batches, j0 = [], 0, 0
        while True:
            batches += 1
            for j in range(NX):
                c = c0 + (j0 + j) * P
                if active and c < nch:
                    seq.append((m, c))
            if not active or c0 + (j0 + NX) * P >= nch:
                break
            j0 += NX
        out.append((seq, batches))
    return out


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 13, 16])
@pytest.mark.parametrize("K,B", [(2560, 352), (4096, 288), (1032, 288), (264, 352), (2568, 320)])
def test_every_chunk_once_in_the_same_order_for_both_batch_sizes(M, K, B):
    v8, v16 = visits(M, K, B, 8), visits(M, K, B, 16)
    seen = {}
    for t, ((s8, _), (s16, _)) in enumerate(zip(v8, v16)):
        assert s8 == s16, f"thread {t}: the chunk order depends on the batch size"
        assert [c for _, c in s8] == sorted(c for _, c in s8)
        for m, c in s8:
            assert m == t // (B // M), "a chunk added by a thread of another row"
            seen[(m, c)] = seen.get((m, c), 0) + 1
    assert seen == {(m, c): 1 for m in range(M) for c in range(K // 8)}


@pytest.mark.parametrize("M", range(1, 9))
def test_one_round_trip_for_x_at_the_headline_width(M):
    # the K-slice kernel at K = 2560: 10 compute warps + the epilogue warp
    assert max(b for _, b in visits(M, 2560, 352, 8)) == 1
    # two batches only once a thread owns more than 8 chunks
    worst = -(-(2560 // 8) // (352 // M))
    assert worst <= 8


def test_two_round_trips_past_eight_chunks_per_thread():
    # K = 4096, M = 8 on 8 compute warps + the epilogue warp: 15 chunks per thread
    v = visits(8, 4096, 288, 8)
    assert max(len(s) for s, _ in v) == 15 and max(b for _, b in v) == 2
    assert max(b for _, b in visits(8, 4096, 288, 16)) == 1
