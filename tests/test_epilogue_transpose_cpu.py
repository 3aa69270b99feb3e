"""The GEMM epilogues' whole-row store (epilogue.cuh store_rows64) moves a
warp's 32 rows x 64 bytes through two rounds of shuffles so that each 32-byte
store instruction covers whole 64-byte runs of 16 rows.  This models the
warp on the CPU, lane by lane and round by round, and checks that every
(row, piece) of every instruction carries exactly the words its row holds
there: a wrong source lane, word offset or destination slot in the exchange
fails it.  Runs without a GPU."""
import numpy as np


def exchange(w):
    """w[lane][16]: lane l's words of row l (two 8-word pieces).  Returns
    o[lane][2][8] after the two rounds, following the kernel's index rules:
    lane l stores piece l % 2 of row 16 s + l / 2 in instruction s; in round
    a it reads from lane 16 (a ^ piece) + rsub, which sends word 8 + k when
    (its own s ^ a) != 0, else word k, and keeps it in o[a ^ piece][k]."""
    o = np.full((32, 2, 8), -1, dtype=np.int64)
    for a in range(2):
        for k in range(8):
            sent = [w[u][8 + k] if ((u >> 4) ^ a) != 0 else w[u][k] for u in range(32)]
            for lane in range(32):
                piece, rsub = lane & 1, lane >> 1
                src = 16 * (a ^ piece) + rsub
                o[lane][a ^ piece][k] = sent[src]
    return o


def test_every_row_piece_reaches_its_store():
    rng = np.random.default_rng(5)
    w = rng.integers(0, 2**32, size=(32, 16), dtype=np.int64)
    o = exchange(w)
    stored = {}
    for s in range(2):
        for lane in range(32):
            piece, rsub = lane & 1, lane >> 1
            row = 16 * s + rsub
            assert (row, piece) not in stored
            stored[(row, piece)] = o[lane][s]
    assert len(stored) == 64                      # 32 rows x 2 pieces, each once
    for (row, piece), words in stored.items():
        np.testing.assert_array_equal(words, w[row][8 * piece: 8 * piece + 8])


def test_each_round_reads_32_distinct_lanes():
    # a round moves 32 distinct words per word index: no two lanes read the
    # same source lane (no word is broadcast, none is lost)
    for a in range(2):
        srcs = {16 * (a ^ (lane & 1)) + (lane >> 1) for lane in range(32)}
        assert srcs == set(range(32))


def test_instruction_covers_whole_runs():
    # each store instruction writes 16 rows x 2 pieces: two lanes per row,
    # adjacent 32-byte pieces, so every row's 64 bytes go out together
    for s in range(2):
        rows = {}
        for lane in range(32):
            rows.setdefault(16 * s + (lane >> 1), set()).add(lane & 1)
        assert len(rows) == 16 and all(p == {0, 1} for p in rows.values())
