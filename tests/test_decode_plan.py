"""The paged decode's work split, checked on the CPU against its stated rules.

The split kernel lays every (request, KV head, 16-token block) triple of the batch
in one request-major sequence of NB blocks and cuts it into W equal ranges, one
per consumer warp: W = min(4 * grid, NB // 16) (at least 1), range k = blocks
[k NB // W, (k + 1) NB // W).  The range holding block b is
k(b) = ((b + 1) W - 1) // NB.  Wherever a range leaves a (request, KV head)
segment it ends a piece; piece j of a segment is range k(first block) + j.  The
workspace holds ceil(max_seq_len / 256) + 1 pieces per (request, query head), and
the merge reads pieces 0 .. k(last) - k(first) of each segment.

These tests walk that rule over random batches and check what the kernels rely
on: every block is read by exactly one range, the pieces of a segment are
numbered 0, 1, 2, ... without gaps, and no segment needs more pieces than the
workspace holds.  (The GPU tests check the kernels' results against the oracle.)
"""

from __future__ import annotations

import math
import random

import pytest

BS = 16           # tokens per block
MIN_BLOCKS = 16   # shortest range: 256 tokens
WARPS_PER_CTA = 4


def blocks_of(L: int, max_seq_len: int, max_blocks: int) -> int:
    if L < 0 or L > max_seq_len or L > max_blocks * BS:
        return 0
    return (L + BS - 1) // BS


def range_of(b: int, NB: int, W: int) -> int:
    return ((b + 1) * W - 1) // NB


def max_pieces(max_seq_len: int) -> int:
    return math.ceil(math.ceil(max_seq_len / BS) / MIN_BLOCKS) + 1


def split(lens, Hkv, max_seq_len, max_blocks, grid):
    """Per range: the list of (request, head, block) it reads, in order."""
    nbl = [blocks_of(L, max_seq_len, max_blocks) for L in lens]
    seq = [(r, h, b) for r in range(len(lens)) for h in range(Hkv) for b in range(nbl[r])]
    NB = len(seq)
    if NB == 0:
        return NB, 0, []
    W = max(1, min(WARPS_PER_CTA * grid, NB // MIN_BLOCKS))
    return NB, W, [seq[k * NB // W:(k + 1) * NB // W] for k in range(W)]


def check_batch(lens, Hkv, max_seq_len, max_blocks, grid):
    NB, W, ranges = split(lens, Hkv, max_seq_len, max_blocks, grid)
    seen = {}
    pieces = {}  # segment -> {piece index: range}
    first_block = {}
    pos = 0
    for r in range(len(lens)):
        nb = blocks_of(lens[r], max_seq_len, max_blocks)
        for h in range(Hkv):
            if nb:
                first_block[(r, h)] = pos
            pos += nb
    for k, rng in enumerate(ranges):
        assert len(rng) >= min(MIN_BLOCKS, NB)   # ranges never shorter than the minimum
        for item in rng:
            assert item not in seen
            seen[item] = k
        for r, h, _ in rng:
            j = k - range_of(first_block[(r, h)], NB, W)
            pieces.setdefault((r, h), set()).add(j)
    assert len(seen) == NB
    for (r, h), js in pieces.items():
        nb = blocks_of(lens[r], max_seq_len, max_blocks)
        first = first_block[(r, h)]
        ns = range_of(first + nb - 1, NB, W) - range_of(first, NB, W) + 1
        assert js == set(range(ns))                 # the merge reads exactly these
        assert ns <= max_pieces(max_seq_len)        # and the workspace holds them


def test_range_of_finds_the_range_holding_each_block():
    rnd = random.Random(1)
    for _ in range(2000):
        NB = rnd.randint(1, 10 ** 6)
        W = rnd.randint(1, min(NB, 4096))
        b = rnd.randrange(NB)
        k = range_of(b, NB, W)
        assert k * NB // W <= b < (k + 1) * NB // W


@pytest.mark.parametrize("seed", range(40))
def test_split_covers_every_block_once_and_fits_the_workspace(seed):
    rnd = random.Random(seed)
    S = rnd.randint(1, 120)
    Hkv = rnd.choice([1, 2, 4, 8])
    max_seq_len = rnd.randint(1, 12000)
    max_blocks = (max_seq_len + BS - 1) // BS + rnd.randint(0, 2)
    lens = [rnd.choice([0, 1, 15, 16, 17, rnd.randint(0, max_seq_len), max_seq_len,
                        max_seq_len + 1, -1]) for _ in range(S)]
    check_batch(lens, Hkv, max_seq_len, max_blocks, grid=rnd.choice([1, 7, 304, 456]))


def test_split_of_the_decode_workload():
    rnd = random.Random(5000)
    lens = [rnd.randint(512, 8192) for _ in range(64)]
    check_batch(lens, 2, 8192, 512, grid=456)


def test_one_long_request_on_a_full_grid():
    # 2 heads x 1024 blocks over up to 1824 warps: 128 ranges of 16 blocks, 65 pieces
    check_batch([16384], 2, 16384, 1024, grid=456)
    _, W, _ = split([16384], 2, 16384, 1024, 456)
    assert W == 128 and max_pieces(16384) == 65
