"""Pins of the oracle's KV keep list (the cut-back cache after verification).

"Towards Green Text Generation: Memory-Based Speculative Decoding", section
2.4 (KV-cached regime: on rejection the cache is cut back to the accepted
prefix), and Edge Inference Notes, "One decode round, end to end" (the
longest agreed path is committed, the other branches collapse).  The pins
do not restate the oracle's formulas: a simulated cache pool, filled with a
tag per (sequence, node) and moved entry by entry as the list says, must
read back the root and the path in order; worked examples are written out
by hand; and the paths of the oracle's own tree verification feed it.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def _simulate(case, src, dst, new_len):
    """Fill a pool with tags, apply the moves in list order, and return what
    each sequence reads at its logical positions base .. new_len - 1."""
    B, N = len(case.num_accepted), case.entries

    def phys(b, pos):
        if case.block_table is None:
            return (b, pos)  # a separate logical cache per sequence
        return case.block_table[b][pos // case.block_size] * case.block_size + pos % case.block_size

    pool = {}
    for b in range(B):
        for j in range(N):
            pool[phys(b, int(case.kv_base[b]) + j)] = (b, j)
    for b in range(B):
        for d in range(case.max_keep):
            if src[b, d] < 0:
                break
            s = (b, int(src[b, d])) if case.block_table is None else int(src[b, d])
            t = (b, int(dst[b, d])) if case.block_table is None else int(dst[b, d])
            pool[t] = pool[s]
    return [[pool[phys(b, p)] for p in range(int(case.kv_base[b]), int(new_len[b]))] for b in range(B)]


@pytest.mark.parametrize("chain,block_size", [(False, 0), (False, 16), (True, 0), (True, 8), (False, 1)])
def test_moved_cache_reads_back_root_then_path(chain, block_size):
    case = W.kv_case(40, 60 if not chain else 9, 6 if not chain else 8, seed=3, chain=chain,
                     block_size=block_size)
    src, dst, new_len, moves, bad = oracle.kv_compact(case.num_accepted, case.kv_base, case.path,
                                                       case.block_table, case.block_size, case.max_keep)
    assert not bad.any()
    got = _simulate(case, src, dst, new_len)
    for b in range(len(got)):
        n = int(case.num_accepted[b])
        kept = [0] + (list(case.path[b, :n]) if case.path is not None else list(range(1, n + 1)))
        assert got[b] == [(b, int(j)) for j in kept]
        assert new_len[b] == case.kv_base[b] + n + 1
        assert moves[b] == int(np.sum(src[b] != dst[b]))  # entries that change slot
        if chain:
            assert moves[b] == 0 and np.array_equal(src[b], dst[b])


def test_worked_example_flat_and_paged():
    # tree path root -> node 2 -> node 5 written from position 100
    src, dst, nl, mv, bad = oracle.kv_compact([2], [100], np.array([[2, 5, -1]]))
    assert src[0].tolist() == [100, 102, 105, -1] and dst[0].tolist() == [100, 101, 102, -1]
    assert nl[0] == 103 and mv[0] == 2 and not bad[0]
    # paged: blocks of 4, logical blocks 0, 1, 2 -> physical 7, 3, 9; root at position 2, path 1, 3, 6
    src, dst, nl, mv, bad = oracle.kv_compact([3], [2], np.array([[1, 3, 6]]), np.array([[7, 3, 9]]), 4)
    assert src[0].tolist() == [30, 31, 13, 36]
    assert dst[0].tolist() == [30, 31, 12, 13]
    assert nl[0] == 6 and mv[0] == 2
    # a chain keeps its prefix where it is: only the length changes
    src, dst, nl, mv, bad = oracle.kv_compact([2], [10], None, max_keep=5)
    assert src[0].tolist() == [10, 11, 12, -1, -1] == dst[0].tolist() and nl[0] == 13 and mv[0] == 0


def test_paths_of_tree_verification():
    """The oracle's greedy tree verification hands a path that kv_compact
    keeps: every kept node's parent is the entry before it."""
    case = W.random_tree_case(6, 40, 300, 5, seed=9)
    o = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, case.max_depth)
    base = np.arange(6, dtype=np.int32) * 50
    src, dst, nl, mv, bad = oracle.kv_compact(o["n"], base, o["path"])
    assert not bad.any()
    for b in range(6):
        n = int(o["n"][b])
        kept = (src[b, :n + 1] - base[b]).tolist()
        assert kept[0] == 0
        for d in range(1, n + 1):
            assert case.parents[b, kept[d]] == kept[d - 1]
        assert dst[b, :n + 1].tolist() == list(range(base[b], base[b] + n + 1))


@pytest.mark.parametrize("what", ["not_increasing", "root_repeated", "n_too_big", "negative_n", "no_block",
                                  "negative_block", "negative_base"])
def test_bad_sequences_left_out(what):
    path = np.array([[1, 4, 9, -1], [2, 3, -1, -1]], np.int32)
    n = np.array([3, 2], np.int32)
    base = np.array([0, 20], np.int32)
    table, bs = None, 0
    if what == "not_increasing":
        path[0, 2] = 4
    elif what == "root_repeated":
        path[0, 0] = 0
    elif what == "n_too_big":
        n[0] = 5
    elif what == "negative_n":
        n[0] = -1
    elif what == "negative_base":
        base[0] = -3
    elif what in ("no_block", "negative_block"):
        table, bs = np.array([[0, 1, 6], [2, 5, 7]], np.int32), 8  # sequence 0 reaches position 9: block 1
        if what == "no_block":
            table = np.array([[0], [2]], np.int32)  # sequence 0 needs a second block
            base[1] = 0
        else:
            table[0, 1] = -1
    src, dst, nl, mv, bad = oracle.kv_compact(n, base, path, table, bs, 5)
    assert bad.tolist() == [True, False]
    assert (src[0] == -1).all() and (dst[0] == -1).all() and nl[0] == -1 and mv[0] == 0
    assert nl[1] == base[1] + 3 and src[1, :3].tolist() != [-1, -1, -1]
