"""GPU parity of the KV keep list (spec_kv_compact) against the oracle.

Bit-exact: every (src, dst) slot, the new length, the move count and which
sequences are left out as malformed must equal the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_utils import lib, to_dev

pytestmark = pytest.mark.gpu


def _gpu(case, status=None):
    sv = lib()
    out = sv.spec_kv_compact(to_dev(case.num_accepted), to_dev(case.kv_base),
                             to_dev(case.path) if case.path is not None else None,
                             to_dev(case.block_table) if case.block_table is not None else None,
                             case.block_size, case.max_keep, out_status=status)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def _compare(case, status=None):
    g = _gpu(case, status)
    src, dst, nl, mv, bad = oracle.kv_compact(case.num_accepted, case.kv_base, case.path, case.block_table,
                                              case.block_size, case.max_keep)
    for name, a, b in zip(("src", "dst", "new_len", "moves"), g, (src, dst, nl, mv)):
        assert np.array_equal(a, b), (name, np.nonzero(a != b)[0][:8])
    return bad


CASES = [
    # (B, N, max_depth, chain, block_size)
    (1, 2, 1, False, 0),
    (8, 60, 6, False, 0),
    (8, 60, 6, False, 16),
    (64, 9, 8, True, 0),
    (256, 13, 12, True, 16),
    (37, 1024, 100, False, 0),     # paths of several 32-entry sweeps
    (37, 1024, 100, False, 1),
    (1000, 48, 8, False, 64),
]


@pytest.mark.parametrize("B,N,max_depth,chain,block_size", CASES)
def test_kv_compact_parity(B, N, max_depth, chain, block_size):
    case = W.kv_case(B, N, max_depth, seed=B + N, chain=chain, block_size=block_size)
    assert not _compare(case).any()


def test_kv_compact_malformed_sequences():
    case = W.kv_case(96, 200, 70, seed=5, block_size=8)
    rng = np.random.default_rng(1)
    n = case.num_accepted
    for b in range(0, 96, 6):
        kind = (b // 6) % 8
        if kind == 0 and n[b] >= 2:
            case.path[b, n[b] - 1] = case.path[b, n[b] - 2]        # not increasing
        elif kind == 1 and n[b] >= 33:
            case.path[b, 32] = case.path[b, 31]                     # across a 32-entry sweep
        elif kind == 2:
            n[b] = case.max_keep                                    # n + 1 > max_keep
        elif kind == 3:
            n[b] = -2
        elif kind == 4:
            case.kv_base[b] = -1
        elif kind == 5:
            case.block_table[b, int(case.kv_base[b]) // 8] = -4     # the root's block is missing
        elif kind == 6 and n[b] >= 1:
            case.path[b, 0] = 0                                     # the root again
        elif kind == 7:
            case.kv_base[b] = 2**31 - 2                              # positions past INT32_MAX
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = _compare(case, status)
    assert bad.any()
    assert int(status.item()) == lib().SPEC_STATUS_BAD_KV


def test_tree_verify_then_kv_compact():
    """The tree verification's own outputs (path, n) feed the keep list on the
    device; the oracle takes its own verification's path."""
    sv = lib()
    case = W.random_tree_case(16, 60, 4000, 6, seed=12)
    tok, path, n = sv.spec_verify_tree_greedy(to_dev(case.logits), to_dev(case.node_tokens),
                                              to_dev(case.parents), case.max_depth)
    base = (np.arange(16, dtype=np.int32) * 97) % 1000
    table = np.random.default_rng(2).permutation(16 * 20).astype(np.int32).reshape(16, 20)
    g = sv.spec_kv_compact(n, to_dev(base), path, to_dev(table), 64)
    torch.cuda.synchronize()
    o = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, case.max_depth)
    ref = oracle.kv_compact(o["n"], base, o["path"], table, 64)
    for a, b in zip(g, ref[:4]):
        assert np.array_equal(a.cpu().numpy(), b)
