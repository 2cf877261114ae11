"""GPU parity of greedy chain and greedy token-tree verification: bit-exact
against the float64 oracle (argmax ties to the lowest index, deepest agreed
node ties to the lowest node index)."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity_utils import lib, run_greedy_gpu, run_tree_gpu, to_dev

pytestmark = pytest.mark.gpu


def _greedy_case(B, k, V, dtype, seed, quantize=None, agree=0.7):
    case = W.random_sample_case(B, k, V, dtype=dtype, seed=seed, quantize=quantize)
    am = np.argmax(W.as_f32(case.target), axis=-1)
    rng = np.random.default_rng(seed)
    tokens = case.tokens.copy()
    for b in range(B):  # long agreeing prefixes, so every n in [0, k] occurs
        for i in range(k):
            if rng.random() < agree:
                tokens[b, i] = am[b, i]
            else:
                break
    return case.target, tokens


@pytest.mark.parametrize("B,k,V,dtype,quantize", [
    (1, 4, 32000, W.F32, None), (16, 5, 32000, W.BF16, None), (64, 8, 128256, W.BF16, None),
    (7, 3, 1, W.BF16, None), (9, 2, 7, W.F32, None), (5, 31, 33, W.BF16, 1.0), (12, 6, 1001, W.BF16, 0.5),
    (4, 12, 152064, W.BF16, None), (256, 1, 152064, W.BF16, None), (3, 4, 100003, W.F32, 1.0),
    # aligned rows of a few vectors (many row pieces per CTA) and rows one vector past a
    # shared-memory stage (a chunk cut at every row's end)
    (40, 3, 64, W.BF16, 1.0), (33, 7, 4104, W.BF16, 1.0), (10, 2, 2052, W.F32, 0.5), (2, 3, 8, W.BF16, None),
])
def test_greedy_parity(B, k, V, dtype, quantize):
    target, tokens = _greedy_case(B, k, V, dtype, seed=B * 100 + k, quantize=quantize)
    got_tok, got_n = run_greedy_gpu(target, tokens)
    o = oracle.verify_greedy(target, tokens)
    assert np.array_equal(got_n, o["n"])
    assert np.array_equal(got_tok, o["tokens"])


def test_greedy_all_equal_and_signed_zero_ties():
    B, k, V = 3, 2, 4000
    target = np.zeros((B, k + 1, V), np.float32)
    target[0, :, :] = -0.0
    target[0, :, 1000] = 0.0      # +0 and -0 tie: lowest index wins (index 0)
    target[1, :, 3999] = 1.0      # unique max at the end
    target[2, :, :] = -np.inf
    target[2, :, 77] = -5.0
    tokens = np.array([[0, 0], [3999, 5], [77, 77]], np.int32)
    for arr in (target, W.bf16_bits(target)):
        got_tok, got_n = run_greedy_gpu(arr, tokens)
        o = oracle.verify_greedy(arr, tokens)
        assert np.array_equal(got_tok, o["tokens"]) and np.array_equal(got_n, o["n"])


def test_greedy_unaligned_rows():
    target, tokens = _greedy_case(6, 4, 5000, W.BF16, seed=1)
    flat = np.concatenate([np.zeros(3, np.uint16), target.ravel()])
    t = to_dev(flat)[3:].view(target.shape)
    assert t.data_ptr() % 16 != 0
    tok, n = lib().spec_verify_greedy(t, to_dev(tokens))
    o = oracle.verify_greedy(target, tokens)
    assert np.array_equal(tok.cpu().numpy(), o["tokens"]) and np.array_equal(n.cpu().numpy(), o["n"])


def test_config4_tree_full_size():
    case = W.config4()
    got_tok, got_path, got_n = run_tree_gpu(case)
    o = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, case.max_depth)
    assert np.array_equal(got_n, o["n"])
    assert np.array_equal(got_path, o["path"])
    assert np.array_equal(got_tok, o["tokens"])
    assert o["n"].max() >= 2  # the 0.6 agreement rule gives real paths


@pytest.mark.parametrize("B,N,V,depth,dtype,quantize,children", [
    (5, 1, 100, 1, W.BF16, None, 4), (7, 2, 9, 1, W.F32, None, 4), (6, 40, 50, 6, W.BF16, 1.0, 4),
    (4, 1024, 300, 12, W.BF16, 1.0, 3), (3, 200, 20000, 8, W.F32, None, 2), (8, 60, 128256, 6, W.BF16, 2.0, 4),
    (5, 100, 64, 6, W.BF16, 1.0, 4), (3, 30, 4104, 6, W.F32, 1.0, 3),
])
def test_tree_parity(B, N, V, depth, dtype, quantize, children):
    case = W.random_tree_case(B, N, V, depth, seed=N + V, dtype=dtype, quantize=quantize, max_children=children)
    got_tok, got_path, got_n = run_tree_gpu(case)
    o = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, case.max_depth)
    assert np.array_equal(got_n, o["n"]) and np.array_equal(got_path, o["path"])
    assert np.array_equal(got_tok, o["tokens"])


def test_tree_bad_parents_and_depth_limit_status():
    sv = lib()
    case = W.random_tree_case(3, 30, 64, 6, seed=4, quantize=1.0, p_match=1.0)
    case.parents[0, 7] = 9          # forward pointer
    case.parents[1, 0] = 0          # root must be -1
    ws = sv.Workspace()
    sv.spec_get_status(ws)
    out = sv.spec_verify_tree_greedy(to_dev(case.logits), to_dev(case.node_tokens), to_dev(case.parents),
                                     case.max_depth, workspace=ws)
    st = sv.spec_get_status(ws)
    assert st & sv.SPEC_STATUS_BAD_PARENT
    o = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, case.max_depth)
    assert np.array_equal(out[2].cpu().numpy(), o["n"])
    assert np.array_equal(out[0].cpu().numpy(), o["tokens"])
    # a depth limit below the tree's depth: agreed nodes deeper than it are ignored
    out = sv.spec_verify_tree_greedy(to_dev(case.logits), to_dev(case.node_tokens), to_dev(case.parents), 2,
                                     workspace=ws)
    o = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, 2)
    assert np.array_equal(out[2].cpu().numpy(), o["n"]) and np.array_equal(out[0].cpu().numpy(), o["tokens"])
    assert sv.spec_get_status(ws) & sv.SPEC_STATUS_DEPTH


@pytest.mark.parametrize("B,V,dtype,quantize", [(1, 1, W.BF16, None), (7, 33, W.F32, None), (64, 128256, W.BF16, None),
                                                (32, 5000, W.BF16, 1.0), (16, 20000, W.F32, 2.0)])
def test_first_draft_check_parity(B, V, dtype, quantize):
    rng = np.random.default_rng(B * 7 + V)
    x = rng.normal(0.0, 3.0, size=(B, V)).astype(np.float32)
    if quantize:
        x = np.round(x / quantize) * quantize
    rows = W.bf16_bits(x) if dtype == W.BF16 else x
    o0 = oracle.first_draft_check(rows, np.zeros(B, np.int32))
    # about half the drafts are the argmax
    draft0 = np.where(rng.random(B) < 0.5, o0["argmax"], rng.integers(0, V, B)).astype(np.int32)
    o = oracle.first_draft_check(rows, draft0)
    acc, am = lib().spec_first_draft_check(to_dev(rows), to_dev(draft0))
    assert np.array_equal(am.cpu().numpy(), o["argmax"])
    assert np.array_equal(acc.cpu().numpy(), o["accept"])
