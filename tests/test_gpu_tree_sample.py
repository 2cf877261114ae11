"""GPU parity of token-tree sampling verification against the float64 oracle.

Paths, accepted counts and drawn tokens must be identical for every tree
whose oracle run met no decision within 1e-6 of its edge (an accept test with
|u - r/q| < 1e-6 or a draw within 1e-6 of an interval edge); such boundary
trees may differ in float32 and are counted, not compared.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_utils import lib, to_dev

pytestmark = pytest.mark.gpu


def run_gpu(case, ws=None, max_depth=None, logits=None):
    sv = lib()
    md = case.max_depth if max_depth is None else max_depth
    out = sv.spec_verify_tree_sample(to_dev(case.logits) if logits is None else logits, to_dev(case.draft),
                                     to_dev(case.node_tokens), to_dev(case.parents), to_dev(case.uniforms), md,
                                     temperature=case.temperature, workspace=ws)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def run_oracle(case, max_depth=None):
    md = case.max_depth if max_depth is None else max_depth
    return oracle.verify_tree_sample(case.logits, case.draft, case.node_tokens, case.parents, case.uniforms, md,
                                     temperature=case.temperature)


def compare(case, gpu, orc, max_boundary=0.05):
    tok, path, n = gpu
    boundary = (orc["flags"] & oracle.BOUNDARY_FLAGS) != 0
    bad = []
    for b in range(case.B):
        if boundary[b]:
            continue
        if n[b] != orc["n"][b] or not np.array_equal(tok[b], orc["tokens"][b]) or \
                not np.array_equal(path[b], orc["path"][b]):
            bad.append((b, int(n[b]), int(orc["n"][b]), tok[b].tolist(), orc["tokens"][b].tolist(),
                        path[b].tolist(), orc["path"][b].tolist(), float(orc["margin"][b])))
    assert not bad, f"{len(bad)} trees differ outside boundary decisions: {bad[:3]}"
    assert boundary.sum() <= max(1, max_boundary * case.B), int(boundary.sum())
    return int(boundary.sum())


@pytest.mark.parametrize("B,N,V,depth,dtype,noise,T", [
    (4, 12, 1000, 3, W.F32, 1.0, 1.0),
    (6, 30, 32000, 4, W.BF16, 1.0, 0.8),
    (3, 5, 7, 2, W.F32, 0.5, 1.0),          # V smaller than the cluster's slices
    (2, 1, 5000, 1, W.BF16, 1.0, 1.0),       # root only: a draw from p
    (5, 20, 100003, 5, W.F32, 1.5, 1.2),     # odd V: unaligned rows
    (16, 24, 4096, 6, W.BF16, 2.0, 0.7),     # far draft: many rejections among siblings
    (3, 40, 152064, 6, W.BF16, 1.0, 1.0),
])
def test_tree_sample_parity(B, N, V, depth, dtype, noise, T):
    case = W.tree_sample_case(B, N, V, depth, seed=B * 1000 + N, dtype=dtype, noise=noise, temperature=T)
    compare(case, run_gpu(case), run_oracle(case))


def test_tree_sample_parity_full_size():
    """8 trees of 60 nodes, depth <= 6, V = 128256, bf16.  One tree of this
    seeded batch ends with an unfiltered draw 3.7e-7 from its interval's edge
    (the oracle flags it); at most one boundary tree is allowed."""
    case = W.tree_sample_case(8, 60, 128256, 6, seed=4)
    assert compare(case, run_gpu(case), run_oracle(case)) <= 1


def test_tree_sample_many_small_trees():
    case = W.tree_sample_case(300, 16, 256, 4, seed=21, dtype=W.F32, noise=1.0)
    nb = compare(case, run_gpu(case), run_oracle(case), max_boundary=0.02)
    assert nb <= 6


def test_q_equal_p_accepts_first_children():
    case = W.tree_sample_case(6, 25, 3000, 4, seed=5, dtype=W.F32, noise=0.0)
    tok, path, n = run_gpu(case)
    orc = run_oracle(case)
    compare(case, (tok, path, n), orc)
    for b in range(case.B):  # every node accepts its first child: the path follows first children
        v = 0
        for d in range(n[b]):
            kids = np.nonzero(case.parents[b] == v)[0]
            kids = kids[kids > v]
            assert path[b, d] == kids[0]
            v = kids[0]


def test_status_bits_and_malformed_trees():
    sv = lib()
    case = W.tree_sample_case(4, 20, 500, 3, seed=6, dtype=W.F32)
    case.parents[0, 7] = 9            # forward pointer: node 7 and its subtree detached
    case.node_tokens[1, 3] = case.V + 2  # out of range: skipped
    case.parents[2, 0] = 0            # root must be -1
    ws = sv.Workspace()
    sv.spec_get_status(ws)
    gpu = run_gpu(case, ws=ws)
    st = sv.spec_get_status(ws)
    assert st & sv.SPEC_STATUS_BAD_PARENT and st & sv.SPEC_STATUS_BAD_TOKEN
    compare(case, gpu, run_oracle(case))
    # a depth limit of 1: children of depth-1 nodes are not tested
    gpu = run_gpu(case, ws=ws, max_depth=1)
    orc = run_oracle(case, max_depth=1)
    compare(case, gpu, orc)
    st = sv.spec_get_status(ws)
    assert bool(st & sv.SPEC_STATUS_DEPTH) == bool((orc["flags"] & oracle.FLAG_DEPTH).any())


def test_nonfinite_row_on_the_walk():
    sv = lib()
    case = W.tree_sample_case(3, 10, 800, 3, seed=7, dtype=W.F32)
    case.logits[:, 0, 5] = np.nan     # the root row of every tree
    ws = sv.Workspace()
    sv.spec_get_status(ws)
    tok, path, n = run_gpu(case, ws=ws)
    assert sv.spec_get_status(ws) & sv.SPEC_STATUS_BAD_ROW
    orc = run_oracle(case)
    assert (n == 0).all() and (tok[:, 0] == -1).all() and (orc["tokens"][:, 0] == -1).all()


def test_workspace_shared_with_other_entry_points():
    """Tree sampling leaves its work counts zeroed and the other entry points'
    regions untouched: chain sampling, greedy tree and tree sampling calls on
    one workspace all keep their parity."""
    from parity_utils import compare_sample, run_sample_gpu, run_sample_oracle

    sv = lib()
    ws = sv.Workspace()
    tcase = W.tree_sample_case(5, 30, 20000, 5, seed=8)
    scase = W.random_sample_case(5, 6, 20000, seed=8, top_p=0.9)
    gcase = W.random_tree_case(5, 30, 20000, 5, seed=8)
    for _ in range(2):
        compare(tcase, run_gpu(tcase, ws=ws), run_oracle(tcase))
        compare_sample(scase, run_sample_gpu(scase, workspace=ws), run_sample_oracle(scase))
        out = sv.spec_verify_tree_greedy(to_dev(gcase.logits), to_dev(gcase.node_tokens), to_dev(gcase.parents),
                                         gcase.max_depth, workspace=ws)
        o = oracle.verify_tree_greedy(gcase.logits, gcase.node_tokens, gcase.parents, gcase.max_depth)
        assert np.array_equal(out[0].cpu().numpy(), o["tokens"])


def test_repeat_calls_identical():
    case = W.tree_sample_case(8, 60, 32000, 6, seed=9)
    a = run_gpu(case)
    b = run_gpu(case)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def _custom_case(parents, V, seed, dtype=W.F32, noise=1.5, T=1.0, max_depth=None):
    """A tree with the given parent arrays [B][N]; rows and tokens as in
    tree_sample_case (children drawn from their parents' draft rows)."""
    parents = np.asarray(parents, np.int32)
    B, N = parents.shape
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 3.0, size=(B, N, V)).astype(np.float32)
    d = (x + rng.normal(0.0, noise, size=x.shape)).astype(np.float32)
    logits = W.bf16_bits(x) if dtype == W.BF16 else x
    draft = W.bf16_bits(d) if dtype == W.BF16 else d
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        rows = W.as_f32(draft[b]).astype(np.float64) / T
        for j in range(1, N):
            g = -np.log(-np.log(rng.random(V).clip(1e-300, None)))
            tokens[b, j] = int(np.argmax(rows[parents[b, j]] + g))
    depth = max_depth
    if depth is None:
        dep = np.zeros((B, N), int)
        for b in range(B):
            for j in range(1, N):
                dep[b, j] = dep[b, parents[b, j]] + 1
        depth = max(1, int(dep.max()))
    return W.TreeSampleCase("custom", dtype, logits, draft, tokens, parents,
                            rng.random((B, N), dtype=np.float32), depth, T, seed)


def test_many_siblings_past_the_prefetched_ones():
    """A root with 70 children (only the first 32 have their logits fetched
    ahead) and a far draft, so that many siblings are rejected in turn."""
    N = 71
    par = np.tile(np.array([-1] + [0] * (N - 1), np.int32), (6, 1))
    case = _custom_case(par, 2000, seed=31, noise=4.0)
    case.uniforms[:, 1:] = np.float32(0.999)  # reject nearly every child
    compare(case, run_gpu(case), run_oracle(case))


def test_deep_chain_tree():
    """A chain of 200 nodes: a depth walk of up to 199 steps per node."""
    N = 200
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (3, 1))
    case = _custom_case(par, 512, seed=32, dtype=W.BF16, noise=0.05)
    compare(case, run_gpu(case), run_oracle(case))


def test_unaligned_pointers():
    sv = lib()
    case = W.tree_sample_case(4, 20, 4000, 4, seed=33, dtype=W.BF16)
    flat = np.concatenate([np.zeros(1, np.uint16), case.logits.ravel()])
    L = to_dev(flat)[1:].view(case.logits.shape)
    assert L.data_ptr() % 16 != 0
    compare(case, run_gpu(case, logits=L), run_oracle(case))


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_masked_vocabulary(dtype):
    """-inf logits in both rows (30% of tokens, and whole chunks of some rows)."""
    case = W.tree_sample_case(6, 24, 20000, 4, seed=34, dtype=W.F32, noise=1.0)
    rng = np.random.default_rng(35)
    L, Dr = case.logits.copy(), case.draft.copy()
    for arr in (L, Dr):
        arr[rng.random(arr.shape) < 0.3] = -np.inf
        arr[:, ::3, 2000:9000] = -np.inf
        arr[:, :, 0] = 0.0
    if dtype == W.BF16:
        L, Dr = W.bf16_bits(L), W.bf16_bits(Dr)
    case = W.TreeSampleCase("masked", dtype, L, Dr, case.node_tokens, case.parents, case.uniforms,
                            case.max_depth, case.temperature, case.seed)
    compare(case, run_gpu(case), run_oracle(case))


def test_maximum_tree_size():
    """N = 1024 nodes (the limit), up to 4 children per node, depth <= 12."""
    case = W.tree_sample_case(2, 1024, 2048, 12, seed=36, dtype=W.BF16, noise=0.7)
    compare(case, run_gpu(case), run_oracle(case))


def test_per_tree_temperatures():
    sv = lib()
    case = W.tree_sample_case(8, 30, 20000, 5, seed=37, dtype=W.BF16)
    temps = np.random.default_rng(38).uniform(0.5, 1.2, size=case.B).astype(np.float32)
    temps[5] = 0.0  # no distribution: that tree ends at its root
    ws = sv.Workspace()
    sv.spec_get_status(ws)
    out = sv.spec_verify_tree_sample(to_dev(case.logits), to_dev(case.draft), to_dev(case.node_tokens),
                                     to_dev(case.parents), to_dev(case.uniforms), case.max_depth,
                                     temperature_per_tree=to_dev(temps), workspace=ws)
    torch.cuda.synchronize()
    gpu = [o.cpu().numpy() for o in out]
    assert sv.spec_get_status(ws) & sv.SPEC_STATUS_BAD_ROW
    orc = oracle.verify_tree_sample(case.logits, case.draft, case.node_tokens, case.parents, case.uniforms,
                                    case.max_depth, temperature_per_tree=temps)
    compare(case, gpu, orc)
    assert gpu[2][5] == 0 and gpu[0][5, 0] == -1


def test_degenerate_residual_goes_back_to_p():
    """p = q = (1, 0) at the root; the first child's token has no mass, its
    rejection leaves a residual of mass 0, which goes back to p: the second
    child (token 0) is accepted for any u, then the leaf's (.5, .5) row is
    drawn with u_0 = 0.3 (token 0).  Oracle-flagged as degenerate, so the
    outcome is checked here directly."""
    B = 4
    P = np.tile(np.array([[[0.0, -np.inf], [0.0, 0.0], [0.0, 0.0]]], np.float32), (B, 1, 1))
    toks = np.tile(np.array([[0, 1, 0]], np.int32), (B, 1))
    par = np.tile(np.array([[-1, 0, 0]], np.int32), (B, 1))
    u = np.array([[0.3, 0.2, x] for x in (0.0, 0.5, 0.9, 0.999)], np.float32)
    case = W.TreeSampleCase("degenerate", W.F32, P, P.copy(), toks, par, u, 1, 1.0)
    tok, path, n = run_gpu(case)
    orc = run_oracle(case)
    assert (orc["flags"] & oracle.FLAG_DEGENERATE).all()
    np.testing.assert_array_equal(n, orc["n"])
    np.testing.assert_array_equal(tok, orc["tokens"])
    np.testing.assert_array_equal(path, orc["path"])
    assert (n == 1).all() and (path[:, 0] == 2).all() and (tok[:, :2] == 0).all()
