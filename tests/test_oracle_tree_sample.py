"""Pins for the token-tree sampling oracle (oracle_verify_tree_sample).

* the exact sibling law (oracle/exact.py) gives the target law for the first
  committed token when a node's children are independent draws from q, for
  any q (Edge Inference Notes, "Why it changes nothing about the output");
  a plausible mistake (the residual not updated between siblings) does not;
* the C oracle's accept thresholds and residual draws, probed through the
  uniforms, sit where that exact law puts them;
* a tree that is a chain gives what the chain oracle gives;
* a hand-worked three-token example;
* structure: depth limit, malformed parents, out-of-range tokens, non-finite
  rows; every output path is a root path of the tree.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import exact
import workloads as W


def _rand_dist(rng, V, zero=False):
    w = [Fraction(int(x)) for x in rng.integers(1, 20, size=V)]
    if zero:
        w[int(rng.integers(0, V))] = Fraction(0)
    s = sum(w)
    return [x / s for x in w]


# ------------------------------------------------------------ exact sibling law


@pytest.mark.parametrize("V,k,seed", [(2, 1, 0), (3, 2, 1), (3, 3, 2), (4, 2, 3), (4, 3, 4)])
def test_sibling_law_keeps_target_law(V, k, seed):
    rng = np.random.default_rng(seed)
    for trial in range(3):
        p = _rand_dist(rng, V, zero=(trial == 1))
        q = _rand_dist(rng, V, zero=(trial == 2))
        law = exact.first_token_law(p, q, k)
        assert sum(law.values()) == 1
        for t in range(V):
            assert law.get(t, Fraction(0)) == p[t], (p, q, k, t)


def test_sibling_law_q_equal_p_accepts_first_child():
    p = [Fraction(1, 2), Fraction(1, 3), Fraction(1, 6)]
    for toks in ([0, 1], [2, 2], [1]):
        assert exact.sibling_law(p, p, toks) == {("accept", 0): Fraction(1)}


def test_target_law_check_catches_a_stale_residual():
    """Testing every sibling against p itself (no residual update) breaks the law."""
    p = [Fraction(1, 2), Fraction(3, 10), Fraction(1, 5)]
    q = [Fraction(1, 5), Fraction(1, 2), Fraction(3, 10)]

    def stale(toks):
        law, reach = {}, Fraction(1)
        for j, x in enumerate(toks):
            a = min(Fraction(1), p[x] / q[x])
            law[("accept", j)] = reach * a
            reach *= 1 - a
        res = [max(Fraction(0), a - b) for a, b in zip(p, q)]
        s = sum(res)
        for t in range(3):
            if res[t]:
                law[("draw", t)] = law.get(("draw", t), Fraction(0)) + reach * res[t] / s
        return law

    out = {}
    for toks in [(a, b) for a in range(3) for b in range(3)]:
        pr = q[toks[0]] * q[toks[1]]
        for (kind, idx), m in stale(toks).items():
            t = toks[idx] if kind == "accept" else idx
            out[t] = out.get(t, Fraction(0)) + pr * m
    assert [out.get(t, 0) for t in range(3)] != p


# ------------------------------------------- C oracle against the exact law


def _star(V, k, seed, temperature=1.0):
    """Root with k leaf children; f32 logits; distributions as the oracle sees them."""
    rng = np.random.default_rng(seed)
    L = rng.normal(0.0, 1.0, size=(1, k + 1, V)).astype(np.float32)
    D = (L + rng.normal(0.0, 1.0, size=L.shape)).astype(np.float32)
    p = oracle.row_probs(L[0, 0], temperature)[0]
    q = oracle.row_probs(D[0, 0], temperature)[0]
    par = np.array([[-1] + [0] * k], np.int32)
    return L, D, par, p, q


def _run(L, D, toks, par, u, max_depth=2, temperature=1.0):
    return oracle.verify_tree_sample(L, D, toks, par, np.asarray(u, np.float32)[None], max_depth,
                                     temperature=temperature)


@pytest.mark.parametrize("seed", range(6))
def test_oracle_thresholds_match_sibling_law(seed):
    V, k = 6, 3
    L, D, par, p, q = _star(V, k, seed)
    rng = np.random.default_rng(100 + seed)
    toks_list = [int(x) for x in rng.integers(0, V, size=k)]
    toks = np.array([[0] + toks_list], np.int32)
    P = [Fraction(float(x)) for x in p]
    Q = [Fraction(float(x)) for x in q]
    law = exact.sibling_law(P, Q, toks_list)
    reach = Fraction(1)
    rejected = [0.9999999] * k
    for j in range(k):
        acc = law.get(("accept", j), Fraction(0))
        a = float(acc / reach) if reach else 0.0
        u = [0.5] + rejected[:j] + [0.0] * (k - j)
        if 1e-4 < a < 1 - 1e-4:
            u[1 + j] = a - 2e-5
            out = _run(L, D, toks, par, u)
            assert out["n"][0] == 1 and out["path"][0, 0] == 1 + j, (j, a)
            u[1 + j] = a + 2e-5
            out = _run(L, D, toks, par, u)
            assert not (out["n"][0] == 1 and out["path"][0, 0] == 1 + j), (j, a)
        if a >= 1 - 1e-4:
            return  # child j is (almost) always accepted: later siblings unreachable
        reach -= acc
    # every child rejected: the draw follows the exact residual
    r = [float(law.get(("draw", t), Fraction(0)) / reach) for t in range(V)]
    cdf = np.cumsum([0.0] + r)
    for t in range(V):
        if r[t] > 1e-4:
            u = [float(cdf[t] + r[t] / 2)] + rejected
            out = _run(L, D, toks, par, u)
            assert out["n"][0] == 0 and out["tokens"][0, 0] == t, (t, r)
            assert not (out["flags"][0] & (oracle.FLAG_ACCEPT_BOUNDARY | oracle.FLAG_DRAW_BOUNDARY))


def test_oracle_first_token_law_monte_carlo():
    """Children drawn from q, uniforms uniform: the first token follows p (chi-square)."""
    from scipy import stats

    V, k, S = 5, 3, 40000
    L, D, par, p, q = _star(V, k, 11)
    rng = np.random.default_rng(12)
    toks = np.zeros((S, k + 1), np.int32)
    toks[:, 1:] = rng.choice(V, size=(S, k), p=q / q.sum())
    u = rng.random((S, k + 1), dtype=np.float32)
    Ls = np.broadcast_to(L, (S, k + 1, V)).copy()
    Ds = np.broadcast_to(D, (S, k + 1, V)).copy()
    pars = np.broadcast_to(par, (S, k + 1)).copy()
    out = oracle.verify_tree_sample(Ls, Ds, toks, pars, u, 2)
    first = out["tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    chi2, pval = stats.chisquare(counts, S * p / p.sum())
    assert pval > 1e-4, (counts, S * p)


# ------------------------------------------------- special cases, hand example


@pytest.mark.parametrize("dtype,seed", [(W.F32, 0), (W.BF16, 1), (W.F32, 2)])
def test_chain_tree_equals_chain_oracle(dtype, seed):
    B, k, V = 6, 4, 300
    case = W.random_sample_case(B, k, V, dtype=dtype, seed=seed, temperature=0.8)
    N = k + 1
    L = case.target
    D = np.concatenate([case.draft, case.draft[:, :1]], axis=1)  # row k unused (leaf)
    toks = np.concatenate([np.zeros((B, 1), np.int32), case.tokens], axis=1)
    par = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    u = np.empty((B, N), np.float32)
    u[:, 1:] = case.uniforms[:, :k]
    u[:, 0] = case.uniforms[:, k]
    cu = case.uniforms.copy()
    cu[:, k + 1] = cu[:, k]  # the tree uses one draw uniform for both ends
    ref = oracle.verify_sample(L, case.draft, case.tokens, cu, temperature=0.8)
    out = oracle.verify_tree_sample(L, D, toks, par, u, k, temperature=0.8)
    np.testing.assert_array_equal(out["n"], ref["n"])
    np.testing.assert_array_equal(out["tokens"], ref["tokens"])
    for b in range(B):
        n = out["n"][b]
        np.testing.assert_array_equal(out["path"][b, :n], np.arange(1, n + 1))


def _hand_tree(child_tokens):
    """p = (0.5, 0.3, 0.2) at the root, q = (0.2, 0.5, 0.3); children are leaves
    whose own rows are uniform."""
    k = len(child_tokens)
    P = np.log(np.array([[0.5, 0.3, 0.2]] + [[1 / 3] * 3] * k)).astype(np.float32)[None]
    Q = np.log(np.array([[0.2, 0.5, 0.3]] + [[1 / 3] * 3] * k)).astype(np.float32)[None]
    toks = np.array([[0] + list(child_tokens)], np.int32)
    par = np.array([[-1] + [0] * k], np.int32)
    return P, Q, toks, par


def test_hand_example_three_tokens():
    # child token 1: accepted iff u < p/q = 0.3/0.5 = 0.6
    P, Q, toks, par = _hand_tree([1, 2])
    out = _run(P, Q, toks, par, [0.1, 0.59, 0.5])
    assert out["n"][0] == 1 and out["path"][0, 0] == 1 and out["tokens"][0, 0] == 1
    # rejected: residual max(0, p - q) = (0.3, 0, 0) -> (1, 0, 0); token 2 has
    # residual mass 0 and is rejected for any u; the next residual
    # max(0, (1, 0, 0) - q) = (0.8, 0, 0) -> (1, 0, 0): the draw gives token 0
    for u0 in (0.0, 0.5, 0.99):
        out = _run(P, Q, toks, par, [u0, 0.61, 0.0])
        assert out["n"][0] == 0 and out["tokens"][0, 0] == 0 and out["tokens"][0, 1] == -1
    # second child token 0 after the rejection: residual (1, 0, 0) over q(0) = 0.2 -> always accepted
    P, Q, toks, par = _hand_tree([1, 0])
    out = _run(P, Q, toks, par, [0.9, 0.7, 0.99])
    assert out["n"][0] == 1 and out["path"][0, 0] == 2 and out["tokens"][0, 0] == 0
    # then the leaf's uniform row is drawn with u_0 = 0.9 -> token 2
    assert out["tokens"][0, 1] == 2
    # no children rejected: without a rejection the draw is from p: u_0 = 0.55 -> token 1
    P, Q, toks, par = _hand_tree([])
    out = _run(P, Q, toks, par, [0.55])
    assert out["n"][0] == 0 and out["tokens"][0, 0] == 1


# ---------------------------------------------------------------- structure


def test_depth_limit_and_flags():
    B, k, V = 4, 4, 50
    case = W.random_sample_case(B, k, V, dtype=W.F32, seed=5, noise=0.0)  # q = p: every test passes
    L = case.target
    D = np.concatenate([case.draft, case.draft[:, :1]], axis=1)
    toks = np.concatenate([np.zeros((B, 1), np.int32), case.tokens], axis=1)
    par = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    u = np.full((B, k + 1), 0.5, np.float32)
    out = oracle.verify_tree_sample(L, D, toks, par, u, 2)
    assert (out["n"] == 2).all()
    assert (out["flags"] & oracle.FLAG_DEPTH).all()
    assert (out["tokens"][:, 2] >= 0).all()
    full = oracle.verify_tree_sample(L, D, toks, par, u, k)
    assert (full["n"] == k).all() and not (full["flags"] & oracle.FLAG_DEPTH).any()


def test_bad_token_is_skipped_and_bad_parent_detached():
    case = W.tree_sample_case(3, 12, 40, 3, seed=8, dtype=W.F32)
    base = oracle.verify_tree_sample(case.logits, case.draft, case.node_tokens, case.parents,
                                     case.uniforms, case.max_depth)
    # an extra last node under the root with an out-of-range token: skipped
    N = case.N
    L = np.concatenate([case.logits, case.logits[:, :1]], axis=1)
    D = np.concatenate([case.draft, case.draft[:, :1]], axis=1)
    toks = np.concatenate([case.node_tokens, np.full((3, 1), case.V + 5, np.int32)], axis=1)
    par = np.concatenate([case.parents, np.zeros((3, 1), np.int32)], axis=1)
    u = np.concatenate([case.uniforms, np.zeros((3, 1), np.float32)], axis=1)
    out = oracle.verify_tree_sample(L, D, toks, par, u, case.max_depth)
    assert (out["flags"] & oracle.FLAG_BAD_TOKEN).all()
    np.testing.assert_array_equal(out["tokens"], base["tokens"])
    np.testing.assert_array_equal(out["path"], base["path"])
    # the same node with a parent pointing forward: detached, flagged
    par[:, N] = N + 3
    toks[:, N] = 1
    out = oracle.verify_tree_sample(L, D, toks, par, u, case.max_depth)
    assert (out["flags"] & oracle.FLAG_BAD_PARENT).all()
    np.testing.assert_array_equal(out["tokens"], base["tokens"])


def test_nonfinite_row_ends_the_walk():
    case = W.tree_sample_case(2, 8, 30, 3, seed=9, dtype=W.F32)
    L = case.logits.copy()
    L[:, 0, 3] = np.nan
    out = oracle.verify_tree_sample(L, case.draft, case.node_tokens, case.parents, case.uniforms,
                                    case.max_depth)
    assert (out["n"] == 0).all() and (out["tokens"][:, 0] == -1).all()
    assert (out["flags"] & oracle.FLAG_BAD_ROW).all()


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_paths_are_root_paths(dtype):
    case = W.tree_sample_case(16, 30, 64, 4, seed=10, dtype=dtype, noise=0.5)
    out = oracle.verify_tree_sample(case.logits, case.draft, case.node_tokens, case.parents,
                                    case.uniforms, case.max_depth)
    for b in range(case.B):
        n = out["n"][b]
        assert 0 <= n <= case.max_depth
        prev = 0
        for d in range(n):
            node = out["path"][b, d]
            assert case.parents[b, node] == prev
            assert out["tokens"][b, d] == case.node_tokens[b, node]
            prev = node
        assert 0 <= out["tokens"][b, n] < case.V
        assert (out["path"][b, n:] == -1).all() and (out["tokens"][b, n + 1:] == -1).all()
    # with a draft close to the target most trees accept at least one node
    assert (out["n"] > 0).mean() > 0.5


def test_masked_tokens_are_never_drawn_or_accepted_from_zero_mass():
    """Tokens with target logit -inf have p = 0: the residual max(0, r - q) is 0
    there too, so no draw lands on them; a child whose token has p = 0 is never
    accepted (u * q(x) < 0 fails for every u >= 0)."""
    rng = np.random.default_rng(41)
    case = W.tree_sample_case(40, 15, 64, 3, seed=41, dtype=W.F32, noise=1.0)
    L = case.logits.copy()
    mask = rng.random(L.shape) < 0.3
    mask[:, :, 0] = False  # every row keeps a finite entry
    L[mask] = -np.inf
    out = oracle.verify_tree_sample(L, case.draft, case.node_tokens, case.parents, case.uniforms, case.max_depth)
    for b in range(case.B):
        n = out["n"][b]
        prev = 0
        for d in range(n):
            node = out["path"][b, d]
            assert not mask[b, prev, case.node_tokens[b, node]]
            prev = node
        assert not mask[b, prev, out["tokens"][b, n]]


# ------------------------------------------------ multi-level trees, exact law


def _table(seed, V, zero=False):
    """A prefix-dependent distribution table with memoised random rational rows."""
    rng = np.random.default_rng(seed)
    cache = {}

    def f(ctx):
        if ctx not in cache:
            w = [Fraction(int(x)) for x in rng.integers(1, 9, size=V)]
            if zero:
                w[int(rng.integers(0, V))] = Fraction(0)
            s = sum(w)
            cache[ctx] = [x / s for x in w]
        return cache[ctx]

    return f


@pytest.mark.parametrize("fanout,V,m,seed", [([1], 3, 3, 0), ([2], 3, 3, 1), ([2, 2], 3, 3, 2),
                                             ([3, 1], 2, 3, 3), ([1, 1, 1], 3, 3, 4), ([2, 1], 3, 2, 5)])
def test_repeated_tree_passes_give_the_target_sequence_law(fanout, V, m, seed):
    """Tree passes repeated from the empty prefix, children drawn from their
    node's draft table: the committed text has exactly the target's law."""
    P = _table(100 + seed, V)
    Q = _table(200 + seed, V, zero=(seed % 2 == 1))
    assert exact.tree_sequence_law(P, Q, fanout, m) == exact.product_law(P, V, m)


def test_c_oracle_tree_pass_follows_the_exact_law():
    """Two-level tree (2 children, 2 grandchildren each), V = 3: the C
    oracle's committed tokens over random child draws and uniforms follow
    exact.tree_pass_law (chi-square over all committed sequences)."""
    from scipy import stats

    V, S = 3, 40000
    P, Q = _table(7, V), _table(8, V)
    ctxs = [()] + [(a,) for a in range(V)] + [(a, c) for a in range(V) for c in range(V)]
    lp = {c: np.log(np.array([float(x) for x in P(c)])).astype(np.float32) for c in ctxs}
    lq = {c: np.log(np.array([float(x) for x in Q(c)])).astype(np.float32) for c in ctxs}
    qf = {c: np.array([float(x) for x in Q(c)]) for c in ctxs}
    rng = np.random.default_rng(9)
    N = 7  # root; 1, 2 under the root; 3, 4 under 1; 5, 6 under 2
    par = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2], np.int32), (S, 1))
    toks = np.zeros((S, N), np.int32)
    toks[:, 1] = rng.choice(V, size=S, p=qf[()])
    toks[:, 2] = rng.choice(V, size=S, p=qf[()])
    L = np.empty((S, N, V), np.float32)
    D = np.empty((S, N, V), np.float32)
    for s in range(S):
        c1, c2 = (int(toks[s, 1]),), (int(toks[s, 2]),)
        toks[s, 3:5] = rng.choice(V, size=2, p=qf[c1])
        toks[s, 5:7] = rng.choice(V, size=2, p=qf[c2])
        ctx = [(), c1, c2, c1 + (int(toks[s, 3]),), c1 + (int(toks[s, 4]),), c2 + (int(toks[s, 5]),),
               c2 + (int(toks[s, 6]),)]
        for j in range(N):
            L[s, j] = lp[ctx[j]] if len(ctx[j]) < 3 else 0.0
            D[s, j] = lq[ctx[j]] if len(ctx[j]) < 3 else 0.0
    u = rng.random((S, N), dtype=np.float32)
    out = oracle.verify_tree_sample(L, D, toks, par, u, 2)
    law = exact.tree_pass_law(P, Q, (), [2, 2])
    keys = sorted(law)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for s in range(S):
        n = int(out["n"][s])
        counts[index[tuple(int(x) for x in out["tokens"][s, :n + 1])]] += 1
    expected = np.array([float(law[k]) for k in keys]) * S
    assert abs(sum(float(law[k]) for k in keys) - 1.0) < 1e-12
    _, pval = stats.chisquare(counts, expected)
    assert pval > 1e-4, list(zip(keys, counts, expected))


def test_per_tree_temperature_equals_separate_runs():
    case = W.tree_sample_case(6, 20, 300, 4, seed=42, dtype=W.F32)
    temps = np.array([0.5, 0.8, 1.0, 1.3, 2.0, 0.7], np.float32)
    out = oracle.verify_tree_sample(case.logits, case.draft, case.node_tokens, case.parents, case.uniforms,
                                    case.max_depth, temperature_per_tree=temps)
    for b in range(case.B):
        sl = slice(b, b + 1)
        one = oracle.verify_tree_sample(case.logits[sl], case.draft[sl], case.node_tokens[sl], case.parents[sl],
                                        case.uniforms[sl], case.max_depth, temperature=float(temps[b]))
        assert out["n"][b] == one["n"][0]
        np.testing.assert_array_equal(out["tokens"][b], one["tokens"][0])
    bad = temps.copy()
    bad[2] = 0.0
    out = oracle.verify_tree_sample(case.logits, case.draft, case.node_tokens, case.parents, case.uniforms,
                                    case.max_depth, temperature_per_tree=bad)
    assert out["n"][2] == 0 and out["tokens"][2, 0] == -1 and out["flags"][2] & oracle.FLAG_BAD_ROW


def test_degenerate_residual_goes_back_to_p():
    """p = q = (1, 0): the first child's token has no mass in either row, so it
    is rejected and the residual max(0, p - q) has mass 0; it goes back to p,
    against which the second child (token 0) is accepted for any u."""
    P = np.array([[[0.0, -np.inf], [0.0, 0.0], [0.0, 0.0]]], np.float32)  # log of (1, 0), (.5, .5), (.5, .5)
    Q = P.copy()
    toks = np.array([[0, 1, 0]], np.int32)
    par = np.array([[-1, 0, 0]], np.int32)
    for u2 in (0.0, 0.5, 0.999):
        out = oracle.verify_tree_sample(P, Q, toks, par, np.array([[0.3, 0.2, u2]], np.float32), 1)
        assert out["n"][0] == 1 and out["path"][0, 0] == 2 and out["tokens"][0, 0] == 0
        assert out["flags"][0] & oracle.FLAG_DEGENERATE
