"""Pins for the float64 oracle: checks against what the pages and the
mathematics fix, never against the oracle itself.

* exact rational law (oracle/exact.py) == target law, for any draft
  (Edge Inference Notes, "Why it changes nothing about the output");
* the C oracle's uniform-driven draws follow that law (chi-square, fixed seed);
* mean committed tokens == (1 - a^(g+1)) / (1 - a) for i.i.d. acceptance a
  (Speculative Decoding Speedup Calculator, step 1);
* 1 <= committed <= k+1 (Edge Inference Notes, "The core idea");
* hand-worked accept / residual / bonus examples (tests/golden);
* filters: brute-force kept sets, softmax special case, closed forms;
* greedy chain and tree against brute force;
* special cases: top-k = 1 reduces sampling to greedy; q = p accepts all.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy import special, stats

import oracle
from oracle import exact
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _logits_from_probs(rows):
    a = np.asarray(rows, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(a).astype(np.float32)


# ---------------------------------------------------------------- exact law


def _rand_table(rng, V, zero_frac=0.0):
    cache = {}

    def table(prefix):
        if prefix not in cache:
            w = [int(x) for x in rng.integers(1, 9, size=V)]
            for i in range(V):
                if rng.random() < zero_frac:
                    w[i] = 0
            if sum(w) == 0:
                w[int(rng.integers(0, V))] = 1
            s = sum(w)
            cache[prefix] = [Fraction(x, s) for x in w]
        return cache[prefix]

    return table


@pytest.mark.parametrize("V,k,m,zq", [(2, 1, 3, 0.0), (3, 2, 3, 0.0), (3, 2, 3, 0.4), (4, 3, 2, 0.3), (3, 3, 4, 0.2)])
def test_exact_law_equals_target(V, k, m, zq):
    rng = np.random.default_rng(V * 100 + k * 10 + m)
    P = _rand_table(rng, V, zero_frac=0.2)
    Q = _rand_table(rng, V, zero_frac=zq)
    assert exact.sequence_law(P, Q, k, m) == exact.product_law(P, V, m)


def test_exact_law_degenerate_drafts():
    V, k, m = 3, 2, 3
    rng = np.random.default_rng(7)
    P = _rand_table(rng, V, zero_frac=0.2)
    same = exact.sequence_law(P, P, k, m)  # q = p: every draft accepted
    assert same == exact.product_law(P, V, m)
    onehot = lambda prefix: [Fraction(1), Fraction(0), Fraction(0)]
    assert exact.sequence_law(P, onehot, k, m) == exact.product_law(P, V, m)
    # q = p gives k+1 tokens every pass
    assert exact.expected_committed(P, P, k) == k + 1


def _iid_rows(alpha: Fraction, V=3):
    """Fixed rows with sum_x min(p, q) = alpha (acceptance alpha at every position)."""
    p = [Fraction(1) - alpha, alpha, Fraction(0)] if V == 3 else None
    q = [Fraction(0), alpha, Fraction(1) - alpha]
    return p, q


@pytest.mark.parametrize("alpha,k", [(Fraction(1, 3), 3), (Fraction(3, 4), 4), (Fraction(1, 2), 1), (Fraction(9, 10), 5)])
def test_exact_expected_tokens_closed_form(alpha, k):
    p, q = _iid_rows(alpha)
    e = exact.expected_committed(lambda _: p, lambda _: q, k)
    assert e == (1 - alpha ** (k + 1)) / (1 - alpha)
    assert sum(alpha ** i for i in range(k + 1)) == e


# ------------------------------------------------- C oracle vs. the exact law


def _run_oracle_batch(p_rows, q_rows, rng, n_seq, k):
    """One verification pass over n_seq independent sequences with fixed rows."""
    V = p_rows.shape[-1]
    target = np.broadcast_to(_logits_from_probs(p_rows), (n_seq, k + 1, V)).copy()
    draft = np.broadcast_to(_logits_from_probs(q_rows), (n_seq, k, V)).copy()
    tokens = np.stack([rng.choice(V, size=n_seq, p=q_rows[i]) for i in range(k)], axis=1).astype(np.int32)
    u = rng.random((n_seq, k + 2), dtype=np.float32)
    return oracle.verify_sample(target, draft, tokens, u, all_rows=False)


def test_oracle_first_token_follows_target_chi2():
    rng = np.random.default_rng(11)
    V, k, n = 5, 3, 60000
    p = rng.dirichlet(np.ones(V), size=k + 1)
    q = rng.dirichlet(np.ones(V) * 0.5, size=k)
    out = _run_oracle_batch(p, q, rng, n, k)
    first = out["tokens"][:, 0]
    obs = np.bincount(first, minlength=V)
    # the first committed token is distributed as p_0 whatever q is
    chi2 = stats.chisquare(obs, n * p[0])
    assert chi2.pvalue > 1e-4, chi2


def test_oracle_multi_pass_sequence_law_chi2():
    """Repeated passes from the committed prefix: first m tokens ~ product of p."""
    V, k, m = 3, 2, 3
    rng_t = np.random.default_rng(5)
    P = _rand_table(rng_t, V)
    Q = _rand_table(rng_t, V, zero_frac=0.3)
    law = exact.product_law(P, V, m)
    rng = np.random.default_rng(6)
    n_chains = 40000
    seqs = [() for _ in range(n_chains)]
    while True:
        active = [c for c in range(n_chains) if len(seqs[c]) < m]
        if not active:
            break
        A = len(active)
        target = np.empty((A, k + 1, V), np.float32)
        draft = np.empty((A, k, V), np.float32)
        tokens = np.empty((A, k), np.int32)
        for a, c in enumerate(active):
            pre = seqs[c]
            drafted = ()
            for i in range(k + 1):
                ctx = pre + drafted
                target[a, i] = _logits_from_probs([float(x) for x in P(ctx)])
                if i < k:
                    qv = np.array([float(x) for x in Q(ctx)])
                    draft[a, i] = _logits_from_probs(qv)
                    x = int(rng.choice(V, p=qv / qv.sum()))
                    tokens[a, i] = x
                    drafted = drafted + (x,)
        u = rng.random((A, k + 2), dtype=np.float32)
        out = oracle.verify_sample(target, draft, tokens, u, all_rows=False)
        for a, c in enumerate(active):
            n = int(out["n"][a])
            seqs[c] = seqs[c] + tuple(int(t) for t in out["tokens"][a, : n + 1])
    keys = sorted(law)
    counts = {key: 0 for key in keys}
    for s in seqs:
        counts[s[:m]] = counts.get(s[:m], 0) + 1
    assert set(counts) == set(keys), "emitted a sequence the target gives probability 0"
    obs = np.array([counts[key] for key in keys], float)
    exp_ = np.array([float(law[key]) for key in keys]) * n_chains
    chi2 = stats.chisquare(obs, exp_)
    assert chi2.pvalue > 1e-4, chi2


@pytest.mark.parametrize("alpha,k", [(0.3, 3), (0.75, 5), (0.9, 8)])
def test_oracle_mean_committed_matches_closed_form(alpha, k):
    rng = np.random.default_rng(int(alpha * 100) + k)
    p = np.array([1 - alpha, alpha, 0.0])
    q = np.array([0.0, alpha, 1 - alpha])
    n_seq = 40000
    out = _run_oracle_batch(np.tile(p, (k + 1, 1)), np.tile(q, (k, 1)), rng, n_seq, k)
    committed = out["n"] + 1
    e = (1 - alpha ** (k + 1)) / (1 - alpha)
    sd = committed.std() / math.sqrt(n_seq)
    assert abs(committed.mean() - e) < 4 * sd + 1e-9
    assert committed.min() >= 1 and committed.max() <= k + 1


# ------------------------------------------------------- worked examples


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("accept_examples.json")["cases"], ids=lambda c: c["name"])
def test_oracle_hand_worked_examples(case):
    target = _logits_from_probs(case["target"])[None]
    draft = _logits_from_probs(case["draft"])[None]
    tokens = np.array([case["tokens"]], np.int32)
    u = np.array([case["uniforms"]], np.float32)
    out = oracle.verify_sample(target, draft, tokens, u)
    assert out["tokens"][0].tolist() == case["expect_tokens"]
    assert int(out["n"][0]) == case["expect_n"]
    assert out["flags"][0] & oracle.BOUNDARY_FLAGS == 0


def test_closed_forms_golden():
    g = _golden("closed_forms.json")
    for c in g["break_even"]["cases"]:
        assert oracle.break_even(c["k"]) == pytest.approx(c["value"], rel=1e-15)
        assert f"{round(100 * oracle.break_even(c['k']))}%" == c["printed"]
    for c in g["expected_tokens"]["cases"]:
        assert oracle.expected_tokens_series(c["alpha"], c["gamma"]) == pytest.approx(c["value"], rel=1e-12)
        if c["alpha"] != 1.0:
            assert oracle.expected_tokens_closed(c["alpha"], c["gamma"]) == pytest.approx(c["value"], rel=1e-12)
    for c in g["improvement_factor"]["cases"]:
        assert oracle.improvement_factor(c["alpha"], c["gamma"], c["c"]) == pytest.approx(c["value"], rel=1e-12)


@pytest.mark.parametrize("case", _golden("closed_forms.json")["filters"]["cases"], ids=lambda c: str(c["logits"]) + str(c["top_k"]))
def test_filter_closed_forms(case):
    probs, _, _, _, ok = oracle.row_probs(np.array(case["logits"], np.float32), case["temperature"],
                                          case["top_k"], case["top_p"])
    assert ok
    np.testing.assert_allclose(probs, case["probs"], rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------ filters


@pytest.mark.parametrize("seed", range(12))
def test_nucleus_and_topk_kept_sets_bruteforce(seed):
    rng = np.random.default_rng(seed)
    V = 8
    logits = rng.normal(0, 2, V).astype(np.float32)
    T = float(rng.uniform(0.5, 1.5))
    z = logits.astype(np.float64) / T
    soft = special.softmax(z)
    for top_p in (0.3, 0.5, 0.8, 0.95):
        probs, margin, *_ = oracle.row_probs(logits, T, 0, top_p)
        want = exact.nucleus_bruteforce(list(soft), top_p)
        assert frozenset(np.nonzero(probs)[0].tolist()) == want
        kept = np.array(sorted(want))
        np.testing.assert_allclose(probs[kept], soft[kept] / soft[kept].sum(), rtol=1e-12)
    for top_k in (1, 3, 5):
        probs, *_ = oracle.row_probs(logits, T, top_k, 1.0)
        want = exact.topk_bruteforce(list(z), top_k)
        assert frozenset(np.nonzero(probs)[0].tolist()) == want
        # top-k then top-p on the renormalised top-k distribution
        sub = np.array(sorted(want))
        sub_soft = soft[sub] / soft[sub].sum()
        probs2, *_ = oracle.row_probs(logits, T, top_k, 0.6)
        nuc = exact.nucleus_bruteforce(list(sub_soft), 0.6)
        assert frozenset(np.nonzero(probs2)[0].tolist()) == frozenset(int(sub[i]) for i in nuc)


@pytest.mark.parametrize("seed", range(6))
def test_topk_ties_keep_lowest_indices(seed):
    rng = np.random.default_rng(100 + seed)
    V = 9
    logits = rng.integers(-2, 3, V).astype(np.float32)  # many exact ties
    for top_k in range(1, V):
        probs, *_ = oracle.row_probs(logits, 1.0, top_k, 1.0)
        want = exact.topk_bruteforce(list(logits.astype(float)), top_k)
        assert frozenset(np.nonzero(probs)[0].tolist()) == want


def test_no_filter_is_softmax_at_temperature():
    rng = np.random.default_rng(3)
    for T in (0.3, 1.0, 2.5):
        logits = rng.normal(0, 3, 1000).astype(np.float32)
        probs, *_ = oracle.row_probs(logits, T, 0, 1.0)
        np.testing.assert_allclose(probs, special.softmax(logits.astype(np.float64) / T), rtol=1e-12, atol=1e-300)
        probs_k, *_ = oracle.row_probs(logits, T, 1000, 1.0)
        np.testing.assert_array_equal(probs, probs_k)


def test_bf16_rows_widen_exactly():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 3, 777).astype(np.float32)
    bits = W.bf16_bits(x)
    probs_b, *_ = oracle.row_probs(bits, 0.7, 0, 1.0)
    probs_f, *_ = oracle.row_probs(W.bits_to_f32(bits), 0.7, 0, 1.0)
    np.testing.assert_array_equal(probs_b, probs_f)
    # widening: bf16 bits are the upper half of the float32 pattern (torch agrees)
    import torch

    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), bits)


def test_masked_logits_get_zero_probability():
    logits = np.array([1.0, -np.inf, 0.5, -np.inf], np.float32)
    probs, *_ = oracle.row_probs(logits, 1.0, 0, 1.0)
    assert probs[1] == 0 and probs[3] == 0
    np.testing.assert_allclose(probs[[0, 2]], special.softmax([1.0, 0.5]), rtol=1e-12)
    _, _, _, _, ok = oracle.row_probs(np.array([1.0, np.nan], np.float32))
    assert not ok
    _, _, _, _, ok = oracle.row_probs(np.array([-np.inf, -np.inf], np.float32))
    assert not ok


# --------------------------------------------------- sampling special cases


def test_inverse_cdf_matches_searchsorted():
    """Residual and bonus draws equal numpy's searchsorted on the running sums."""
    rng = np.random.default_rng(9)
    V, k, B = 50, 2, 200
    target = rng.normal(0, 2, (B, k + 1, V)).astype(np.float32)
    draft = rng.normal(0, 2, (B, k, V)).astype(np.float32)
    tokens = rng.integers(0, V, (B, k)).astype(np.int32)
    # force a rejection at position 0 for even b: the draft token is masked in the target
    for b in range(0, B, 2):
        target[b, 0, tokens[b, 0]] = -np.inf
    u = rng.random((B, k + 2), dtype=np.float32)
    out = oracle.verify_sample(target, draft, tokens, u)
    checked = 0
    for b in range(B):
        n = int(out["n"][b])
        if n < k:
            p, *_ = oracle.row_probs(target[b, n])
            q, *_ = oracle.row_probs(draft[b, n])
            r = np.maximum(p - q, 0.0)
            c = np.cumsum(r)
            j = int(np.searchsorted(c, float(u[b, k + 1]) * c[-1], side="right"))
        else:
            p, *_ = oracle.row_probs(target[b, k])
            c = np.cumsum(p)
            j = int(np.searchsorted(c, float(u[b, k]) * c[-1], side="right"))
        if out["flags"][b] & oracle.BOUNDARY_FLAGS:
            continue
        assert out["tokens"][b, n] == j
        checked += 1
    assert checked > B * 0.9
    assert np.all(out["n"][0::2] == 0)


@pytest.mark.parametrize("seed", range(4))
def test_topk1_sampling_equals_greedy(seed):
    case = W.random_sample_case(B=40, k=4, V=300, dtype=W.BF16, seed=seed, quantize=0.5 if seed % 2 else None)
    for T in (0.6, 1.3):
        s = oracle.verify_sample(case.target, case.draft, case.tokens, case.uniforms, T, top_k=1)
        g = oracle.verify_greedy(case.target, case.tokens)
        np.testing.assert_array_equal(s["n"], g["n"])
        np.testing.assert_array_equal(s["tokens"], g["tokens"])


def test_identical_draft_accepts_everything():
    case = W.random_sample_case(B=50, k=6, V=400, dtype=W.BF16, seed=1)
    draft = case.target[:, :-1].copy()
    out = oracle.verify_sample(case.target, draft, case.tokens, case.uniforms, 0.8, top_p=0.9)
    # a draft token outside the (shared) kept set has p = q = 0 and is rejected
    for b in range(case.B):
        n = int(out["n"][b])
        if n < case.k:
            assert out["p_draft"][b, n] == 0 and out["q_draft"][b, n] == 0
        for i in range(n):
            assert out["p_draft"][b, i] == out["q_draft"][b, i] > 0


@pytest.mark.parametrize("cfg", ["C1", "C2", "rand"])
def test_commit_bounds_and_padding(cfg):
    if cfg == "C1":
        case = W.config1()
    elif cfg == "C2":
        case = W.config2(B=4)
    else:
        case = W.random_sample_case(B=64, k=7, V=97, seed=3, top_k=5, top_p=0.7, per_seq_temperature=True)
    out = oracle.verify_sample(case.target, case.draft, case.tokens, case.uniforms, case.temperature,
                               case.top_k, case.top_p, case.temperature_per_seq)
    for b in range(case.B):
        n = int(out["n"][b])
        assert 0 <= n <= case.k
        row = out["tokens"][b]
        assert np.all(row[: n + 1] >= 0) and np.all(row[: n + 1] < case.V)
        assert np.all(row[n + 1:] == -1)
        assert np.array_equal(row[:n], case.tokens[b, :n])


# ------------------------------------------------------- greedy and tree


@pytest.mark.parametrize("seed", range(4))
def test_greedy_against_argmax_chain(seed):
    case = W.random_sample_case(B=30, k=5, V=64, seed=seed, quantize=1.0)
    target_f = W.as_f32(case.target)
    am = np.argmax(target_f, axis=-1)  # numpy: first occurrence = lowest index
    tokens = case.tokens.copy()
    rng = np.random.default_rng(seed)
    for b in range(case.B):  # make some long agreeing prefixes
        cut = int(rng.integers(0, case.k + 1))
        tokens[b, :cut] = am[b, :cut]
    out = oracle.verify_greedy(case.target, tokens)
    for b in range(case.B):
        n = 0
        while n < case.k and tokens[b, n] == am[b, n]:
            n += 1
        assert out["n"][b] == n
        assert out["tokens"][b, :n].tolist() == tokens[b, :n].tolist()
        assert out["tokens"][b, n] == am[b, n]
        assert np.all(out["tokens"][b, n + 1:] == -1)


def _tree_bruteforce(am, tokens, parents, max_depth):
    N = len(parents)
    best, best_path = 0, []
    for j in range(1, N):
        path = []
        c = j
        ok = True
        while c != 0:
            p = parents[c]
            if not (0 <= p < c):
                ok = False
                break
            if tokens[c] != am[p]:
                ok = False
            path.append(c)
            c = p
        if not ok or len(path) > max_depth:
            continue
        if len(path) > len(best_path):
            best, best_path = j, path[::-1]
    return best, best_path


@pytest.mark.parametrize("seed", range(5))
def test_tree_against_path_enumeration(seed):
    case = W.random_tree_case(B=12, N=40, V=50, max_depth=6, seed=seed, quantize=1.0 if seed % 2 else None)
    out = oracle.verify_tree_greedy(case.logits, case.node_tokens, case.parents, case.max_depth)
    am = np.argmax(W.as_f32(case.logits), axis=-1)
    for b in range(case.B):
        best, path = _tree_bruteforce(am[b], case.node_tokens[b], case.parents[b], case.max_depth)
        L = len(path)
        assert out["n"][b] == L
        assert out["path"][b, :L].tolist() == path
        assert out["tokens"][b, :L].tolist() == [int(case.node_tokens[b, j]) for j in path]
        assert out["tokens"][b, L] == am[b, best]
        assert np.all(out["tokens"][b, L + 1:] == -1)


def test_tree_chain_equals_greedy_chain():
    """A tree that is a single chain is the greedy chain verification."""
    case = W.random_sample_case(B=20, k=6, V=80, seed=2, quantize=1.0)
    am = np.argmax(W.as_f32(case.target), axis=-1)
    tokens = case.tokens.copy()
    tokens[::2, :3] = am[::2, :3]
    g = oracle.verify_greedy(case.target, tokens)
    N = case.k + 1
    parents = np.tile(np.arange(-1, N - 1, dtype=np.int32), (case.B, 1))
    node_tokens = np.concatenate([np.full((case.B, 1), -1, np.int32), tokens], axis=1)
    t = oracle.verify_tree_greedy(case.target, node_tokens, parents, case.k)
    np.testing.assert_array_equal(t["n"], g["n"])
    np.testing.assert_array_equal(t["tokens"], g["tokens"])


def test_tree_malformed_parents_flagged():
    logits = np.zeros((1, 4, 5), np.float32)
    tokens = np.array([[-1, 0, 0, 0]], np.int32)
    parents = np.array([[-1, 0, 3, 1]], np.int32)  # node 2 points forward
    out = oracle.verify_tree_greedy(logits, tokens, parents, 3)
    assert out["flags"][0] & 1
    assert out["n"][0] == 2 and out["path"][0, :2].tolist() == [1, 3]


# The calculator's draft-length scan (gamma = 1..12, the peak speedup), pinned
# by the cases the mathematics decides without the scan:
#  - c = 0: the speedup is E itself, which grows with gamma when alpha > 0, so
#    the scan ends at gamma_max (alpha = 0: E = 1 for every gamma, so 1);
#  - alpha = 0: the speedup is 1 / (gamma c + 1), falling with gamma when c > 0;
#  - alpha = 1: E = gamma + 1 and the speedup (gamma + 1) / (gamma c + 1) rises
#    for c < 1, falls for c > 1 and is 1 for c = 1 (ties: the smallest gamma);
#  - the speedup at the chosen gamma is no lower than at every gamma scanned,
#    and equals improvement_factor there.
def test_best_gamma_special_cases():
    assert oracle.best_gamma(0.7, 0.0, 12) == (12, pytest.approx(oracle.expected_tokens_series(0.7, 12)))
    assert oracle.best_gamma(0.0, 0.0, 12)[0] == 1
    for c in (0.05, 0.5, 2.0):
        g, f = oracle.best_gamma(0.0, c, 12)
        assert g == 1 and f == pytest.approx(1.0 / (c + 1.0), rel=1e-15)
    assert oracle.best_gamma(1.0, 0.3, 12) == (12, pytest.approx(13.0 / (12 * 0.3 + 1.0), rel=1e-15))
    assert oracle.best_gamma(1.0, 1.5, 12) == (1, pytest.approx(2.0 / 2.5, rel=1e-15))
    assert oracle.best_gamma(1.0, 1.0, 12) == (1, pytest.approx(1.0, rel=1e-15))


@pytest.mark.parametrize("alpha,c", [(0.8, 0.05), (0.6, 0.1), (0.9, 0.02), (0.5, 0.3), (0.95, 0.2)])
def test_best_gamma_is_the_scan_peak(alpha, c):
    g, f = oracle.best_gamma(alpha, c, 12)
    assert 1 <= g <= 12 and f == oracle.improvement_factor(alpha, g, c)
    for gg in range(1, 13):
        assert oracle.improvement_factor(alpha, gg, c) <= f
        if gg < g:
            assert oracle.improvement_factor(alpha, gg, c) < f
    # the speedup rises to the peak and falls after it (the page: concave in gamma)
    vals = [oracle.improvement_factor(alpha, gg, c) for gg in range(1, 13)]
    assert all(vals[i] < vals[i + 1] for i in range(g - 1))
    assert all(vals[i] >= vals[i + 1] for i in range(g - 1, 11))


# The rejection fast path, pinned by hand-made rows: the lowest index wins a
# tie, -0 equals +0, and a mismatching draft yields the argmax to commit.
def test_first_draft_check_hand_rows():
    rows = np.array([[0.0, 3.0, 1.0, 3.0],       # tie at 1 and 3: lowest index, 1
                     [-0.0, -1.0, 0.0, -2.0],    # -0 == +0: index 0
                     [-np.inf, -5.0, -np.inf, -7.0],
                     [2.0, 1.0, 0.5, 9.5]], np.float32)
    draft0 = np.array([1, 2, 1, 0], np.int32)
    for arr in (rows, W.bf16_bits(rows)):
        o = oracle.first_draft_check(arr, draft0)
        assert o["argmax"].tolist() == [1, 0, 1, 3]
        assert o["accept"].tolist() == [1, 0, 1, 0]
