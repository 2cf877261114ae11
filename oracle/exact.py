"""Exact rational enumeration of the speculative-sampling law (test infrastructure).

An independent statement of the accept-or-correct rule (Edge Inference Notes,
post on speculative decoding and EAGLE-3, "The core idea: draft, then check")
in exact arithmetic with :class:`fractions.Fraction`.  It works with outcome
probabilities, not with uniforms, so it shares nothing with the uniform-driven
C oracle beyond the rule itself:

* the draft proposes x_i ~ q(. | prefix);
* the target accepts x_i with probability min(1, p(x_i) / q(x_i));
* at the first rejection one token is drawn from max(0, p - q) / S;
* if all k drafts are accepted a bonus token is drawn from the last p.

Its law is pinned by the page's claim ("Why it changes nothing about the
output"): the emitted text has exactly the target's distribution, for any q.

Distributions are given as callables ``prefix(tuple) -> list[Fraction]``
(prefix-dependent tables), so that multi-token continuations are exercised.
"""
from __future__ import annotations

from fractions import Fraction
from itertools import combinations, product
from typing import Callable, Dict, List, Sequence, Tuple

Dist = List[Fraction]
Table = Callable[[Tuple[int, ...]], Dist]


def _residual(p: Dist, q: Dist) -> Dist:
    r = [max(Fraction(0), a - b) for a, b in zip(p, q)]
    s = sum(r)
    if s == 0:
        return list(p)
    return [x / s for x in r]


def step_law(P: Table, Q: Table, prefix: Tuple[int, ...], k: int) -> Dict[Tuple[int, ...], Fraction]:
    """Law of the tokens one verification pass commits after ``prefix``."""
    law: Dict[Tuple[int, ...], Fraction] = {}

    def walk(acc: Tuple[int, ...], mass: Fraction, i: int) -> None:
        ctx = prefix + acc
        p = P(ctx)
        if i == k:  # every draft accepted: bonus token from the last row
            for t, pt in enumerate(p):
                if pt:
                    key = acc + (t,)
                    law[key] = law.get(key, Fraction(0)) + mass * pt
            return
        q = Q(ctx)
        res = _residual(p, q)
        for x, qx in enumerate(q):
            if qx == 0:
                continue
            a = min(Fraction(1), p[x] / qx)
            if a:
                walk(acc + (x,), mass * qx * a, i + 1)
            if a != 1:
                rej = mass * qx * (1 - a)
                for t, rt in enumerate(res):
                    if rt:
                        key = acc + (t,)
                        law[key] = law.get(key, Fraction(0)) + rej * rt

    walk((), Fraction(1), 0)
    return law


def sequence_law(P: Table, Q: Table, k: int, m: int) -> Dict[Tuple[int, ...], Fraction]:
    """Law of the first ``m`` tokens when passes are repeated from the empty prefix."""
    out: Dict[Tuple[int, ...], Fraction] = {}

    def run(prefix: Tuple[int, ...], mass: Fraction) -> None:
        if len(prefix) >= m:
            key = prefix[:m]
            out[key] = out.get(key, Fraction(0)) + mass
            return
        for emitted, pr in step_law(P, Q, prefix, k).items():
            run(prefix + emitted, mass * pr)

    run((), Fraction(1))
    return out


def product_law(P: Table, V: int, m: int) -> Dict[Tuple[int, ...], Fraction]:
    """Law of m tokens decoded one by one from the target alone."""
    out: Dict[Tuple[int, ...], Fraction] = {}
    for seq in product(range(V), repeat=m):
        pr = Fraction(1)
        for i in range(m):
            pr *= P(seq[:i])[seq[i]]
            if pr == 0:
                break
        if pr:
            out[seq] = pr
    return out


def expected_committed(P: Table, Q: Table, k: int) -> Fraction:
    """Mean number of tokens one pass commits from the empty prefix."""
    return sum(len(s) * pr for s, pr in step_law(P, Q, (), k).items())


def nucleus_bruteforce(probs: Sequence[float], top_p: float) -> frozenset:
    """Smallest token set whose mass reaches top_p; among sets of that size the
    one with the largest mass (unique when the probabilities are distinct)."""
    V = len(probs)
    for size in range(1, V + 1):
        best = None
        for s in combinations(range(V), size):
            mass = sum(probs[i] for i in s)
            if mass >= top_p and (best is None or mass > best[0]):
                best = (mass, s)
        if best is not None:
            return frozenset(best[1])
    return frozenset(range(V))


def topk_bruteforce(values: Sequence[float], top_k: int) -> frozenset:
    """The top_k-element set with the largest value sum; among equal sums the
    lexicographically smallest index set (lowest indices win ties)."""
    best = None
    for s in combinations(range(len(values)), top_k):
        tot = sum(values[i] for i in s)
        if best is None or tot > best[0]:
            best = (tot, s)
    return frozenset(best[1])


def sibling_law(p: Dist, q: Dist, tokens: Sequence[int]) -> Dict[Tuple[str, int], Fraction]:
    """Law of one tree node's outcome for fixed child tokens, tried in order.

    The rule applied down the branches (Edge Inference Notes, "One decode
    round, end to end"), with the sibling reading: a rejected child removes
    the draft mass from the residual, r <- max(0, r - q) / S, and the next
    child is accepted with probability min(1, r(x) / q(x)) (1 when q(x) = 0
    and r(x) > 0).  A residual of mass 0 is replaced by p.  Keys are
    ("accept", j) for the j-th child and ("draw", t) for a drawn token t once
    every child is rejected.
    """
    law: Dict[Tuple[str, int], Fraction] = {}
    r = list(p)
    reach = Fraction(1)
    for j, x in enumerate(tokens):
        if q[x]:
            a = min(Fraction(1), r[x] / q[x])
        else:
            a = Fraction(1) if r[x] > 0 else Fraction(0)
        if a:
            law[("accept", j)] = reach * a
        reach *= 1 - a
        if reach == 0:
            return law
        w = [max(Fraction(0), a_ - b_) for a_, b_ in zip(r, q)]
        s = sum(w)
        r = [x_ / s for x_ in w] if s else list(p)
    for t, rt in enumerate(r):
        if rt:
            law[("draw", t)] = reach * rt
    return law


def first_token_law(p: Dist, q: Dist, k: int) -> Dict[int, Fraction]:
    """Law of the first committed token when a node has k children drawn
    independently from q and they are checked with :func:`sibling_law`."""
    out: Dict[int, Fraction] = {}
    V = len(p)
    for toks in product(range(V), repeat=k):
        pr = Fraction(1)
        for x in toks:
            pr *= q[x]
        if pr == 0:
            continue
        for (kind, idx), m in sibling_law(p, q, toks).items():
            t = toks[idx] if kind == "accept" else idx
            out[t] = out.get(t, Fraction(0)) + pr * m
    return out


def tree_pass_law(P: Table, Q: Table, prefix: Tuple[int, ...], fanout: Sequence[int]) -> Dict[Tuple[int, ...], Fraction]:
    """Law of the tokens one tree-verification pass commits after ``prefix``.

    The draft tree has ``fanout[d]`` children under every node at depth d
    (leaves at depth len(fanout)); the children of the node reached by path
    ``acc`` are independent draws from Q(prefix + acc).  At each node the
    children are checked with :func:`sibling_law` against P(prefix + acc);
    an accepted child moves the walk into its subtree, a node that accepts
    none commits its draw, and a leaf commits a bonus token from its P.
    """
    law: Dict[Tuple[int, ...], Fraction] = {}

    def node(acc: Tuple[int, ...], mass: Fraction, depth: int) -> None:
        ctx = prefix + acc
        p = P(ctx)
        if depth == len(fanout):
            for t, pt in enumerate(p):
                if pt:
                    key = acc + (t,)
                    law[key] = law.get(key, Fraction(0)) + mass * pt
            return
        q = Q(ctx)
        V = len(p)
        for toks in product(range(V), repeat=fanout[depth]):
            pr = Fraction(1)
            for x in toks:
                pr *= q[x]
            if pr == 0:
                continue
            for (kind, idx), m in sibling_law(p, q, toks).items():
                if kind == "accept":
                    node(acc + (toks[idx],), mass * pr * m, depth + 1)
                else:
                    key = acc + (idx,)
                    law[key] = law.get(key, Fraction(0)) + mass * pr * m

    node((), Fraction(1), 0)
    return law


def tree_sequence_law(P: Table, Q: Table, fanout: Sequence[int], m: int) -> Dict[Tuple[int, ...], Fraction]:
    """Law of the first ``m`` tokens when tree passes are repeated from the empty prefix."""
    out: Dict[Tuple[int, ...], Fraction] = {}

    def run(prefix: Tuple[int, ...], mass: Fraction) -> None:
        if len(prefix) >= m:
            key = prefix[:m]
            out[key] = out.get(key, Fraction(0)) + mass
            return
        for emitted, pr in tree_pass_law(P, Q, prefix, fanout).items():
            run(prefix + emitted, mass * pr)

    run((), Fraction(1))
    return out
