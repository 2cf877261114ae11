"""Pins of the oracle's boundary flags: the 1e-6 width of every flag.

A sequence whose outcome lies within 1e-6 of a decision edge is flagged by
the oracle and left out of the exact GPU comparison, so the width of each
flag decides what parity compares.  Each case below builds rows by hand
(float32 logits of chosen probabilities), computes the decision's distance
to its edge here in float64 from those logits, independently of the oracle,
and places it 5e-7 from the edge (the oracle must flag it) and 2e-6 from the
edge (it must not).  The decisions are those of Edge Inference Notes, "The
core idea: draft, then check", step 3: the accept test u q(x) < p(x), the
inverse-CDF draw from max(0, p - q) or from p, and the top-p cut of "Why it
changes nothing about the output", which matters only when the neighbouring
cut changes the committed tokens.  The same accept and draw cases are pinned
for token-tree sampling ("One decode round, end to end").
"""
import numpy as np
import pytest

import oracle

NEAR, FAR = 5e-7, 2e-6


def _logits(probs):
    return np.log(np.asarray(probs, np.float64)).astype(np.float32)


def _softmax(logits32, T=1.0):
    z = logits32.astype(np.float64) / T
    e = np.exp(z - z.max())
    s = 0.0
    for v in e:  # in index order, as a plain sequential sum
        s += v
    return e / s


def _f32(x):
    return float(np.float32(x))


def _sample(target_rows, draft_rows, x, u, top_p=1.0, top_k=0):
    t = np.asarray(target_rows, np.float32)[None]
    d = np.asarray(draft_rows, np.float32)[None]
    return oracle.verify_sample(t, d, np.asarray([x], np.int32), np.asarray([u], np.float32), 1.0, top_k, top_p)


P0 = [0.1, 0.2, 0.3, 0.4]
Q0 = [0.4, 0.3, 0.2, 0.1]
P1 = [0.25, 0.25, 0.25, 0.25]


def _mid_of(cum, j):
    """A uniform in the middle of interval j of a cumulative array (normalised)."""
    lo = cum[j - 1] if j > 0 else 0.0
    return _f32((lo + cum[j]) / 2 / cum[-1])


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_accept_flag_width(side, dist, flagged):
    t0, d0, t1 = _logits(P0), _logits(Q0), _logits(P1)
    p, q = _softmax(t0), _softmax(d0)
    r = p[0] / q[0]  # x = 0: p < q, accepted with probability p/q
    u0 = _f32(r + side * dist)
    assert abs(abs(u0 - r) - dist) < 0.1 * dist  # the construction sits where intended
    # whichever way the test goes, the draw that follows sits mid-interval
    w = np.maximum(p - q, 0.0)
    u_res = _mid_of(np.cumsum(w), 3)
    u_bonus = _mid_of(np.cumsum(_softmax(t1)), 1)
    o = _sample([t0, t1], [d0], [0], [u0, u_bonus, u_res])
    assert o["n"][0] == (1 if u0 < r else 0)
    assert bool(o["flags"][0] & oracle.FLAG_ACCEPT_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_residual_draw_flag_width(side, dist, flagged):
    t0, d0, t1 = _logits(P0), _logits(Q0), _logits(P1)
    p, q = _softmax(t0), _softmax(d0)
    w = np.maximum(p - q, 0.0)
    S = w.sum()
    c2 = w[:3].sum()  # the edge between tokens 2 and 3 of the residual
    u_res = _f32(c2 / S + side * dist)
    assert abs(abs(u_res * S - c2) / S - dist) < 0.1 * dist
    o = _sample([t0, t1], [d0], [0], [0.9, 0.5, u_res])  # u_0 = 0.9 rejects x = 0 (p/q = 0.25)
    assert o["n"][0] == 0
    assert o["tokens"][0, 0] == (3 if side > 0 else 2)
    assert bool(o["flags"][0] & oracle.FLAG_DRAW_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_bonus_draw_flag_width(side, dist, flagged):
    t0, d0 = _logits(P0), _logits(P0)
    t1 = _logits([0.15, 0.35, 0.3, 0.2])
    p1 = _softmax(t1)
    c = np.cumsum(p1)
    u_bonus = _f32(c[1] / c[-1] + side * dist)
    assert abs(abs(u_bonus * c[-1] - c[1]) / c[-1] - dist) < 0.1 * dist
    o = _sample([t0, t1], [d0], [2], [0.0, u_bonus, 0.5])  # q = p: the draft is accepted
    assert o["n"][0] == 1
    assert o["tokens"][0, 1] == (2 if side > 0 else 1)
    assert bool(o["flags"][0] & oracle.FLAG_DRAW_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


def _cut_row(before):
    """Probabilities of a 3-token row sorted by value whose second token's
    mass-before equals `before`: [before, 0.8 - before, 0.2]."""
    return [before, 0.8 - before, 0.2]


def _before_second(logits32):
    p = _softmax(logits32)
    return p[0]


@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_topp_cut_flag_width_last_kept(dist, flagged):
    """The second token is kept because the mass before it, 0.5 - dist, is
    below top_p = 0.5; the draft token is that token, accepted (u = 0); with
    the neighbouring cut (one token fewer) it would have p = 0 and be
    rejected, so the committed tokens change."""
    t0 = _logits(_cut_row(0.5 - dist))
    assert abs((0.5 - _before_second(t0)) - dist) < 0.1 * dist
    d0 = _logits([0.2, 0.7, 0.1])  # the draft's own cut is far from its edge
    t1 = _logits([0.6, 0.3, 0.1])
    o = _sample([t0, t1], [d0], [1], [0.0, 0.25, 0.5], top_p=0.5)
    assert o["n"][0] == 1 and o["tokens"][0, 0] == 1
    assert bool(o["flags"][0] & oracle.FLAG_CUT_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_topp_cut_flag_width_first_dropped(dist, flagged):
    """The second token is dropped because the mass before it, 0.5 + dist,
    reaches top_p = 0.5; the draft token is that token and is rejected (u =
    0.2 against p = 0); with the neighbouring cut (one token more) it would
    have p = 0.375 against q = 1 and be accepted."""
    t0 = _logits(_cut_row(0.5 + dist))
    assert abs((_before_second(t0) - 0.5) - dist) < 0.1 * dist
    d0 = _logits([0.2, 0.7, 0.1])
    t1 = _logits([0.6, 0.3, 0.1])
    o = _sample([t0, t1], [d0], [1], [0.2, 0.25, 0.5], top_p=0.5)
    assert o["n"][0] == 0
    assert bool(o["flags"][0] & oracle.FLAG_CUT_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


def test_topp_cut_near_edge_but_outcome_unchanged_is_not_flagged():
    """A cut 5e-7 from its edge that no decision depends on: the draft token
    is the top token (kept by either cut) and is accepted either way; the
    bonus row has no cut near its edge and its uniform sits mid-interval."""
    t0 = _logits(_cut_row(0.5 - NEAR))
    d0 = _logits([0.7, 0.2, 0.1])
    t1 = _logits([0.6, 0.3, 0.1])
    o = _sample([t0, t1], [d0], [0], [0.0, 0.3, 0.5], top_p=0.5)
    assert o["n"][0] == 1
    assert o["flags"][0] & oracle.BOUNDARY_FLAGS == 0


# ------------------------------------------------------------- token trees


def _tree(root_p, root_q, leaf_p, tok, u):
    """Root (node 0) with one child (node 1) carrying token tok."""
    logits = np.stack([_logits(root_p), _logits(leaf_p)])[None]
    draft = np.stack([_logits(root_q), _logits(root_q)])[None]
    return oracle.verify_tree_sample(logits, draft, np.asarray([[0, tok]], np.int32),
                                     np.asarray([[-1, 0]], np.int32), np.asarray([u], np.float32), 2)


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_tree_accept_flag_width(side, dist, flagged):
    p, q = _softmax(_logits(P0)), _softmax(_logits(Q0))
    r = p[0] / q[0]
    u1 = _f32(r + side * dist)
    assert abs(abs(u1 - r) - dist) < 0.1 * dist
    # the final draw sits mid-interval either way: from the residual (rejected) or the leaf row (accepted)
    accepted = u1 < r
    cum = np.cumsum(_softmax(_logits(P1))) if accepted else np.cumsum(np.maximum(p - q, 0.0))
    u0 = _mid_of(cum, 1 if accepted else 3)
    o = _tree(P0, Q0, P1, 0, [u0, u1])
    assert o["n"][0] == (1 if accepted else 0)
    assert bool(o["flags"][0] & oracle.FLAG_ACCEPT_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_tree_residual_draw_flag_width(side, dist, flagged):
    p, q = _softmax(_logits(P0)), _softmax(_logits(Q0))
    w = np.maximum(p - q, 0.0)
    S = w.sum()
    c2 = w[:3].sum()
    u0 = _f32(c2 / S + side * dist)
    assert abs(abs(u0 * S - c2) / S - dist) < 0.1 * dist
    o = _tree(P0, Q0, P1, 0, [u0, 0.9])  # u_1 = 0.9 rejects the child (p/q = 0.25)
    assert o["n"][0] == 0
    assert o["tokens"][0, 0] == (3 if side > 0 else 2)
    assert bool(o["flags"][0] & oracle.FLAG_DRAW_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("dist,flagged", [(NEAR, True), (FAR, False)])
def test_tree_leaf_draw_flag_width(side, dist, flagged):
    leaf = [0.15, 0.35, 0.3, 0.2]
    c = np.cumsum(_softmax(_logits(leaf)))
    u0 = _f32(c[1] / c[-1] + side * dist)
    assert abs(abs(u0 * c[-1] - c[1]) / c[-1] - dist) < 0.1 * dist
    o = _tree(P0, P0, leaf, 2, [u0, 0.0])  # q = p: the child is accepted, the leaf row draws
    assert o["n"][0] == 1
    assert o["tokens"][0, 1] == (2 if side > 0 else 1)
    assert bool(o["flags"][0] & oracle.FLAG_DRAW_BOUNDARY) == flagged
    assert bool(o["flags"][0] & oracle.BOUNDARY_FLAGS) == flagged
