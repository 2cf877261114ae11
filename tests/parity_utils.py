"""Shared helpers for the GPU parity tests: move seeded numpy inputs to the
device, run the library through its C ABI binding, run the oracle on the same
arrays and compare."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import workloads as W

ABS_TOL_PROB = 1e-5          # normalised probabilities (spec tolerance)


def to_dev(arr: np.ndarray) -> torch.Tensor:
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(arr).cuda()


def lib():
    import draft_token_verification_gb300 as sv

    sv.build()
    return sv


def run_sample_gpu(case: W.SampleCase, **kw):
    sv = lib()
    tps = to_dev(case.temperature_per_seq) if case.temperature_per_seq is not None else None
    out = sv.spec_verify_sample(to_dev(case.target), to_dev(case.draft), to_dev(case.tokens),
                                to_dev(case.uniforms), case.temperature, case.top_k, case.top_p, tps, **kw)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def run_sample_oracle(case: W.SampleCase, seqs=None):
    """The oracle on the chosen sequences (all by default), split over the
    host's cores a few sequences per call (the C oracle runs outside the GIL)."""
    idx = np.arange(case.B) if seqs is None else np.asarray(seqs)
    tps_all = case.temperature_per_seq
    chunks = [idx[i:i + 4] for i in range(0, len(idx), 4)]

    def one(ix):
        tps = tps_all[ix] if tps_all is not None else None
        return oracle.verify_sample(case.target[ix], case.draft[ix], case.tokens[ix], case.uniforms[ix],
                                    case.temperature, case.top_k, case.top_p, tps, all_rows=True)

    workers = max(1, min(len(chunks), len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(workers) as pool:
        parts = list(pool.map(one, chunks))
    return {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}


def _cut_boundary_row(row, T, top_k, top_p) -> bool:
    """The row's top-p cut is within 1e-6 of top_p: a neighbouring cut changes
    the normalisation of every kept token."""
    _, margin, _, _, _ = oracle.row_probs(row, T, top_k, top_p)
    return margin < 1e-6


def compare_sample(case: W.SampleCase, gpu, orc, seqs=None):
    """Exact tokens / accept counts outside boundary draws; p(x), q(x) within
    1e-5.  Returns (boundary sequences, decisions: draws + consulted tests)."""
    g_tok, g_n, g_p, g_q = gpu
    idx = np.arange(case.B) if seqs is None else np.asarray(seqs)
    g_tok, g_n, g_p, g_q = g_tok[idx], g_n[idx], g_p[idx], g_q[idx]
    flags = orc["flags"]
    boundary = (flags & oracle.BOUNDARY_FLAGS) != 0
    bad = []
    for j, b in enumerate(idx):
        n = int(g_n[j])
        assert 0 <= n <= case.k, (b, n)
        assert np.all(g_tok[j, n + 1:] == -1)
        if boundary[j]:
            continue
        if n != orc["n"][j] or not np.array_equal(g_tok[j], orc["tokens"][j]):
            bad.append((int(b), n, int(orc["n"][j]), g_tok[j].tolist(), orc["tokens"][j].tolist(),
                        int(flags[j]), float(orc["margin"][j])))
    assert not bad, f"{len(bad)} sequences differ outside boundary draws: {bad[:4]}"
    temps = case.temps()
    for name, g, o in (("p", g_p, orc["p_draft"]), ("q", g_q, orc["q_draft"])):
        diff = np.abs(g.astype(np.float64) - o)
        for j, i in zip(*np.nonzero(~(diff <= ABS_TOL_PROB))):
            b = idx[j]
            row = case.target[b, i] if name == "p" else case.draft[b, i]
            assert _cut_boundary_row(row, float(temps[b]), case.top_k, case.top_p), (
                f"{name}(x) differs at seq {b} pos {i}: gpu {g[j, i]} oracle {o[j, i]}")
    # decisions: each sequence's draw plus the accept tests its scan consulted
    n_o = orc["n"].astype(np.int64)
    draws = int(np.sum(1 + np.minimum(n_o + 1, case.k)))
    return int(boundary.sum()), draws


def run_greedy_gpu(target: np.ndarray, tokens: np.ndarray):
    sv = lib()
    out = sv.spec_verify_greedy(to_dev(target), to_dev(tokens))
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def run_tree_gpu(case: W.TreeCase):
    sv = lib()
    out = sv.spec_verify_tree_greedy(to_dev(case.logits), to_dev(case.node_tokens), to_dev(case.parents),
                                     case.max_depth)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def q_support_mask(top_k, top_p):
    """Candidate mask for draft tokens: the draft's own filtered support."""
    def fn(row, T):
        probs, *_ = oracle.row_probs(row, T, top_k, top_p)
        return probs > 0
    return fn
