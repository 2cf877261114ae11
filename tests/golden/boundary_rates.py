"""Boundary-draw rates of the oracle on the configurations' inputs.

A sequence is a boundary case when one of its decisions (an accept test, the
draw, or a top-p cut that matters) lies within 1e-6 of its edge; the GPU
comparison leaves such sequences out, and their share must stay below 1e-5
of all decisions.  This script counts them over many seeded batches of each
configuration's recipe (C1, C2, C3, and C5 at k = 8 for every sigma), with
the float64 oracle alone, and writes boundary_rates.json beside it.

A sequence's decisions are its draw plus the accept tests the left-to-right
scan consulted (n + 1, or k when every draft is accepted).

    python tests/golden/boundary_rates.py [--min-decisions 100000] [--workers N]
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _case(name: str, seed: int):
    import workloads as W

    if name == "C1":
        return W.config1(seed=1000 + seed, B=8)
    if name == "C2":
        return W.config2(seed=2000 + seed, B=16)
    if name == "C3":
        return W.config3(seed=3000 + seed, B=8)
    if name.startswith("C5"):
        sigma = float(name.split("s")[1])
        return W.config5(8, 8, sigma, seed=5000 + seed)
    raise ValueError(name)


def _one(args):
    name, seed = args
    import oracle

    c = _case(name, seed)
    o = oracle.verify_sample(c.target, c.draft, c.tokens, c.uniforms, c.temperature, c.top_k, c.top_p,
                             c.temperature_per_seq, all_rows=False)
    n = o["n"].astype(np.int64)
    decisions = int(np.sum(1 + np.minimum(n + 1, c.k)))
    flagged = int(np.sum((o["flags"] & oracle.BOUNDARY_FLAGS) != 0))
    kinds = {k: int(np.sum((o["flags"] & v) != 0)) for k, v in (
        ("accept", oracle.FLAG_ACCEPT_BOUNDARY), ("draw", oracle.FLAG_DRAW_BOUNDARY),
        ("degenerate", oracle.FLAG_DEGENERATE), ("cut", oracle.FLAG_CUT_BOUNDARY))}
    return name, c.B, decisions, flagged, kinds


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--min-decisions", type=int, default=100000)
    ap.add_argument("--workers", type=int, default=len(os.sched_getaffinity(0)))
    ap.add_argument("--configs", default="C1,C2,C3,C5s0.5,C5s2,C5s4")
    args = ap.parse_args()
    out = {"what": "sequences within 1e-6 of a decision edge (oracle flags) per decision "
                   "(draw + consulted accept tests), seeded batches of each configuration's recipe",
           "min_decisions": args.min_decisions, "configs": {}}
    ctx = mp.get_context("spawn")
    with ctx.Pool(args.workers) as pool:
        for name in args.configs.split(","):
            t0 = time.time()
            tot = dict(sequences=0, decisions=0, flagged=0, accept=0, draw=0, degenerate=0, cut=0)
            seed = 0
            while tot["decisions"] < args.min_decisions:
                # a round of batches, sized from the decisions per batch seen so far
                per = tot["decisions"] / max(1, seed) if seed else 30.0
                need = max(args.workers, int((args.min_decisions - tot["decisions"]) / per) + 1)
                jobs = [(name, s) for s in range(seed, seed + need)]
                seed += need
                for _, b, d, f, kinds in pool.imap_unordered(_one, jobs):
                    tot["sequences"] += b
                    tot["decisions"] += d
                    tot["flagged"] += f
                    for k, v in kinds.items():
                        tot[k] += v
            tot["rate"] = tot["flagged"] / tot["decisions"]
            tot["seconds"] = round(time.time() - t0, 1)
            out["configs"][name] = tot
            print(name, tot, flush=True)
    with open(os.path.join(HERE, "boundary_rates.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
