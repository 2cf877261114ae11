"""Times the float64 oracle on the host cores, per configuration, for the
CPU-baseline table: single-threaded and with one thread per core over
sequences (trees).  Test infrastructure, like the rest of oracle/.

    python oracle/time_configs.py [--threads N] [--out file.json]

Each configuration runs a bounded sample of its workload (the first few
sequences or trees; the full batch where it is small) and reports the time
per sequence, scaled to the configuration's batch.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def _jobs():
    c1 = W.config1(B=8)
    c2 = W.config2()
    c3 = W.config3()
    c4 = W.config4()
    c5 = W.config5(64, 8, 2.0)
    samp = lambda c, b: oracle.verify_sample(c.target[b:b + 1], c.draft[b:b + 1], c.tokens[b:b + 1],
                                            c.uniforms[b:b + 1], c.temperature, c.top_k, c.top_p,
                                            c.temperature_per_seq[b:b + 1] if c.temperature_per_seq is not None
                                            else None, all_rows=False)
    tree = lambda c, b: oracle.verify_tree_greedy(c.logits[b:b + 1], c.node_tokens[b:b + 1],
                                                  c.parents[b:b + 1], c.max_depth)
    return [
        ("C1 sampling B=1 k=4 V=32000 fp32", c1, 1, 8, samp),
        ("C2 sampling B=16 k=5 V=32000 bf16 top-k 50", c2, 16, 16, samp),
        ("C3 sampling B=64 k=8 V=128256 bf16 top-p 0.9", c3, 64, 16, samp),
        ("C4 greedy tree 8x60 V=128256 bf16", c4, 8, 8, tree),
        ("C5 sampling B=64 k=8 V=152064 bf16 top-p 0.95 sigma 2", c5, 64, 16, samp),
    ]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--threads", type=int, default=len(os.sched_getaffinity(0)))
    ap.add_argument("--out", default="")
    args = ap.parse_args()
    oracle.build()
    res = []
    for name, case, batch, sample, fn in _jobs():
        idx = list(range(min(sample, case.B)))
        t0 = time.perf_counter()
        for b in idx:
            fn(case, b)
        one = (time.perf_counter() - t0) / len(idx)
        t0 = time.perf_counter()
        with ThreadPoolExecutor(args.threads) as pool:
            list(pool.map(lambda b: fn(case, b), idx * max(1, args.threads // len(idx) + 1)))
        nrun = len(idx) * max(1, args.threads // len(idx) + 1)
        many = (time.perf_counter() - t0) / nrun
        r = {"config": name, "batch": batch, "sample": len(idx), "threads": args.threads,
             "one_core_s_per_batch": one * batch, "n_core_s_per_batch": many * batch}
        res.append(r)
        print(json.dumps(r), flush=True)
    if args.out:
        with open(args.out, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()
