"""Throughput benchmark of draft-token verification on GB300.

One step = one pass of the whole verification hot path over one batch:
  * speculative-sampling verification of 64 sequences, k = 8 drafts,
    V = 128256, bf16, T = 0.9, top-p 0.9 on target and draft rows;
  * greedy chain verification of the same target rows (a separate copy, so
    no kernel reads another's inputs out of L2);
  * greedy token-tree verification of 8 trees of 60 nodes, depth <= 6,
    V = 128256, bf16.
Metric: verified draft positions per second (64*8 + 64*8 + 8*59 per step).

Each step also lists the KV-cache keep entries of the sampled chains and of
the trees (spec_kv_compact), the bookkeeping a decode loop needs next.

Default: python bench.py [--gpus N --steps K --warmup W]; prints one JSON line.
--impl reference times the float64 CPU oracle on a bounded sample instead.
--sweep times sampling and greedy verification over the V = 152064 sweep
(B in 1..256, k in 1..12, three draft noise levels) and the draft-length scan
fed with the measured verification cost; it prints one JSON line.
Under torchrun every rank runs its own batch on its own GPU (weak scaling,
no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verified draft positions/sec on 1 GB300 and achieved HBM GB/s vs roofline"
UNIT = "positions/s"
SAMPLE = dict(B=64, k=8, V=128256, T=0.9, top_k=0, top_p=0.9)
TREE = dict(B=8, N=60, V=128256, depth=6)


def positions_per_step():
    return SAMPLE["B"] * SAMPLE["k"] * 2 + TREE["B"] * (TREE["N"] - 1)


def sample_bytes():
    return SAMPLE["B"] * (2 * SAMPLE["k"] + 1) * SAMPLE["V"] * 2


def greedy_bytes():
    return SAMPLE["B"] * (SAMPLE["k"] + 1) * SAMPLE["V"] * 2


def tree_bytes():
    return TREE["B"] * TREE["N"] * TREE["V"] * 2


def tree_sample_bytes(case, n, path):
    """Bytes the tree-sampling kernels must read: both rows of every node with a
    child to test, plus the target row of a stop node without one."""
    total = 0
    for b in range(case.B):
        par = case.parents[b]
        dep = np.zeros(case.N, int)
        for j in range(1, case.N):
            dep[j] = dep[par[j]] + 1
        internal = {int(par[j]) for j in range(1, case.N)
                    if dep[par[j]] < case.max_depth and 0 <= case.node_tokens[b, j] < case.V}
        stop = 0 if n[b] == 0 else int(path[b, n[b] - 1])
        total += (2 * len(internal) + (stop not in internal)) * case.V * 2
    return total


def time_tree_sample(sv, dev, ws, stream, seed, iters=20):
    """Token-tree sampling verification, timed alone outside the step: 8 trees
    of 60 nodes, depth <= 6, V = 128256, bf16, children drawn from their
    parents' draft rows.  A 512 MB buffer (4x L2) is written before every timed call
    (the rows it reads fit in L2)."""
    import torch

    c = W.tree_sample_case(TREE["B"], TREE["N"], TREE["V"], TREE["depth"], seed=seed)
    args = [to_torch(x, dev) for x in (c.logits, c.draft, c.node_tokens, c.parents, c.uniforms)]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        out = sv.spec_verify_tree_sample(*args, TREE["depth"], workspace=ws, stream=stream)
    ts = []
    for _ in range(iters):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        out = sv.spec_verify_tree_sample(*args, TREE["depth"], workspace=ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    n, path = out[2].cpu().numpy(), out[1].cpu().numpy()
    return float(np.median(ts)), tree_sample_bytes(c, n, path), float(n.mean())


def time_per_seq_temperature(sv, dev, ws, stream, seed, iters=20):
    """Sampling verification of the main workload with a temperature per
    sequence (T_b ~ U(0.5, 1.2)), timed alone: the same 64 x 8 x 128256 bf16
    rows as the step with a per-sequence temperature array.  The rows (279 MB)
    exceed L2, so every call reads them from HBM."""
    import torch

    c = W.config3(seed=seed, per_seq_temperature=True, B=SAMPLE["B"], k=SAMPLE["k"], V=SAMPLE["V"])
    args = [to_torch(x, dev) for x in (c.target, c.draft, c.tokens, c.uniforms)]
    tps = to_torch(c.temperature_per_seq, dev)
    for _ in range(3):
        out = sv.spec_verify_sample(*args, SAMPLE["T"], 0, SAMPLE["top_p"], tps, workspace=ws, stream=stream)
    ts = []
    for _ in range(iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        out = sv.spec_verify_sample(*args, SAMPLE["T"], 0, SAMPLE["top_p"], tps, workspace=ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return float(np.median(ts)), float(out[1].float().mean().item())


KERNEL_SOURCES = {
    "sample": ("sample_kernel.cu", "device_common.cuh", "internal.h"),
    "argmax": ("argmax_kernel.cu", "device_common.cuh", "internal.h"),
    "tree_sample": ("tree_sample_kernel.cu", "device_common.cuh", "internal.h"),
}


def kernel_source_hash(kernel: str):
    """Hash of the files a kernel is compiled from: a recorded DRAM traffic
    figure is used only while this hash is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "draft_token_verification_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(kernel)
        src = "argmax" if kernel.startswith("argmax") else kernel
        if e and e.get("kernel_source_hash") == kernel_source_hash(src):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples (every 200 ms) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads


def make_inputs(seed_offset: int = 0):
    s = W.config3(seed=3 + seed_offset, B=SAMPLE["B"], k=SAMPLE["k"], V=SAMPLE["V"])
    t = W.config4(seed=4 + seed_offset, B=TREE["B"], N=TREE["N"], V=TREE["V"], max_depth=TREE["depth"])
    return s, t


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as tdist

    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_rate(positions_per_rank_step: int, world: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank's positions over the slowest rank's time."""
    return positions_per_rank_step * world * steps / (elapsed_ms / 1e3)


def to_torch(arr, device=None, pin=False):
    import torch

    arr = np.ascontiguousarray(arr)
    t = torch.from_numpy(arr.view(np.int16) if arr.dtype == np.uint16 else arr)
    if arr.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    if pin:
        return t.pin_memory()
    return t.to(device) if device is not None else t


# ------------------------------------------------------------ GPU leg


def run_gpu(args, rank, world):
    import torch

    import draft_token_verification_gb300 as sv

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.build()
    sv.spec_sample_launch_mode({"auto": sv.SPEC_LAUNCH_AUTO, "fused": sv.SPEC_LAUNCH_FUSED, "rows": sv.SPEC_LAUNCH_ROWS,
                                "split": sv.SPEC_LAUNCH_SPLIT}[args.sample_launch])
    s, t = make_inputs(seed_offset=rank)
    d = {
        "target": to_torch(s.target, dev), "draft": to_torch(s.draft, dev), "tokens": to_torch(s.tokens, dev),
        "uniforms": to_torch(s.uniforms, dev), "greedy_target": to_torch(s.target, dev),
        "tree_logits": to_torch(t.logits, dev), "tree_tokens": to_torch(t.node_tokens, dev),
        "parents": to_torch(t.parents, dev),
    }
    B, k = s.B, s.k
    o = {
        "tok": torch.empty((B, k + 1), dtype=torch.int32, device=dev), "n": torch.empty(B, dtype=torch.int32, device=dev),
        "p": torch.empty((B, k), dtype=torch.float32, device=dev), "q": torch.empty((B, k), dtype=torch.float32, device=dev),
        "gtok": torch.empty((B, k + 1), dtype=torch.int32, device=dev), "gn": torch.empty(B, dtype=torch.int32, device=dev),
        "ttok": torch.empty((t.B, t.max_depth + 1), dtype=torch.int32, device=dev),
        "tpath": torch.empty((t.B, t.max_depth + 1), dtype=torch.int32, device=dev),
        "tn": torch.empty(t.B, dtype=torch.int32, device=dev),
    }
    # KV keep lists: chains from cache position 1000 + 100 b, trees from 2000 + 100 b
    kv = {"sbase": torch.arange(B, dtype=torch.int32, device=dev) * 100 + 1000,
          "tbase": torch.arange(t.B, dtype=torch.int32, device=dev) * 100 + 2000}
    for name, rows, keep in (("s", B, k + 1), ("t", t.B, t.max_depth + 2)):
        for f in ("src", "dst"):
            kv[name + f] = torch.empty((rows, keep), dtype=torch.int32, device=dev)
        kv[name + "len"] = torch.empty(rows, dtype=torch.int32, device=dev)
        kv[name + "moves"] = torch.empty(rows, dtype=torch.int32, device=dev)
    kv_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def kv_compact(path, n, base, prefix, rows, keep, st):
        sv.spec_kv_compact(n, base, path, max_keep=keep, out_status=kv_status, out_src=kv[prefix + "src"],
                           out_dst=kv[prefix + "dst"], out_new_len=kv[prefix + "len"],
                           out_num_moves=kv[prefix + "moves"], stream=st)
    ws = sv.Workspace(dev)
    stream = torch.cuda.current_stream()
    # --streams 3: the greedy chain and the greedy tree run on streams (and
    # workspaces) of their own beside the sampling call, joined at the end of
    # every step
    ws_g3, ws_t3 = sv.Workspace(dev), sv.Workspace(dev)
    s_g3, s_t3 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    conc = {"on": args.streams == 3}

    def step(ev=None, inputs=d):
        # events bracket each verification call alone (on its own stream); the
        # KV keep lists run between them
        if conc["on"]:
            ws_g, ws_t, s_g, s_t = ws_g3, ws_t3, s_g3, s_t3
        else:
            ws_g, ws_t, s_g, s_t = ws, ws, stream, stream
        if conc["on"]:
            fork = torch.cuda.Event()
            fork.record(stream)
            s_g.wait_event(fork)
            s_t.wait_event(fork)
        if ev is not None:
            ev[0].record(stream)
        sv.spec_verify_sample(inputs["target"], inputs["draft"], inputs["tokens"], inputs["uniforms"], SAMPLE["T"],
                              SAMPLE["top_k"], SAMPLE["top_p"], None, o["tok"], o["n"], o["p"], o["q"], ws, stream)
        if ev is not None:
            ev[1].record(stream)
        kv_compact(None, o["n"], kv["sbase"], "s", B, k + 1, stream)
        if ev is not None:
            ev[2].record(s_g)
        sv.spec_verify_greedy(inputs["greedy_target"], inputs["tokens"], o["gtok"], o["gn"], ws_g, s_g)
        if ev is not None:
            ev[3].record(s_g)
            ev[5].record(s_t)
        sv.spec_verify_tree_greedy(inputs["tree_logits"], inputs["tree_tokens"], inputs["parents"], TREE["depth"],
                                   o["ttok"], o["tpath"], o["tn"], ws_t, s_t)
        if ev is not None:
            ev[4].record(s_t)
        kv_compact(o["tpath"], o["tn"], kv["tbase"], "t", t.B, t.max_depth + 2, s_t)
        if conc["on"]:
            for st in (s_g, s_t):
                join = torch.cuda.Event()
                join.record(st)
                stream.wait_event(join)

    dist = world > 1
    if dist:
        import torch.distributed as tdist

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = sv.spec_get_status(ws)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        tdist.barrier()
    elapsed_ms = start.elapsed_time(end)
    per = np.array([[e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3]), e[5].elapsed_time(e[4])] for e in evs])
    # the same K steps with the other stream layout (reported beside the main line)
    conc["on"] = args.streams != 3
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    alt0 = torch.cuda.Event(enable_timing=True)
    alt1 = torch.cuda.Event(enable_timing=True)
    alt0.record(stream)
    for i in range(args.steps):
        step()
    alt1.record(stream)
    torch.cuda.synchronize()
    alt_ms = alt0.elapsed_time(alt1)
    if dist:
        alt_ms = max_over_ranks(alt_ms, dev)
    conc["on"] = args.streams == 3
    if dist:
        elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # acceptance statistics of the last step (MAL = accepted drafts per pass)
    n_acc = o["n"].cpu().numpy()
    gn = o["gn"].cpu().numpy()

    # -------- end to end through the C ABI with host buffers (pinned), copies timed
    e2e_steps = max(3, min(20, args.steps // 50))
    h = {key: to_torch(arr, pin=True) for key, arr in (
        ("target", s.target), ("draft", s.draft), ("tokens", s.tokens), ("uniforms", s.uniforms),
        ("tree_logits", t.logits), ("tree_tokens", t.node_tokens), ("parents", t.parents))}
    host_out = {key: torch.empty(o[key].shape, dtype=o[key].dtype).pin_memory() for key in ("tok", "n", "gtok", "gn", "ttok", "tn")}
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    # Two sets of device inputs: the next step's host-to-device copy runs on its
    # own stream while this step verifies (the link, about 210 GB/s here, is the
    # bound); every step still copies all of its inputs in and its results out.
    d_sets = [d, {key: torch.empty_like(d[key]) for key in h}]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        ds = d_sets[b]
        copy_stream.wait_event(freed[b])  # the set's previous step has finished with it
        with torch.cuda.stream(copy_stream):
            for key, v in h.items():
                ds[key].copy_(v, non_blocking=True)
        copied[b].record(copy_stream)
        stream.wait_event(copied[b])
        d_in = dict(ds)
        d_in["greedy_target"] = ds["target"]
        step(None, d_in)
        freed[b].record(stream)
        for key, v in host_out.items():
            v.copy_(o[key], non_blocking=True)

    for ev in freed:
        ev.record(stream)
    e2e_step(0)
    e2e_step(1)
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for ev in freed:
        ev.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if dist:
        e2e_ms = max_over_ranks(e2e_ms, dev)
    status |= sv.spec_get_status(ws) | sv.spec_get_status(ws_g3) | sv.spec_get_status(ws_t3)
    ts_us, ts_bytes, ts_mal = time_tree_sample(sv, dev, ws, stream, seed=4 + rank)
    status |= sv.spec_get_status(ws)
    tb_us, tb_mal = time_per_seq_temperature(sv, dev, ws, stream, seed=3 + rank)
    status |= sv.spec_get_status(ws) | int(kv_status.item())

    return dict(elapsed_ms=elapsed_ms, alt_ms=alt_ms, per=per, clk=clk, status=status, e2e_ms=e2e_ms, e2e_steps=e2e_steps,
                h2d=h2d, d2h=d2h, mal=float(n_acc.mean()), greedy_mal=float(gn.mean()),
                tree_sample=(ts_us, ts_bytes, ts_mal), per_seq_t=(tb_us, tb_mal),
                kv_moves=int(kv["tmoves"].sum().item()))


# ------------------------------------------------------------ CPU leg


def cpu_baseline(passes: int = 6, threads: int | None = None):
    """The float64 oracle, as it stands, on a bounded sample of the same
    workload: `passes` passes over the whole benchmark batch (64 sampling and
    64 greedy sequences, 8 trees), about 10-30 s of CPU work, spread over the
    host's cores one sequence or tree per task."""
    import oracle

    s, t = make_inputs()
    cores = threads or len(os.sched_getaffinity(0))
    jobs = []
    for _ in range(passes):
        for b in range(SAMPLE["B"]):
            jobs.append(("sample", b))
            jobs.append(("greedy", b))
        for b in range(TREE["B"]):
            jobs.append(("tree", b))

    def run(job):
        kind, b = job
        sl = slice(b, b + 1)
        t0 = time.perf_counter()
        if kind == "sample":
            oracle.verify_sample(s.target[sl], s.draft[sl], s.tokens[sl], s.uniforms[sl], SAMPLE["T"],
                                 SAMPLE["top_k"], SAMPLE["top_p"], all_rows=False)
            n = SAMPLE["k"]
        elif kind == "greedy":
            oracle.verify_greedy(s.target[sl], s.tokens[sl])
            n = SAMPLE["k"]
        else:
            oracle.verify_tree_greedy(t.logits[sl], t.node_tokens[sl], t.parents[sl], t.max_depth)
            n = TREE["N"] - 1
        return n, time.perf_counter() - t0

    oracle.build()
    t0 = time.perf_counter()
    with ThreadPoolExecutor(cores) as pool:
        done = list(pool.map(run, jobs))
    dt = time.perf_counter() - t0
    positions = sum(n for n, _ in done)
    cpu_s = sum(d for _, d in done)
    return {"value": positions / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{passes} passes over the benchmark batch (64 sampling + 64 greedy sequences, k=8, "
                      f"V=128256, and 8 trees of 60 nodes): {positions} positions, {cpu_s:.1f} s of CPU work, "
                      f"{dt:.2f} s on {cores} threads"}


# ------------------------------------------------------------ sweep


def run_sweep(args):
    """Sampling and greedy verification over the V = 152064 sweep: every B in
    1..256, k in 1..12 and draft noise sigma in {0.5, 2, 4} (T = 1, top-p 0.95
    for sampling).  Each call is timed alone with CUDA events after a 512 MB
    write that evicts L2, median of `iters`.  The draft-length scan of the
    Speedup Calculator (steps 1-3) is then fed with measured numbers: the
    acceptance rate alpha seen at each (B, sigma), and the verification cost
    per pass, fitted as a + b k over the five k and expressed in target
    forward passes of t_T = 2 bytes x target parameters / measured HBM
    bandwidth (one decode pass reads every weight once).  Adding a + b gamma
    to the calculator's cost gamma c + 1 divides the speedup by a constant and
    replaces c by (c + b) / (1 + a), so the best gamma is the calculator's
    scan at that effective c."""
    import torch

    import draft_token_verification_gb300 as sv

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    sv.build()
    stream = torch.cuda.current_stream()
    ws = sv.Workspace(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peak, peak_kind = measured_peaks()
    V = 152064
    iters = args.sweep_iters

    def timed(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(iters):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            out = fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return float(np.median(ts)), out

    points = []
    clocks = ClockSampler(0)
    clocks.start()
    only = None
    if args.sweep_points:
        only = {(int(b), int(kk), float(sg)) for b, kk, sg in (p.split(":") for p in args.sweep_points.split(","))}
    for sigma in W.C5_SIGMAS:
        for k in W.C5_DRAFTS:
            batches = [B for B in W.C5_BATCHES if only is None or (B, k, float(sigma)) in only]
            if not batches:
                continue
            Bmax = max(batches)
            tgt, drf, tok, uni = W.config5_device(Bmax, k, sigma, device=dev, V=V)
            for B in batches:
                t, d, x, u = tgt[:B], drf[:B], tok[:B], uni[:B]
                us_s, out = timed(lambda: sv.spec_verify_sample(t, d, x, u, 1.0, 0, 0.95, None, workspace=ws,
                                                                stream=stream, want_probs=False))
                n = out[1].cpu().numpy().astype(np.int64)
                prev = sv.spec_sample_launch_mode(sv.SPEC_LAUNCH_ROWS)
                us_r, rout = timed(lambda: sv.spec_verify_sample(t, d, x, u, 1.0, 0, 0.95, None, workspace=ws,
                                                                 stream=stream, want_probs=False))
                sv.spec_sample_launch_mode(sv.SPEC_LAUNCH_FUSED)
                us_f, fout = timed(lambda: sv.spec_verify_sample(t, d, x, u, 1.0, 0, 0.95, None, workspace=ws,
                                                                 stream=stream, want_probs=False))
                sv.spec_sample_launch_mode(prev)
                us_g, gout = timed(lambda: sv.spec_verify_greedy(t, x, workspace=ws, stream=stream))
                gn = gout[1].cpu().numpy()
                sb, gb = B * (2 * k + 1) * V * 2, B * (k + 1) * V * 2
                points.append({
                    "B": B, "k": k, "sigma": sigma,
                    "sample": {"us": us_s, "positions_per_s": B * k / us_s * 1e6, "sequences_per_s": B / us_s * 1e6,
                               "GB/s": sb / us_s / 1e3, "frac": sb / us_s / 1e3 / peak,
                               "mal": float(n.mean()), "accepted": int(n.sum()),
                               "tests": int(np.minimum(n + 1, k).sum())},
                    "sample_rows": {"us": us_r, "GB/s": sb / us_r / 1e3, "frac": sb / us_r / 1e3 / peak,
                                    "what": "the same call with SPEC_LAUNCH_ROWS (one CTA per row)"},
                    "sample_fused": {"us": us_f, "GB/s": sb / us_f / 1e3, "frac": sb / us_f / 1e3 / peak,
                                     "what": "the same call with SPEC_LAUNCH_FUSED (stream + tail items, draw)"},
                    "greedy": {"us": us_g, "positions_per_s": B * k / us_g * 1e6, "sequences_per_s": B / us_g * 1e6,
                               "GB/s": gb / us_g / 1e3, "frac": gb / us_g / 1e3 / peak, "mal": float(gn.mean())},
                })
            del tgt, drf, tok, uni
            torch.cuda.empty_cache()
    clk = clocks.stop()
    status = sv.spec_get_status(ws)

    # the draft-length scan on measured numbers
    t_target_us = 2.0 * args.target_params / (peak * 1e9) * 1e6
    scan = []
    for B in W.C5_BATCHES:
        kdone = [k for k in W.C5_DRAFTS if any(p["B"] == B and p["k"] == k for p in points)]
        if len(kdone) < 2:  # (a partial sweep: no fit for this batch)
            continue
        ks = np.array(kdone, float)
        us = np.array([np.median([p["sample"]["us"] for p in points if p["B"] == B and p["k"] == k])
                       for k in kdone])
        b, a = np.polyfit(ks, us, 1)  # us = a + b k
        for sigma in W.C5_SIGMAS:
            sel = [p for p in points if p["B"] == B and p["sigma"] == sigma]
            alpha = sum(p["sample"]["accepted"] for p in sel) / max(1, sum(p["sample"]["tests"] for p in sel))
            v0, v1 = a / t_target_us, b / t_target_us
            c_eff = (args.draft_cost + v1) / (1.0 + v0)
            g_calc, f_calc = sv.spec_best_gamma(alpha, args.draft_cost, 12)
            g_meas, f_meas = sv.spec_best_gamma(alpha, c_eff, 12)
            scan.append({"B": B, "sigma": sigma, "alpha": alpha, "verify_us": {"a": a, "b_per_draft": b},
                         "v0": v0, "v1": v1, "c_draft": args.draft_cost, "c_eff": c_eff,
                         "best_gamma_calculator": g_calc, "speedup_calculator": f_calc,
                         "best_gamma_measured_verify": g_meas, "speedup_measured_verify": f_meas / (1.0 + v0)})
    line = {"metric": "sweep: verified draft positions/s and sequences/s, V=152064 bf16", "unit": "positions/s",
            "dtype": "bf16", "data": "synthetic", "config": {
                "workload": "C5 sweep: B in 1,4,16,64,128,256; k in 1,2,4,8,12; sigma in 0.5,2,4; V=152064 bf16; "
                            "T=1, top-p 0.95 (sampling); greedy on the same rows",
                "l2": "512 MB written before every timed call", "iters": iters,
                "target_forward_us": t_target_us, "target_params": args.target_params,
                "draft_cost_c": args.draft_cost, "peak_gbs": peak, "peak_source": f"{peak_kind} hbm_gbs"},
            "clocks": clk, "status_bits": status, "points": points, "gamma_scan": scan}
    print(json.dumps(line))


# ------------------------------------------------------------------ main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="time the V=152064 sweep instead of the step")
    ap.add_argument("--sweep-iters", type=int, default=10)
    ap.add_argument("--streams", type=int, default=1, choices=[1, 3],
                    help="1: the step's calls in order on one stream; 3: greedy chain and greedy tree on streams "
                         "of their own beside the sampling call")
    ap.add_argument("--sweep-points", default=None,
                    help="only these sweep points, as B:k:sigma separated by commas (e.g. 64:8:2,256:12:4)")
    ap.add_argument("--sample-launch", default="auto", choices=["auto", "fused", "rows", "split"],
                    help="sampling kernels: the library's choice per call (default), fused stream + tail items, "
                         "one CTA per row, or stream / row / draw launches")
    ap.add_argument("--target-params", type=float, default=8.03e9,
                    help="target model parameters for the gamma scan (default: an 8B target)")
    ap.add_argument("--draft-cost", type=float, default=0.05,
                    help="draft forward / target forward time for the gamma scan")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        cb = cpu_baseline()
        steps_equiv = None
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": positions_per_step() / cb["value"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(), "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        del steps_equiv
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
    r = run_gpu(args, rank, world)
    if rank != 0:
        if world > 1:
            import torch.distributed as tdist

            tdist.destroy_process_group()
        return
    K = args.steps
    per = r["per"]
    # the step's sampling call: top-p 0.9 with one temperature, which the library's own choice runs fused
    step_launch = "fused" if args.sample_launch == "auto" else args.sample_launch
    pos = positions_per_step() * world
    value = job_rate(positions_per_step(), world, K, r["elapsed_ms"])
    peak, peak_kind = measured_peaks()
    t_sample = float(per[:, 0].mean()) / 1e3
    achieved = sample_bytes() / t_sample / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": r["elapsed_ms"] / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": workload_config(world),
        "clocks": r["clk"],
        "e2e": {"value": pos * r["e2e_steps"] / (r["e2e_ms"] / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "what": "through the C ABI from pinned host buffers: every step copies its inputs in and its results "
                        "out; the next step's copy (its own stream, a second set of device inputs) overlaps this "
                        "step's verification"},
        "sequences_per_s": {
            "step": (2 * SAMPLE["B"] + TREE["B"]) * world * K / (r["elapsed_ms"] / 1e3),
            "sample": SAMPLE["B"] / t_sample, "greedy": SAMPLE["B"] / (float(per[:, 1].mean()) / 1e3),
            "tree": TREE["B"] / (float(per[:, 2].mean()) / 1e3),
            "what": "sequences (chains or trees) verified per second: the whole step (64 sampled + 64 greedy "
                    "chains + 8 trees per GPU), and each kernel alone from its own events"},
        # sampling: fused stream+tail and draw kernels (rows: one row kernel); greedy; tree; two KV keep lists
        "gpu_launches": {"fused": 6, "rows": 5, "split": 7}[step_launch] * K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic("sample") if step_launch == "fused" else None,
                     "kernel": {"fused": "sampling verify: fused_kernel (stream + tail) + draw_kernel<bf16>, timed together",
                                "rows": "sampling verify: row_kernel<bf16> (one CTA per row)",
                                "split": "sampling verify: split_stream_kernel + split_row_kernel + "
                                         "split_draw_kernel<bf16>, timed together"}[step_launch],
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "kernels": {
            "sample": {"us": t_sample * 1e6, "GB/s": achieved, "frac": achieved / peak,
                       "algorithmic_bytes": sample_bytes(),
                       "traffic": recorded_traffic("sample") if step_launch == "fused" else None},
            "greedy": {"us": float(per[:, 1].mean()) * 1e3,
                       "GB/s": greedy_bytes() / (float(per[:, 1].mean()) / 1e3) / 1e9,
                       "frac": greedy_bytes() / (float(per[:, 1].mean()) / 1e3) / 1e9 / peak,
                       "algorithmic_bytes": greedy_bytes(), "traffic": recorded_traffic("argmax_chain")},
            "tree": {"us": float(per[:, 2].mean()) * 1e3,
                     "GB/s": tree_bytes() / (float(per[:, 2].mean()) / 1e3) / 1e9,
                     "frac": tree_bytes() / (float(per[:, 2].mean()) / 1e3) / 1e9 / peak,
                     "algorithmic_bytes": tree_bytes(), "traffic": recorded_traffic("argmax_tree")},
        },
        "outside_step": {
            "tree_sample": {"us": r["tree_sample"][0], "algorithmic_bytes": r["tree_sample"][1],
                            "GB/s": r["tree_sample"][1] / r["tree_sample"][0] / 1e3,
                            "frac": r["tree_sample"][1] / r["tree_sample"][0] / 1e3 / peak,
                            "mean_accepted": r["tree_sample"][2], "traffic": recorded_traffic("tree_sample"),
                            "what": "token-tree sampling verification, 8 trees x 60 nodes, depth <= 6, "
                                    "V=128256 bf16, T=1; plan + node + walk kernels, timed alone after an L2 flush"},
            "sample_per_seq_temperature": {
                "us": r["per_seq_t"][0], "GB/s": sample_bytes() / r["per_seq_t"][0] / 1e3,
                "frac": sample_bytes() / r["per_seq_t"][0] / 1e3 / peak,
                "sequences_per_s": SAMPLE["B"] / (r["per_seq_t"][0] / 1e6), "mean_accepted": r["per_seq_t"][1],
                "what": "the step's sampling workload with T_b ~ U(0.5, 1.2) per sequence (the library's choice "
                        "for a temperature per sequence: the split launch), timed alone "
                        "(median of 20; rows exceed L2)"},
        },
        "step_other_streams": {
            "value": job_rate(positions_per_step(), world, K, r["alt_ms"]), "unit": UNIT,
            "ms_per_step": r["alt_ms"] / K,
            "what": ("the same K steps with greedy chain and greedy tree on streams (and workspaces) of their own "
                     "beside the sampling call, joined at the end of every step" if args.streams == 1 else
                     "the same K steps with every call in order on one stream")},
        "acceptance": {"sample_mal": r["mal"], "greedy_mal": r["greedy_mal"], "k": SAMPLE["k"]},
        "boundary_rate": boundary_rates(),
        "kv_keep": {"tree_entries_moved_last_step": r["kv_moves"],
                    "what": "spec_kv_compact after the sampled chains and after the trees, inside every step"},
        "status_bits": r["status"],
    }
    line["config"]["sample_launch"] = args.sample_launch + (" (fused for this call)" if args.sample_launch == "auto" else "")
    line["config"]["streams"] = ("the step's calls in order on one stream" if args.streams == 1 else
                                 "greedy chain and greedy tree on streams of their own beside the sampling call, "
                                 "joined at the end of every step")
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as tdist

        tdist.destroy_process_group()


def boundary_rates():
    """Share of oracle decisions within 1e-6 of their edge on each recipe,
    from the committed oracle-only count (tests/golden/boundary_rates.json)."""
    path = os.path.join(ROOT, "tests", "golden", "boundary_rates.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: {"rate": v["rate"], "decisions": v["decisions"]} for k, v in d["configs"].items()}
    except Exception:
        return None


def workload_config(world: int = 1):
    return {
        "workload": "sampling verify B=64 k=8 V=128256 bf16 T=0.9 top-p 0.9 (+ greedy on the same target rows) "
                    "+ greedy tree 8x60 nodes depth<=6 V=128256 bf16",
        "B": SAMPLE["B"], "k": SAMPLE["k"], "V": SAMPLE["V"], "tree_B": TREE["B"], "tree_N": TREE["N"],
        "positions_per_step_per_gpu": positions_per_step(),
        "l2": "inputs larger than L2: each kernel's inputs were last touched >= 2x L2 bytes earlier",
        "parallelism": f"replicas{world}" if world > 1 else "single GPU",
        "drafts": "Gumbel-max samples of the unfiltered draft softmax at T",
    }


if __name__ == "__main__":
    main()
