"""Seeded synthetic inputs for draft-token verification.

This module only draws random numbers and lays them out: logit rows, draft
tokens, uniforms and tree shapes.  It holds none of the verification
arithmetic.  Both the CUDA path (through the tests and the benchmark) and the
float64 oracle (through the tests) receive the same arrays from here.

Logits are generated in float32 and, for bf16 workloads, rounded once to
bfloat16 (round to nearest even); bf16 arrays are returned as their raw 16-bit
patterns in uint16 arrays.  Draft tokens are drawn by the Gumbel-max trick,
argmax_t (D_t / T + G_t), optionally restricted to a caller-supplied candidate
mask (the tests pass the draft's filtered support; the benchmark passes none).

Workloads (sizes, value distributions and filters):
  C1  sampling, B=1, k=4, V=32000, fp32; L ~ N(0, 2^2), D = L + N(0, 1);
      T = 1, no filter; uniforms [1][k+2] from seed 0; greedy on the same L.
  C2  sampling, B=16, k=5, V=32000, bf16; L ~ N(0, 3^2) - 1.1 ln(id + 1)
      (a Zipf(1.1) log-bias over token ids), D = L + N(0, 1.5^2);
      T = 0.7, top-k 50 on both.
  C3  sampling, B=64, k=8, V=128256, bf16; L ~ N(0, 4^2),
      D = 0.8 L + N(0, 2^2); T = 0.9, top-p 0.9 on both; variant with a
      per-sequence temperature T_b ~ U(0.5, 1.2).
  C4  greedy token tree, B=8 trees of N=60 nodes, depth <= 6, 1-4 children
      per expanded node (breadth-first), V=128256, bf16 rows ~ N(0, 3^2);
      node token = argmax of the parent's row with probability 0.6, else
      uniform over V.
  C5  sweep, V=152064, bf16, B in {1,4,16,64,128,256}, k in {1,2,4,8,12};
      L ~ N(0, 3^2), D = L + N(0, sigma^2), sigma in {0.5, 2, 4};
      T = 1, top-p 0.95; sampling and greedy.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

BF16 = "bf16"
F32 = "f32"


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(arr: np.ndarray) -> np.ndarray:
    return bits_to_f32(arr) if arr.dtype == np.uint16 else np.asarray(arr, dtype=np.float32)


def f32(x: float) -> float:
    """The float32 value nearest to x, as a Python float."""
    return float(np.float32(x))


def _rng(ss: np.random.SeedSequence) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(ss))


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(x) if dtype == BF16 else np.ascontiguousarray(x, dtype=np.float32)


MaskFn = Callable[[np.ndarray, float], Optional[np.ndarray]]


def gumbel_drafts(draft: np.ndarray, temps: np.ndarray, rng: np.random.Generator,
                  mask_fn: Optional[MaskFn] = None) -> np.ndarray:
    """Draft tokens x[b][i] = argmax_t (D[b,i,t] / T_b + Gumbel noise), over the
    candidate set mask_fn(row, T_b) when one is given."""
    B, k, V = draft.shape
    out = np.empty((B, k), np.int32)
    for b in range(B):
        for i in range(k):
            row = draft[b, i]
            g = -np.log(-np.log(rng.random(V, dtype=np.float64).clip(1e-300, None)))
            score = as_f32(row).astype(np.float64) / float(temps[b]) + g
            if mask_fn is not None:
                mask = mask_fn(row, float(temps[b]))
                if mask is not None:
                    score = np.where(mask, score, -np.inf)
            out[b, i] = int(np.argmax(score))
    return out


@dataclass
class SampleCase:
    name: str
    dtype: str
    target: np.ndarray            # [B][k+1][V]
    draft: np.ndarray             # [B][k][V]
    tokens: np.ndarray            # [B][k] int32
    uniforms: np.ndarray          # [B][k+2] float32
    temperature: float
    top_k: int
    top_p: float
    temperature_per_seq: Optional[np.ndarray] = None
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def k(self) -> int:
        return self.target.shape[1] - 1

    @property
    def V(self) -> int:
        return self.target.shape[2]

    def temps(self) -> np.ndarray:
        if self.temperature_per_seq is not None:
            return self.temperature_per_seq
        return np.full(self.B, self.temperature, np.float32)


@dataclass
class TreeSampleCase:
    name: str
    dtype: str
    logits: np.ndarray            # [B][N][V] target row of every node
    draft: np.ndarray             # [B][N][V] draft row the children of every node came from
    node_tokens: np.ndarray       # [B][N] int32 (node 0 = root, token unused)
    parents: np.ndarray           # [B][N] int32
    uniforms: np.ndarray          # [B][N] float32: u_0 final draw, u_j test of node j
    max_depth: int
    temperature: float
    seed: int = 0

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def N(self) -> int:
        return self.logits.shape[1]

    @property
    def V(self) -> int:
        return self.logits.shape[2]


@dataclass
class TreeCase:
    name: str
    dtype: str
    logits: np.ndarray            # [B][N][V]
    node_tokens: np.ndarray       # [B][N] int32 (node 0 = root, token unused)
    parents: np.ndarray           # [B][N] int32
    max_depth: int
    seed: int = 0

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def N(self) -> int:
        return self.logits.shape[1]

    @property
    def V(self) -> int:
        return self.logits.shape[2]


def _uniforms(rng: np.random.Generator, B: int, k: int) -> np.ndarray:
    return rng.random((B, k + 2), dtype=np.float32)


def _finish_sample(name, dtype, L, D, T, top_k, top_p, ss, tps=None, mask_fn=None, seed=0, meta=None):
    s_tok, s_u = ss
    target = _cast(L, dtype)
    draft = _cast(D, dtype)
    B = target.shape[0]
    temps = tps if tps is not None else np.full(B, f32(T), np.float32)
    tokens = gumbel_drafts(draft, temps, _rng(s_tok), mask_fn)
    uniforms = _uniforms(_rng(s_u), B, target.shape[1] - 1)
    # the C ABI takes temperature and top_p as float32: both sides get those values
    return SampleCase(name, dtype, target, draft, tokens, uniforms, f32(T), int(top_k), f32(top_p),
                      tps, seed, meta or {})


def config1(mask_fn: Optional[MaskFn] = None, seed: int = 0, B: int = 1) -> SampleCase:
    """C1: B=1, k=4, V=32000, fp32, T=1, no filter, everything from seed 0
    (other seeds and batch sizes give more sequences of the same recipe)."""
    k, V = 4, 32000
    ss = np.random.SeedSequence(seed)
    s_l, s_d, s_tok, s_u = ss.spawn(4)
    L = _rng(s_l).normal(0.0, 2.0, size=(B, k + 1, V)).astype(np.float32)
    D = (L[:, :k] + _rng(s_d).normal(0.0, 1.0, size=(B, k, V))).astype(np.float32)
    return _finish_sample("C1", F32, L, D, 1.0, 0, 1.0, (s_tok, s_u), mask_fn=mask_fn, seed=seed)


def config2(seed: int = 2, mask_fn: Optional[MaskFn] = None, B: int = 16) -> SampleCase:
    """C2: B=16, k=5, V=32000, bf16, Zipf(1.1) log-bias, T=0.7, top-k 50."""
    k, V = 5, 32000
    ss = np.random.SeedSequence(seed)
    s_l, s_d, s_tok, s_u = ss.spawn(4)
    bias = (-1.1 * np.log(np.arange(V, dtype=np.float64) + 1.0)).astype(np.float32)
    L = (_rng(s_l).normal(0.0, 3.0, size=(B, k + 1, V)).astype(np.float32) + bias).astype(np.float32)
    D = (L[:, :k] + _rng(s_d).normal(0.0, 1.5, size=(B, k, V))).astype(np.float32)
    return _finish_sample("C2", BF16, L, D, 0.7, 50, 1.0, (s_tok, s_u), mask_fn=mask_fn, seed=seed)


def config3(seed: int = 3, per_seq_temperature: bool = False, mask_fn: Optional[MaskFn] = None,
            B: int = 64, k: int = 8, V: int = 128256) -> SampleCase:
    """C3: B=64, k=8, V=128256, bf16, T=0.9 (or T_b ~ U(0.5, 1.2)), top-p 0.9."""
    ss = np.random.SeedSequence(seed)
    s_l, s_d, s_tok, s_u, s_t = ss.spawn(5)
    L = _rng(s_l).normal(0.0, 4.0, size=(B, k + 1, V)).astype(np.float32)
    D = (0.8 * L[:, :k] + _rng(s_d).normal(0.0, 2.0, size=(B, k, V))).astype(np.float32)
    tps = _rng(s_t).uniform(0.5, 1.2, size=B).astype(np.float32) if per_seq_temperature else None
    name = "C3-Tb" if per_seq_temperature else "C3"
    return _finish_sample(name, BF16, L, D, 0.9, 0, 0.9, (s_tok, s_u), tps=tps, mask_fn=mask_fn, seed=seed)


def config5(B: int, k: int, sigma: float, seed: int = 5, mask_fn: Optional[MaskFn] = None,
            V: int = 152064) -> SampleCase:
    """C5 sweep point: V=152064, bf16, L ~ N(0, 3^2), D = L + N(0, sigma^2), T=1, top-p 0.95."""
    ss = np.random.SeedSequence([seed, B, k, int(round(sigma * 100))])
    s_l, s_d, s_tok, s_u = ss.spawn(4)
    L = _rng(s_l).normal(0.0, 3.0, size=(B, k + 1, V)).astype(np.float32)
    D = (L[:, :k] + _rng(s_d).normal(0.0, sigma, size=(B, k, V))).astype(np.float32)
    return _finish_sample(f"C5-B{B}-k{k}-s{sigma:g}", BF16, L, D, 1.0, 0, 0.95, (s_tok, s_u),
                          mask_fn=mask_fn, seed=seed, meta=dict(sigma=sigma))


def config5_device(B: int, k: int, sigma: float, seed: int = 5, device="cuda", V: int = 152064):
    """C5 sweep point drawn on the device (torch's Philox generator), for the
    benchmark's sweep, where numpy would take minutes: the recipe of config5
    (L ~ N(0, 3^2), D = L + N(0, sigma^2), both rounded to bf16, drafts by
    Gumbel-max on the bf16 draft rows at T = 1, uniforms U[0, 1)) from other
    random streams.  Returns (target, draft, tokens, uniforms) torch tensors."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([seed, B, k, int(round(sigma * 100))]).generate_state(1)[0]))
    target = (torch.randn((B, k + 1, V), generator=g, device=device) * 3.0)
    draft = (target[:, :k] + sigma * torch.randn((B, k, V), generator=g, device=device)).to(torch.bfloat16)
    target = target.to(torch.bfloat16)
    tokens = torch.empty((B, k), dtype=torch.int32, device=device)
    for b in range(B):  # one sequence at a time keeps the noise buffer small
        u = torch.rand((k, V), generator=g, device=device, dtype=torch.float64).clamp_min(1e-300)
        score = draft[b].double() - torch.log(-torch.log(u))
        tokens[b] = score.argmax(dim=-1).to(torch.int32)
    uniforms = torch.rand((B, k + 2), generator=g, device=device, dtype=torch.float32)
    return target, draft, tokens, uniforms


C5_BATCHES = (1, 4, 16, 64, 128, 256)
C5_DRAFTS = (1, 2, 4, 8, 12)
C5_SIGMAS = (0.5, 2.0, 4.0)


def tree_parents(rng: np.random.Generator, n_nodes: int, max_depth: int, max_children: int = 4) -> np.ndarray:
    """Breadth-first tree: every dequeued node above max_depth gets U{1..max_children}
    children until n_nodes exist; if the queue empties first, nodes above max_depth
    get one more child each, in index order."""
    parents = [-1]
    depth = [0]
    queue = deque([0])
    while queue and len(parents) < n_nodes:
        u = queue.popleft()
        if depth[u] >= max_depth:
            continue
        for _ in range(int(rng.integers(1, max_children + 1))):
            if len(parents) >= n_nodes:
                break
            parents.append(u)
            depth.append(depth[u] + 1)
            queue.append(len(parents) - 1)
    while len(parents) < n_nodes:
        for u in range(len(parents)):
            if len(parents) >= n_nodes:
                break
            if depth[u] < max_depth:
                parents.append(u)
                depth.append(depth[u] + 1)
    return np.asarray(parents, np.int32)


def config4(seed: int = 4, B: int = 8, N: int = 60, V: int = 128256, max_depth: int = 6,
            p_match: float = 0.6, sigma: float = 3.0, dtype: str = BF16) -> TreeCase:
    """C4: B=8 trees, N=60 nodes, depth <= 6, bf16 rows ~ N(0, 3^2), V=128256."""
    ss = np.random.SeedSequence(seed)
    s_l, s_t, s_k = ss.spawn(3)
    rl, rt = _rng(s_l), _rng(s_t)
    logits = _cast(rl.normal(0.0, sigma, size=(B, N, V)).astype(np.float32), dtype)
    parents = np.stack([tree_parents(rt, N, max_depth) for _ in range(B)])
    rk = _rng(s_k)
    tokens = np.full((B, N), -1, np.int32)
    for b in range(B):
        am = np.argmax(as_f32(logits[b]), axis=-1)  # lowest index on ties
        for j in range(1, N):
            if rk.random() < p_match:
                tokens[b, j] = am[parents[b, j]]
            else:
                tokens[b, j] = rk.integers(0, V)
    return TreeCase("C4", dtype, logits, tokens, parents, max_depth, seed)


def random_sample_case(B: int, k: int, V: int, dtype: str = BF16, seed: int = 0, sigma: float = 3.0,
                       noise: float = 1.0, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                       per_seq_temperature: bool = False, mask_fn: Optional[MaskFn] = None,
                       quantize: Optional[float] = None, spike: Optional[float] = None) -> SampleCase:
    """Small random case for edge coverage.  ``quantize`` rounds logits to a grid
    (many exact ties); ``spike`` adds that much to one random token of every
    target row and to the same token of the draft row at that position (one
    token towering over the rest)."""
    ss = np.random.SeedSequence([seed, B, k, V])
    s_l, s_d, s_tok, s_u, s_t = ss.spawn(5)
    L = _rng(s_l).normal(0.0, sigma, size=(B, k + 1, V)).astype(np.float32)
    D = (L[:, :k] + _rng(s_d).normal(0.0, noise, size=(B, k, V))).astype(np.float32)
    if spike:
        at = _rng(ss.spawn(1)[0]).integers(0, V, size=(B, k + 1))
        for b in range(B):
            for j in range(k + 1):
                L[b, j, at[b, j]] += np.float32(spike)
                if j < k:
                    D[b, j, at[b, j]] += np.float32(spike)
    if quantize:
        L = (np.round(L / quantize) * quantize).astype(np.float32)
        D = (np.round(D / quantize) * quantize).astype(np.float32)
    tps = _rng(s_t).uniform(0.5, 1.2, size=B).astype(np.float32) if per_seq_temperature else None
    return _finish_sample(f"rand-B{B}-k{k}-V{V}", dtype, L, D, temperature, top_k, top_p, (s_tok, s_u),
                          tps=tps, mask_fn=mask_fn, seed=seed)


def random_tree_case(B: int, N: int, V: int, max_depth: int, seed: int = 0, dtype: str = BF16,
                     p_match: float = 0.6, sigma: float = 3.0, quantize: Optional[float] = None,
                     max_children: int = 4) -> TreeCase:
    ss = np.random.SeedSequence([seed, B, N, V, max_depth])
    s_l, s_t, s_k = ss.spawn(3)
    x = _rng(s_l).normal(0.0, sigma, size=(B, N, V)).astype(np.float32)
    if quantize:
        x = (np.round(x / quantize) * quantize).astype(np.float32)
    logits = _cast(x, dtype)
    rt = _rng(s_t)
    parents = np.stack([tree_parents(rt, N, max_depth, max_children) for _ in range(B)])
    rk = _rng(s_k)
    tokens = np.full((B, N), -1, np.int32)
    for b in range(B):
        am = np.argmax(as_f32(logits[b]), axis=-1)
        for j in range(1, N):
            tokens[b, j] = am[parents[b, j]] if rk.random() < p_match else rk.integers(0, V)
    return TreeCase(f"tree-B{B}-N{N}-V{V}", dtype, logits, tokens, parents, max_depth, seed)


def tree_sample_case(B: int, N: int, V: int, max_depth: int, seed: int = 0, dtype: str = BF16,
                     sigma: float = 3.0, noise: float = 1.0, temperature: float = 1.0,
                     max_children: int = 4) -> TreeSampleCase:
    """Draft tree for sampling verification: target rows NL ~ N(0, sigma^2),
    draft rows DL = NL + N(0, noise^2) per node, breadth-first parents (as in
    the greedy tree cases) and every child's token drawn from its parent's
    draft distribution softmax(DL[parent] / T) by the Gumbel-max trick, so
    siblings are independent draws from q."""
    ss = np.random.SeedSequence([seed, B, N, V, max_depth, 7])
    s_l, s_d, s_t, s_k, s_u = ss.spawn(5)
    x = _rng(s_l).normal(0.0, sigma, size=(B, N, V)).astype(np.float32)
    d = (x + _rng(s_d).normal(0.0, noise, size=(B, N, V))).astype(np.float32)
    logits, draft = _cast(x, dtype), _cast(d, dtype)
    rt = _rng(s_t)
    parents = np.stack([tree_parents(rt, N, max_depth, max_children) for _ in range(B)])
    rk = _rng(s_k)
    tokens = np.full((B, N), -1, np.int32)
    for b in range(B):
        rows = as_f32(draft[b]).astype(np.float64) / float(temperature)
        for j in range(1, N):
            g = -np.log(-np.log(rk.random(V, dtype=np.float64).clip(1e-300, None)))
            tokens[b, j] = int(np.argmax(rows[parents[b, j]] + g))
    uniforms = _rng(s_u).random((B, N), dtype=np.float32)
    return TreeSampleCase(f"tree-sample-B{B}-N{N}-V{V}", dtype, logits, draft, tokens, parents, uniforms,
                          max_depth, float(temperature), seed)


@dataclass
class KvCase:
    """Inputs of the KV keep-list step: accept counts, cache positions of the
    roots, accepted paths (None for chains) and an optional block table."""
    num_accepted: np.ndarray
    kv_base: np.ndarray
    path: Optional[np.ndarray]
    block_table: Optional[np.ndarray]
    block_size: int
    max_keep: int
    entries: int          # cache entries the pass wrote per sequence (N, or k + 1)


def kv_case(B: int, N: int, max_depth: int, seed: int = 0, chain: bool = False, block_size: int = 0,
            base_max: int = 4000) -> KvCase:
    """B sequences whose pass wrote N entries each (a chain: N = k + 1).
    n ~ U{0..max_depth}; a tree path is n distinct node ids from 1..N-1 in
    increasing order (the shape every root-to-node path of a tree whose
    parents precede their children has), -1 padded to max_depth + 1 entries;
    roots at positions U{0..base_max}.  With block_size > 0 every sequence
    gets ceil((base_max + N) / block_size) logical blocks mapped to distinct
    physical blocks of one shared pool, in random order."""
    rng = _rng(np.random.SeedSequence(seed))
    n = rng.integers(0, max_depth + 1, B).astype(np.int32)
    base = rng.integers(0, base_max + 1, B).astype(np.int32)
    path = None
    if not chain:
        path = np.full((B, max_depth + 1), -1, np.int32)
        for b in range(B):
            path[b, :n[b]] = np.sort(rng.choice(np.arange(1, N), size=n[b], replace=False))
    table = None
    if block_size > 0:
        M = -(-(base_max + N) // block_size)
        table = rng.permutation(B * M).astype(np.int32).reshape(B, M)
    return KvCase(n, base, path, table, block_size, (N if chain else max_depth + 1), N)
