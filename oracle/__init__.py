"""Float64 CPU oracle for draft-token verification (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, float64, full sorts, sequential
scans); this module compiles it with gcc and marshals numpy arrays through
ctypes.  ``exact.py`` holds an independent rational-arithmetic enumerator of
the verification law used to pin the oracle.

Logit arrays are passed either as float32 (dtype ``"f32"``) or as the raw
16-bit patterns of bfloat16 values in a uint16 array (dtype ``"bf16"``); the C
code widens bf16 to float64 exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1

FLAG_ACCEPT_BOUNDARY = 1
FLAG_DRAW_BOUNDARY = 2
FLAG_DEGENERATE = 4
FLAG_CUT_BOUNDARY = 8
FLAG_BAD_TOKEN = 16
FLAG_BAD_ROW = 32
FLAG_BAD_PARENT = 64
FLAG_DEPTH = 128
#: flags that mark a sequence whose outcome sits within 1e-6 of a decision edge
BOUNDARY_FLAGS = FLAG_ACCEPT_BOUNDARY | FLAG_DRAW_BOUNDARY | FLAG_DEGENERATE | FLAG_CUT_BOUNDARY


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_row_probs.argtypes = [P, I, I, D, I, D, P, P, P, P]
            lib.oracle_row_probs.restype = I
            lib.oracle_verify_sample.argtypes = [P, P, I, P, P, I, I, I, D, P, I, D, I, P, P, P, P, P, P]
            lib.oracle_verify_sample.restype = I
            lib.oracle_verify_greedy.argtypes = [P, I, P, I, I, I, P, P]
            lib.oracle_verify_greedy.restype = I
            lib.oracle_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P]
            lib.oracle_verify_tree_sample.argtypes = [P, P, I, P, P, P, I, I, I, I, D, P, P, P, P, P, P]
            lib.oracle_verify_tree_greedy.restype = I
            for name in ("oracle_expected_tokens_series", "oracle_expected_tokens_closed"):
                getattr(lib, name).argtypes = [D, I]
                getattr(lib, name).restype = D
            lib.oracle_improvement_factor.argtypes = [D, I, D]
            lib.oracle_improvement_factor.restype = D
            lib.oracle_break_even.argtypes = [I]
            lib.oracle_break_even.restype = D
            lib.oracle_best_gamma.argtypes = [D, D, I, ctypes.POINTER(D)]
            lib.oracle_best_gamma.restype = I
            lib.oracle_first_draft_check.argtypes = [P, I, P, I, I, P, P]
            lib.oracle_first_draft_check.restype = I
            _lib = lib
    return _lib


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return F32
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def row_probs(row: np.ndarray, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0):
    """Filtered, normalised distribution of one logit row.

    Returns (probs[V] float64, cut_margin, last_kept_id, first_dropped_id, ok).
    """
    row = np.ascontiguousarray(row)
    V = row.shape[-1]
    probs = np.empty(V, dtype=np.float64)
    margin = ctypes.c_double()
    lo = ctypes.c_int()
    hi = ctypes.c_int()
    rc = _load().oracle_row_probs(
        _ptr(row), _dtype_code(row), V, float(temperature), int(top_k), float(top_p),
        _ptr(probs), ctypes.byref(margin), ctypes.byref(lo), ctypes.byref(hi),
    )
    return probs, margin.value, lo.value, hi.value, rc == 0


def verify_sample(target, draft, tokens, uniforms, temperature=1.0, top_k=0, top_p=1.0,
                  temperature_per_seq=None, all_rows=True):
    """Speculative-sampling verification of B sequences.

    target [B][k+1][V], draft [B][k][V] (float32 or bf16 bits), tokens [B][k]
    int32, uniforms [B][k+2] float32.  Returns a dict with tokens [B][k+1],
    n [B], p_draft / q_draft [B][k], flags [B], margin [B].
    """
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    B, k1, V = target.shape
    k = k1 - 1
    assert draft.shape == (B, k, V) and draft.dtype == target.dtype
    assert tokens.shape == (B, k) and uniforms.shape == (B, k + 2)
    tps = None if temperature_per_seq is None else np.ascontiguousarray(temperature_per_seq, dtype=np.float32)
    out = dict(
        tokens=np.empty((B, k + 1), np.int32), n=np.empty(B, np.int32),
        p_draft=np.empty((B, k), np.float64), q_draft=np.empty((B, k), np.float64),
        flags=np.empty(B, np.uint32), margin=np.empty(B, np.float64),
    )
    _load().oracle_verify_sample(
        _ptr(target), _ptr(draft), _dtype_code(target), _ptr(tokens), _ptr(uniforms),
        B, k, V, float(temperature), _ptr(tps), int(top_k), float(top_p), int(bool(all_rows)),
        _ptr(out["tokens"]), _ptr(out["n"]), _ptr(out["p_draft"]), _ptr(out["q_draft"]),
        _ptr(out["flags"]), _ptr(out["margin"]),
    )
    return out


def verify_greedy(target, tokens):
    """Greedy chain verification: target [B][k+1][V], tokens [B][k]."""
    target = np.ascontiguousarray(target)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B, k1, V = target.shape
    k = k1 - 1
    out = dict(tokens=np.empty((B, k + 1), np.int32), n=np.empty(B, np.int32))
    _load().oracle_verify_greedy(_ptr(target), _dtype_code(target), _ptr(tokens), B, k, V,
                                 _ptr(out["tokens"]), _ptr(out["n"]))
    return out


def first_draft_check(prev_rows, draft0):
    """Rejection fast path: prev_rows [B][V] (the previous step's logits), draft0 [B]."""
    prev_rows = np.ascontiguousarray(prev_rows)
    draft0 = np.ascontiguousarray(draft0, dtype=np.int32)
    B, V = prev_rows.shape
    out = dict(accept=np.empty(B, np.int32), argmax=np.empty(B, np.int32))
    _load().oracle_first_draft_check(_ptr(prev_rows), _dtype_code(prev_rows), _ptr(draft0), B, V,
                                     _ptr(out["accept"]), _ptr(out["argmax"]))
    return out


def verify_tree_greedy(logits, node_tokens, parents, max_depth):
    """Greedy token-tree verification: logits [B][N][V], node_tokens/parents [B][N]."""
    logits = np.ascontiguousarray(logits)
    node_tokens = np.ascontiguousarray(node_tokens, dtype=np.int32)
    parents = np.ascontiguousarray(parents, dtype=np.int32)
    B, N, V = logits.shape
    D = max_depth + 1
    out = dict(tokens=np.empty((B, D), np.int32), path=np.empty((B, D), np.int32),
               n=np.empty(B, np.int32), flags=np.empty(B, np.uint32))
    _load().oracle_verify_tree_greedy(
        _ptr(logits), _dtype_code(logits), _ptr(node_tokens), _ptr(parents), B, N, V, int(max_depth),
        _ptr(out["tokens"]), _ptr(out["path"]), _ptr(out["n"]), _ptr(out["flags"]),
    )
    return out


def verify_tree_sample(logits, draft_logits, node_tokens, parents, uniforms, max_depth,
                       temperature=1.0, temperature_per_tree=None):
    """Token-tree sampling verification.

    logits, draft_logits [B][N][V] (same dtype); node_tokens, parents [B][N];
    uniforms [B][N] float32 (u_0 the final draw, u_j the test of node j);
    temperature_per_tree [B] float32 or None (then the scalar temperature).
    Returns tokens / path [B][max_depth+1], n [B], flags [B], margin [B].
    """
    logits = np.ascontiguousarray(logits)
    draft_logits = np.ascontiguousarray(draft_logits)
    if draft_logits.dtype != logits.dtype or draft_logits.shape != logits.shape:
        raise ValueError("logits and draft_logits must share dtype and shape")
    node_tokens = np.ascontiguousarray(node_tokens, dtype=np.int32)
    parents = np.ascontiguousarray(parents, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    tpt = None if temperature_per_tree is None else np.ascontiguousarray(temperature_per_tree, dtype=np.float32)
    B, N, V = logits.shape
    D = max_depth + 1
    out = dict(tokens=np.empty((B, D), np.int32), path=np.empty((B, D), np.int32),
               n=np.empty(B, np.int32), flags=np.empty(B, np.uint32), margin=np.empty(B, np.float64))
    rc = _load().oracle_verify_tree_sample(
        _ptr(logits), _ptr(draft_logits), _dtype_code(logits), _ptr(node_tokens), _ptr(parents),
        _ptr(uniforms), B, N, V, int(max_depth), float(temperature), _ptr(tpt), _ptr(out["tokens"]),
        _ptr(out["path"]), _ptr(out["n"]), _ptr(out["flags"]), _ptr(out["margin"]),
    )
    if rc != 0:
        raise ValueError("oracle_verify_tree_sample rejected its arguments")
    return out


def expected_tokens_series(alpha: float, gamma: int) -> float:
    return _load().oracle_expected_tokens_series(float(alpha), int(gamma))


def expected_tokens_closed(alpha: float, gamma: int) -> float:
    return _load().oracle_expected_tokens_closed(float(alpha), int(gamma))


def improvement_factor(alpha: float, gamma: int, c: float) -> float:
    return _load().oracle_improvement_factor(float(alpha), int(gamma), float(c))


def break_even(k: int) -> float:
    return _load().oracle_break_even(int(k))


def best_gamma(alpha: float, c: float, gamma_max: int = 12):
    """Speedup Calculator's draft-length scan: (gamma, speedup) of the best gamma in 1..gamma_max."""
    best = ctypes.c_double()
    g = _load().oracle_best_gamma(float(alpha), float(c), int(gamma_max), ctypes.byref(best))
    return g, best.value


def kv_compact(num_accepted, kv_base, path=None, block_table=None, block_size=0, max_keep=None):
    """KV-cache keep list after a verification pass, written out per sequence.

    "Towards Green Text Generation: Memory-Based Speculative Decoding",
    section 2.4 (KV-cached regime): on rejection the cache is cut back to the
    accepted prefix.  Edge Inference Notes, "One decode round, end to end": the
    longest agreed path is committed and the other branches collapse.  Reading
    taken: the pass wrote node j's entry (node 0 the root, the last committed
    token; a chain's node j is its draft j - 1) at logical position base + j;
    the kept entries are the root's and the path's, in path order, and go to
    positions base, base + 1, ..., base + n.  A paged cache maps position p
    to block_table[p // block_size] * block_size + p % block_size.

    Returns (src [B][max_keep], dst [B][max_keep], new_len [B], moves [B],
    bad [B]); a sequence whose path is not strictly increasing from the root,
    whose n does not fit, or whose lookups fall outside its table is bad and
    gets -1 everywhere and 0 moves.
    """
    n_all = np.asarray(num_accepted, np.int64)
    base_all = np.asarray(kv_base, np.int64)
    B = len(n_all)
    if max_keep is None:
        max_keep = np.asarray(path).shape[1] + 1
    src = np.full((B, max_keep), -1, np.int32)
    dst = np.full((B, max_keep), -1, np.int32)
    new_len = np.full(B, -1, np.int32)
    moves = np.zeros(B, np.int32)
    bad = np.zeros(B, bool)
    int_max = 2**31 - 1

    for b in range(B):
        n, base = int(n_all[b]), int(base_all[b])

        def slot(pos):
            if block_table is None:
                return pos if pos <= int_max else None
            row = block_table[b]
            blk = pos // block_size
            if blk >= len(row) or int(row[blk]) < 0:
                return None
            s = int(row[blk]) * block_size + pos % block_size
            return s if s <= int_max else None

        ok = n >= 0 and n + 1 <= max_keep and base >= 0 and base + n + 1 <= int_max
        if ok and path is not None and n > np.asarray(path).shape[1]:
            ok = False
        kept = []
        if ok:
            kept = [0] + ([int(path[b][d]) for d in range(n)] if path is not None else list(range(1, n + 1)))
            ok = all(kept[d] > kept[d - 1] for d in range(1, n + 1))
        pairs = []
        if ok:
            for d in range(n + 1):
                s, t = slot(base + kept[d]), slot(base + d)
                if s is None or t is None:
                    ok = False
                    break
                pairs.append((s, t))
        if not ok:
            bad[b] = True
            continue
        for d, (s, t) in enumerate(pairs):
            src[b, d], dst[b, d] = s, t
        new_len[b] = base + n + 1
        moves[b] = sum(1 for d in range(n + 1) if kept[d] != d)
    return src, dst, new_len, moves, bad
