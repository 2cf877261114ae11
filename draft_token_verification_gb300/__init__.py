"""Python binding of libspecverify.so (draft-token verification on GB300).

Argument marshalling only: every step of verification runs in the library's
CUDA kernels.  Tensors must be CUDA tensors; PyTorch supplies device memory
and the current stream.  The binding fails loudly if the library is missing:
there is no CPU fallback.

Entry points (same names as the C ABI in include/spec_verify.h):
  spec_verify_sample, spec_verify_greedy, spec_verify_tree_greedy, spec_verify_tree_sample,
  spec_verify_sample_noalloc, spec_transform_probs, spec_get_status, spec_verify_workspace_size,
  spec_error_string, spec_expected_tokens, spec_improvement_factor,
  spec_break_even_acceptance
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SPEC_F32 = 0
SPEC_BF16 = 1

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = -1
SPEC_ERR_DTYPE = -2
SPEC_ERR_WORKSPACE = -3
SPEC_ERR_LAUNCH = -4
SPEC_ERR_DEVICE_DATA = -5
SPEC_ERR_TIMEOUT = -6
SPEC_ERR_UNSUPPORTED = -7
SPEC_ERR_SCRATCH_LIMIT = -8

SPEC_STATUS_BAD_TOKEN = 1
SPEC_STATUS_BAD_ROW = 2
SPEC_STATUS_BAD_PARENT = 4
SPEC_STATUS_DEPTH = 8
SPEC_STATUS_TIMEOUT = 16
SPEC_STATUS_BAD_KV = 32

SPEC_MAX_K = 31
SPEC_MAX_TREE_NODES = 1024
SPEC_NOALLOC_MAX_B = 256
SPEC_NOALLOC_MAX_UNITS = 256

EXPORTS = (
    "spec_verify_workspace_size", "spec_verify_sample", "spec_verify_greedy", "spec_verify_tree_greedy",
    "spec_transform_probs", "spec_get_status", "spec_error_string", "spec_expected_tokens",
    "spec_improvement_factor", "spec_break_even_acceptance", "spec_verify_sample_noalloc",
    "spec_sample_launch_mode", "spec_best_gamma", "spec_first_draft_check", "spec_verify_tree_sample",
)
SPEC_LAUNCH_SEPARATE = 0
SPEC_LAUNCH_FUSED = 1
SPEC_LAUNCH_FUSED_WAIT_TEST = 2
SPEC_LAUNCH_ROWS = 3
SPEC_LAUNCH_SPLIT = 4
SPEC_LAUNCH_AUTO = 5


class SpecSamplingParams(ctypes.Structure):
    _fields_ = [
        ("temperature", ctypes.c_float),
        ("temperature_per_seq", ctypes.c_void_p),
        ("top_k", ctypes.c_int),
        ("top_p", ctypes.c_float),
    ]


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {error_string(code)} ({code})")
        self.code = code


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the library in-tree (nvcc, sm_103a)."""
    from . import _build

    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"libspecverify.so not found at {LIB_PATH}; build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')"
                )
            L = ctypes.CDLL(LIB_PATH)
            P, I, SZ, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
            L.spec_verify_workspace_size.argtypes = [I, I, I, I]
            L.spec_verify_workspace_size.restype = SZ
            L.spec_verify_sample.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P, P, P, SZ, P]
            L.spec_verify_sample.restype = I
            L.spec_verify_sample_noalloc.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P, P, P, P]
            L.spec_verify_sample_noalloc.restype = I
            L.spec_verify_greedy.argtypes = [P, P, I, I, I, I, P, P, P, SZ, P]
            L.spec_verify_greedy.restype = I
            L.spec_verify_tree_greedy.argtypes = [P, P, P, I, I, I, I, I, P, P, P, P, SZ, P]
            L.spec_verify_tree_greedy.restype = I
            L.spec_verify_tree_sample.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_float, P, P, P, P, P, SZ, P]
            L.spec_verify_tree_sample.restype = I
            L.spec_transform_probs.argtypes = [P, I, I, I, P, P, P, SZ, P]
            L.spec_transform_probs.restype = I
            L.spec_get_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
            L.spec_get_status.restype = I
            L.spec_error_string.argtypes = [I]
            L.spec_error_string.restype = ctypes.c_char_p
            L.spec_expected_tokens.argtypes = [D, I]
            L.spec_expected_tokens.restype = D
            L.spec_improvement_factor.argtypes = [D, I, D]
            L.spec_improvement_factor.restype = D
            L.spec_break_even_acceptance.argtypes = [I]
            L.spec_break_even_acceptance.restype = D
            L.spec_sample_launch_mode.argtypes = [I]
            L.spec_sample_launch_mode.restype = I
            L.spec_best_gamma.argtypes = [D, D, I, ctypes.POINTER(D)]
            L.spec_best_gamma.restype = I
            L.spec_first_draft_check.argtypes = [P, P, I, I, I, P, P, P, SZ, P]
            L.spec_kv_compact.argtypes = [P, I, P, P, P, I, I, I, I, P, P, P, P, P, P]
            L.spec_kv_compact.restype = I
            L.spec_first_draft_check.restype = I
            _lib = L
    return _lib


def spec_best_gamma(alpha: float, c: float, gamma_max: int = 12):
    """The draft length in 1..gamma_max with the largest speedup: (gamma, speedup)."""
    best = ctypes.c_double()
    g = lib().spec_best_gamma(float(alpha), float(c), int(gamma_max), ctypes.byref(best))
    if g < 0:
        raise SpecVerifyError(g, "spec_best_gamma")
    return g, best.value


def spec_sample_launch_mode(mode: int) -> int:
    """Set how the sampling entry points launch (SPEC_LAUNCH_*); returns the previous mode."""
    rc = lib().spec_sample_launch_mode(int(mode))
    if rc < 0:
        raise SpecVerifyError(rc, "spec_sample_launch_mode")
    return rc


def error_string(code: int) -> str:
    return lib().spec_error_string(int(code)).decode()


spec_error_string = error_string


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t: Optional[torch.Tensor], name: str, dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(code: int, what: str) -> None:
    if code != SPEC_OK:
        raise SpecVerifyError(code, what)


def spec_verify_workspace_size(B: int, k: int, V: int, dtype: int = SPEC_BF16) -> int:
    return int(lib().spec_verify_workspace_size(B, k, V, dtype))


class Workspace:
    """Zeroed device workspace, grown on demand; one per stream of calls."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _workspace(ws, nbytes: int, device) -> torch.Tensor:
    if ws is None:
        key = (device.index if device.index is not None else torch.cuda.current_device())
        ws = _default_ws.setdefault(key, Workspace(torch.device("cuda", key)))
    if isinstance(ws, Workspace):
        return ws.get(nbytes)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError("workspace too small")
    return ws


def _params(temperature, top_k, top_p, temperature_per_seq):
    tps = _dev(temperature_per_seq, "temperature_per_seq", torch.float32) if temperature_per_seq is not None else None
    return SpecSamplingParams(float(temperature), tps, int(top_k), float(top_p))


def spec_verify_sample(target_logits: torch.Tensor, draft_logits: torch.Tensor, draft_tokens: torch.Tensor,
                       uniforms: torch.Tensor, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                       temperature_per_seq: Optional[torch.Tensor] = None, out_tokens=None, out_num_accepted=None,
                       out_p_draft=None, out_q_draft=None, workspace=None, stream=None, want_probs: bool = True):
    """Speculative-sampling verification.  Returns (tokens [B][k+1], n [B], p_x [B][k], q_x [B][k])."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if want_probs and out_p_draft is None:
        out_p_draft = torch.empty((B, k), dtype=torch.float32, device=dev)
    if want_probs and out_q_draft is None:
        out_q_draft = torch.empty((B, k), dtype=torch.float32, device=dev)
    dt = _dtype_code(target_logits)
    ws = _workspace(workspace, spec_verify_workspace_size(B, k, V, dt), dev)
    sp = _params(temperature, top_k, top_p, temperature_per_seq)
    rc = lib().spec_verify_sample(
        _dev(target_logits, "target_logits"), _dev(draft_logits, "draft_logits", target_logits.dtype),
        _dev(draft_tokens, "draft_tokens", torch.int32), _dev(uniforms, "uniforms", torch.float32),
        B, k, V, dt, ctypes.byref(sp), _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_num_accepted, "out_num_accepted", torch.int32), _dev(out_p_draft, "out_p_draft"),
        _dev(out_q_draft, "out_q_draft"), ws.data_ptr(), ws.numel(), _stream(stream),
    )
    _check(rc, "spec_verify_sample")
    return out_tokens, out_num_accepted, out_p_draft, out_q_draft


def spec_verify_sample_noalloc(target_logits: torch.Tensor, draft_logits: torch.Tensor, draft_tokens: torch.Tensor,
                               uniforms: torch.Tensor, out_tokens: torch.Tensor, out_num_accepted: torch.Tensor,
                               out_p_draft: Optional[torch.Tensor] = None, out_q_draft: Optional[torch.Tensor] = None,
                               out_status: Optional[torch.Tensor] = None, temperature: float = 1.0, top_k: int = 0,
                               top_p: float = 1.0, temperature_per_seq: Optional[torch.Tensor] = None, stream=None):
    """spec_verify_sample for callers that cannot allocate device memory.

    The library keeps a fixed scratch array on each device instead of taking
    a workspace; the caller passes every output (this wrapper creates no
    tensor).  out_status, if given, is a one-element int32/uint32-sized CUDA
    tensor that receives this call's status bits.  Calls that overlap on the
    GPU share the scratch and race.
    """
    B, k1, V = target_logits.shape
    k = k1 - 1
    dt = _dtype_code(target_logits)
    sp = _params(temperature, top_k, top_p, temperature_per_seq)
    rc = lib().spec_verify_sample_noalloc(
        _dev(target_logits, "target_logits"), _dev(draft_logits, "draft_logits", target_logits.dtype),
        _dev(draft_tokens, "draft_tokens", torch.int32), _dev(uniforms, "uniforms", torch.float32),
        B, k, V, dt, ctypes.byref(sp), _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_num_accepted, "out_num_accepted", torch.int32), _dev(out_p_draft, "out_p_draft", torch.float32),
        _dev(out_q_draft, "out_q_draft", torch.float32), _dev(out_status, "out_status"), _stream(stream),
    )
    _check(rc, "spec_verify_sample_noalloc")
    return out_tokens, out_num_accepted, out_p_draft, out_q_draft


def spec_verify_greedy(target_logits: torch.Tensor, draft_tokens: torch.Tensor, out_tokens=None,
                       out_num_accepted=None, workspace=None, stream=None):
    """Greedy chain verification.  Returns (tokens [B][k+1], n [B])."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    dt = _dtype_code(target_logits)
    ws = _workspace(workspace, spec_verify_workspace_size(B, k, V, dt), dev)
    rc = lib().spec_verify_greedy(
        _dev(target_logits, "target_logits"), _dev(draft_tokens, "draft_tokens", torch.int32), B, k, V, dt,
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_num_accepted, "out_num_accepted", torch.int32),
        ws.data_ptr(), ws.numel(), _stream(stream),
    )
    _check(rc, "spec_verify_greedy")
    return out_tokens, out_num_accepted


def spec_first_draft_check(prev_rows: torch.Tensor, draft0: torch.Tensor, out_accept=None, out_argmax=None,
                           workspace=None, stream=None):
    """Rejection fast path: (accept [B], argmax [B]) of the previous step's rows [B][V] against draft0 [B]."""
    B, V = prev_rows.shape
    dev = prev_rows.device
    if out_accept is None:
        out_accept = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_argmax is None:
        out_argmax = torch.empty((B,), dtype=torch.int32, device=dev)
    dt = _dtype_code(prev_rows)
    ws = _workspace(workspace, spec_verify_workspace_size(B, 1, V, dt), dev)
    rc = lib().spec_first_draft_check(
        _dev(prev_rows, "prev_rows"), _dev(draft0, "draft0", torch.int32), B, V, dt,
        _dev(out_accept, "out_accept", torch.int32), _dev(out_argmax, "out_argmax", torch.int32),
        ws.data_ptr(), ws.numel(), _stream(stream),
    )
    _check(rc, "spec_first_draft_check")
    return out_accept, out_argmax


def spec_verify_tree_greedy(node_logits: torch.Tensor, node_tokens: torch.Tensor, parents: torch.Tensor,
                            max_depth: int, out_tokens=None, out_path=None, out_num_accepted=None,
                            workspace=None, stream=None):
    """Greedy token-tree verification.  Returns (tokens, path [B][max_depth+1], n [B])."""
    B, N, V = node_logits.shape
    dev = node_logits.device
    D = int(max_depth) + 1
    if out_tokens is None:
        out_tokens = torch.empty((B, D), dtype=torch.int32, device=dev)
    if out_path is None:
        out_path = torch.empty((B, D), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    dt = _dtype_code(node_logits)
    ws = _workspace(workspace, spec_verify_workspace_size(B, N - 1, V, dt), dev)
    rc = lib().spec_verify_tree_greedy(
        _dev(node_logits, "node_logits"), _dev(node_tokens, "node_tokens", torch.int32),
        _dev(parents, "parents", torch.int32), B, N, V, int(max_depth), dt,
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_path, "out_path", torch.int32),
        _dev(out_num_accepted, "out_num_accepted", torch.int32), ws.data_ptr(), ws.numel(), _stream(stream),
    )
    _check(rc, "spec_verify_tree_greedy")
    return out_tokens, out_path, out_num_accepted


def spec_verify_tree_sample(node_logits: torch.Tensor, draft_logits: torch.Tensor, node_tokens: torch.Tensor,
                            parents: torch.Tensor, uniforms: torch.Tensor, max_depth: int,
                            temperature: float = 1.0, temperature_per_tree: Optional[torch.Tensor] = None,
                            out_tokens=None, out_path=None, out_num_accepted=None, workspace=None, stream=None):
    """Token-tree sampling verification.  node_logits / draft_logits [B][N][V],
    node_tokens / parents [B][N] int32, uniforms [B][N] float32 (u_0 the final
    draw, u_j the test of node j); temperature_per_tree [B] float32 or None.
    Returns (tokens, path [B][max_depth+1], n [B])."""
    B, N, V = node_logits.shape
    if tuple(draft_logits.shape) != (B, N, V) or draft_logits.dtype != node_logits.dtype:
        raise ValueError("draft_logits must match node_logits in shape and dtype")
    dev = node_logits.device
    D = int(max_depth) + 1
    if out_tokens is None:
        out_tokens = torch.empty((B, D), dtype=torch.int32, device=dev)
    if out_path is None:
        out_path = torch.empty((B, D), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    dt = _dtype_code(node_logits)
    ws = _workspace(workspace, spec_verify_workspace_size(B, N - 1, V, dt), dev)
    rc = lib().spec_verify_tree_sample(
        _dev(node_logits, "node_logits"), _dev(draft_logits, "draft_logits"),
        _dev(node_tokens, "node_tokens", torch.int32), _dev(parents, "parents", torch.int32),
        _dev(uniforms, "uniforms", torch.float32), B, N, V, int(max_depth), dt, float(temperature),
        _dev(temperature_per_tree, "temperature_per_tree", torch.float32),
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_path, "out_path", torch.int32),
        _dev(out_num_accepted, "out_num_accepted", torch.int32), ws.data_ptr(), ws.numel(), _stream(stream),
    )
    _check(rc, "spec_verify_tree_sample")
    return out_tokens, out_path, out_num_accepted


def spec_kv_compact(num_accepted: torch.Tensor, kv_base: torch.Tensor, path: Optional[torch.Tensor] = None,
                    block_table: Optional[torch.Tensor] = None, block_size: int = 0, max_keep: Optional[int] = None,
                    out_status: Optional[torch.Tensor] = None, out_src=None, out_dst=None, out_new_len=None,
                    out_num_moves=None, stream=None):
    """KV-cache keep list after verification: (src [B][max_keep], dst [B][max_keep],
    new_len [B], num_moves [B]) slots of the kept entries before and after the
    cut.  path [B][S] (tree out_path) or None for a chain; block_table [B][M]
    maps logical blocks of block_size entries to physical ones, or None."""
    B = num_accepted.shape[0]
    dev = num_accepted.device
    if max_keep is None:
        max_keep = (path.shape[1] + 1) if path is not None else None
        if max_keep is None:
            raise ValueError("max_keep is required for a chain (k + 1)")
    src = out_src if out_src is not None else torch.empty((B, max_keep), dtype=torch.int32, device=dev)
    dst = out_dst if out_dst is not None else torch.empty((B, max_keep), dtype=torch.int32, device=dev)
    new_len = out_new_len if out_new_len is not None else torch.empty((B,), dtype=torch.int32, device=dev)
    moves = out_num_moves if out_num_moves is not None else torch.empty((B,), dtype=torch.int32, device=dev)
    if src.shape != (B, max_keep) or dst.shape != (B, max_keep) or new_len.shape != (B,) or moves.shape != (B,):
        raise ValueError("spec_kv_compact: output shapes must be [B][max_keep] and [B]")
    rc = lib().spec_kv_compact(
        _dev(path, "path", torch.int32), path.shape[1] if path is not None else 0,
        _dev(num_accepted, "num_accepted", torch.int32), _dev(kv_base, "kv_base", torch.int32),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1] if block_table is not None else 0,
        block_size, B, max_keep, _dev(src, "out_src", torch.int32), _dev(dst, "out_dst", torch.int32),
        _dev(new_len, "out_new_len", torch.int32), _dev(moves, "out_num_moves", torch.int32), _dev(out_status, "out_status", torch.int32) if out_status is not None else None,
        _stream(stream),
    )
    _check(rc, "spec_kv_compact")
    return src, dst, new_len, moves


def spec_transform_probs(logits: torch.Tensor, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                         temperature_per_seq: Optional[torch.Tensor] = None, out_probs=None, workspace=None,
                         stream=None) -> torch.Tensor:
    """Filtered, normalised rows: logits [R][V] -> probabilities [R][V] float32."""
    R, V = logits.shape
    dev = logits.device
    if out_probs is None:
        out_probs = torch.empty((R, V), dtype=torch.float32, device=dev)
    dt = _dtype_code(logits)
    ws = _workspace(workspace, spec_verify_workspace_size(R, 0, V, dt), dev)
    sp = _params(temperature, top_k, top_p, temperature_per_seq)
    rc = lib().spec_transform_probs(_dev(logits, "logits"), R, V, dt, ctypes.byref(sp),
                                    _dev(out_probs, "out_probs", torch.float32), ws.data_ptr(), ws.numel(),
                                    _stream(stream))
    _check(rc, "spec_transform_probs")
    return out_probs


def spec_get_status(workspace=None, stream=None) -> int:
    """Reads and clears the device status bits of a workspace (synchronises)."""
    if workspace is None:
        workspace = _default_ws.get(torch.cuda.current_device())
        if workspace is None:
            return 0
    buf = workspace.get(0) if isinstance(workspace, Workspace) else workspace
    st = ctypes.c_uint32(0)
    rc = lib().spec_get_status(buf.data_ptr(), ctypes.byref(st), _stream(stream))
    if rc not in (SPEC_OK, SPEC_ERR_DEVICE_DATA, SPEC_ERR_TIMEOUT):
        raise SpecVerifyError(rc, "spec_get_status")
    return int(st.value)


def spec_expected_tokens(alpha: float, gamma: int) -> float:
    return float(lib().spec_expected_tokens(float(alpha), int(gamma)))


def spec_improvement_factor(alpha: float, gamma: int, c: float) -> float:
    return float(lib().spec_improvement_factor(float(alpha), int(gamma), float(c)))


def spec_break_even_acceptance(k: int) -> float:
    return float(lib().spec_break_even_acceptance(int(k)))
