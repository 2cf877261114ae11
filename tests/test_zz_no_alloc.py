"""spec_verify_sample_noalloc: sampling verification without a workspace.

Some callers cannot allocate device memory at the point where they verify
drafts: a server whose memory manager has already handed nearly all of HBM
to its KV-cache pool, a library embedded in a runtime that forbids
allocations outside its own allocator, or a decode loop that cannot pay for
the device-wide synchronisation of cudaFree.  For them the library keeps a
fixed scratch array in its own device memory.  These tests call that entry
point through the C ABI and check that it gives what spec_verify_sample
gives on the same inputs, on consecutive calls that reuse the array with
different shapes.

This file is named so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from parity_utils import ABS_TOL_PROB, lib, to_dev


def _noalloc(sv, case: W.SampleCase):
    B, k = case.B, case.k
    dev = torch.device("cuda")
    out_tokens = torch.full((B, k + 1), -7, dtype=torch.int32, device=dev)
    out_n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out_p = torch.full((B, k), -1.0, dtype=torch.float32, device=dev)
    out_q = torch.full((B, k), -1.0, dtype=torch.float32, device=dev)
    out_status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    tps = to_dev(case.temperature_per_seq) if case.temperature_per_seq is not None else None
    sv.spec_verify_sample_noalloc(to_dev(case.target), to_dev(case.draft), to_dev(case.tokens),
                                  to_dev(case.uniforms), out_tokens, out_n, out_p, out_q, out_status,
                                  case.temperature, case.top_k, case.top_p, tps)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (out_tokens, out_n, out_p, out_q)], int(out_status.item())


def _with_workspace(sv, case: W.SampleCase):
    ws = sv.Workspace()
    tps = to_dev(case.temperature_per_seq) if case.temperature_per_seq is not None else None
    out = sv.spec_verify_sample(to_dev(case.target), to_dev(case.draft), to_dev(case.tokens),
                                to_dev(case.uniforms), case.temperature, case.top_k, case.top_p, tps,
                                workspace=ws)
    torch.cuda.synchronize()
    status = ctypes.c_uint32(0)
    sv.lib().spec_get_status(ws.get(0).data_ptr(), ctypes.byref(status), sv._stream(None))
    return [o.cpu().numpy() for o in out], int(status.value)


def _assert_same(got, want, what):
    np.testing.assert_array_equal(got[0], want[0], err_msg=f"{what}: tokens")
    np.testing.assert_array_equal(got[1], want[1], err_msg=f"{what}: n")
    np.testing.assert_allclose(got[2], want[2], rtol=0, atol=ABS_TOL_PROB, err_msg=f"{what}: p(x)")
    np.testing.assert_allclose(got[3], want[3], rtol=0, atol=ABS_TOL_PROB, err_msg=f"{what}: q(x)")


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    sv = lib()
    # Two different shapes back to back: the second call reuses the scratch
    # that the first one left behind, with a different layout inside it.
    first = W.config2(seed=41)                                                  # top-k 50, V = 32000
    second = W.config3(seed=42, per_seq_temperature=True, B=8)                  # top-p 0.9, V = 128256
    for i, case in enumerate((first, second)):
        got, got_status = _noalloc(sv, case)
        want, want_status = _with_workspace(sv, case)
        _assert_same(got, want, f"call {i + 1} ({case.name})")
        assert got_status == want_status == 0


@pytest.mark.gpu
def test_noalloc_status_is_per_call():
    sv = lib()
    bad = W.random_sample_case(4, 3, 5000, seed=43, top_p=0.95)
    bad.tokens[1, 0] = 5000                  # outside [0, V)
    got, got_status = _noalloc(sv, bad)
    want, want_status = _with_workspace(sv, bad)
    _assert_same(got, want, "bad token")
    assert got_status == want_status == sv.SPEC_STATUS_BAD_TOKEN
    clean = W.random_sample_case(4, 3, 5000, seed=44, top_p=0.95)
    got, got_status = _noalloc(sv, clean)
    want, _ = _with_workspace(sv, clean)
    _assert_same(got, want, "clean call after a bad one")
    assert got_status == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import draft_token_verification_gb300 as sv

    L = sv.lib()
    sp = sv.SpecSamplingParams(1.0, None, 0, 1.0)
    for B, k in ((sv.SPEC_NOALLOC_MAX_B + 1, 1), (1024, 8), (sv.SPEC_NOALLOC_MAX_B, 4)):
        rc = L.spec_verify_sample_noalloc(None, None, None, None, B, k, 1000, sv.SPEC_BF16, ctypes.byref(sp),
                                          None, None, None, None, None, None)
        assert rc == sv.SPEC_ERR_SCRATCH_LIMIT, (B, k, rc)
    assert "scratch" in sv.error_string(sv.SPEC_ERR_SCRATCH_LIMIT)
