"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/spec_verify.h declares, rejects bad arguments
before launching anything, and its calculator helpers match the pages' closed
forms."""
import ctypes
import json
import os
import re
import subprocess

import pytest

import draft_token_verification_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    sv.build()
    return sv.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(spec_\w+)\s*\(", text, flags=re.M)))


def test_header_declarations_are_all_exported(L):
    names = _declared_functions()
    assert len(names) >= 10, names
    out = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)
    assert set(sv.EXPORTS) <= set(names)


def test_library_does_not_link_torch():
    out = subprocess.run(["ldd", sv.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_error_strings(L):
    for code in range(0, -8, -1):
        assert sv.error_string(code) and sv.error_string(code) != "unknown error code"
    assert sv.error_string(-99) == "unknown error code"


def test_workspace_size_limits(L):
    assert sv.spec_verify_workspace_size(64, 8, 128256, sv.SPEC_BF16) > 0
    assert sv.spec_verify_workspace_size(0, 8, 128256, sv.SPEC_BF16) == 0
    assert sv.spec_verify_workspace_size(1, 8, 0, sv.SPEC_BF16) == 0
    assert sv.spec_verify_workspace_size(1, 8, 100, 7) == 0
    a = sv.spec_verify_workspace_size(16, 5, 32000, sv.SPEC_BF16)
    b = sv.spec_verify_workspace_size(32, 5, 32000, sv.SPEC_BF16)
    assert b > a and a % 256 == 0


FAKE = ctypes.c_void_p(4096)  # never dereferenced: every call below fails validation first


def _sample(L, **over):
    sp = sv.SpecSamplingParams(1.0, None, 0, 1.0)
    args = dict(t=FAKE, d=FAKE, x=FAKE, u=FAKE, B=2, k=3, V=100, dt=sv.SPEC_BF16, sp=ctypes.byref(sp), ot=FAKE,
                on=FAKE, op=None, oq=None, ws=ctypes.c_void_p(4096), wsb=1 << 20, st=None)
    if "sp" in over and isinstance(over["sp"], sv.SpecSamplingParams):
        over["sp"] = ctypes.byref(over["sp"])
    args.update(over)
    return L.spec_verify_sample(*args.values())


def test_sample_rejects_bad_arguments(L):
    assert _sample(L, t=None) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, B=0) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, k=0) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, k=32) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, V=0) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, dt=3) == sv.SPEC_ERR_DTYPE
    assert _sample(L, sp=None) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, sp=sv.SpecSamplingParams(0.0, None, 0, 1.0)) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, sp=sv.SpecSamplingParams(float("nan"), None, 0, 1.0)) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, sp=sv.SpecSamplingParams(1.0, None, -1, 1.0)) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, sp=sv.SpecSamplingParams(1.0, None, 0, 0.0)) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, sp=sv.SpecSamplingParams(1.0, None, 0, 1.5)) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, ws=None) == sv.SPEC_ERR_INVALID_ARG
    assert _sample(L, ws=ctypes.c_void_p(4096 + 16)) == sv.SPEC_ERR_WORKSPACE
    assert _sample(L, wsb=16) == sv.SPEC_ERR_WORKSPACE
    assert _sample(L, t=ctypes.c_void_p(4097)) == sv.SPEC_ERR_INVALID_ARG  # bf16 needs 2-byte alignment


def test_greedy_and_tree_reject_bad_arguments(L):
    g = L.spec_verify_greedy
    assert g(None, FAKE, 2, 3, 100, 1, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 2, 32, 100, 1, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 2, 3, 100, 9, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_DTYPE
    assert g(FAKE, FAKE, 2, 3, 100, 1, FAKE, FAKE, FAKE, 8, None) == sv.SPEC_ERR_WORKSPACE
    t = L.spec_verify_tree_greedy
    assert t(FAKE, FAKE, FAKE, 2, 1025, 100, 6, 1, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, FAKE, FAKE, 2, 60, 100, 0, 1, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, FAKE, None, 2, 60, 100, 6, 1, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    p = L.spec_transform_probs
    sp = sv.SpecSamplingParams(1.0, None, 0, 1.0)
    assert p(FAKE, 0, 100, 1, ctypes.byref(sp), FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert p(FAKE, 3, 100, 1, ctypes.byref(sp), None, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    st = ctypes.c_uint32()
    assert L.spec_get_status(None, ctypes.byref(st), None) == sv.SPEC_ERR_INVALID_ARG


def test_tree_sample_rejects_bad_arguments(L):
    ts = L.spec_verify_tree_sample

    def call(nl=FAKE, dl=FAKE, uni=FAKE, B=2, N=60, V=100, depth=6, dt=1, T=1.0, tpt=None, wsb=1 << 30):
        return ts(nl, dl, FAKE, FAKE, uni, B, N, V, depth, dt, T, tpt, FAKE, FAKE, FAKE, FAKE, wsb, None)

    assert call(dt=9) == sv.SPEC_ERR_DTYPE
    assert call(dl=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(N=1025) == sv.SPEC_ERR_INVALID_ARG
    assert call(depth=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(T=0.0) == sv.SPEC_ERR_INVALID_ARG
    assert call(T=float("nan")) == sv.SPEC_ERR_INVALID_ARG
    assert call(uni=ctypes.c_void_p(4098)) == sv.SPEC_ERR_INVALID_ARG  # float needs 4-byte alignment
    assert call(wsb=8) == sv.SPEC_ERR_WORKSPACE
    # per-tree temperatures replace the scalar one (checked on the device, per tree)
    assert call(T=0.0, tpt=FAKE, wsb=8) == sv.SPEC_ERR_WORKSPACE
    assert call(tpt=ctypes.c_void_p(4098)) == sv.SPEC_ERR_INVALID_ARG
    # a CTA's share of both rows must fit its shared memory: V = 300000 f32 does not
    assert call(V=300000, dt=0) == sv.SPEC_ERR_UNSUPPORTED


def test_kv_compact_rejects_bad_arguments(L):
    kv = L.spec_kv_compact

    def call(path=FAKE, stride=7, n=FAKE, base=FAKE, table=None, mb=0, bs=0, B=4, keep=8, moves=None, st=None):
        return kv(path, stride, n, base, table, mb, bs, B, keep, FAKE, FAKE, FAKE, moves, st, None)

    assert call(n=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(base=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(B=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(keep=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(stride=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(table=FAKE, mb=4, bs=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(table=FAKE, mb=0, bs=16) == sv.SPEC_ERR_INVALID_ARG
    assert call(st=ctypes.c_void_p(4098)) == sv.SPEC_ERR_INVALID_ARG
    assert call(moves=ctypes.c_void_p(4098)) == sv.SPEC_ERR_INVALID_ARG


def test_calculator_helpers_match_golden(L):
    with open(os.path.join(ROOT, "tests", "golden", "closed_forms.json")) as f:
        g = json.load(f)
    for c in g["expected_tokens"]["cases"]:
        assert sv.spec_expected_tokens(c["alpha"], c["gamma"]) == pytest.approx(c["value"], rel=1e-12)
    for c in g["improvement_factor"]["cases"]:
        assert sv.spec_improvement_factor(c["alpha"], c["gamma"], c["c"]) == pytest.approx(c["value"], rel=1e-12)
    for c in g["break_even"]["cases"]:
        assert sv.spec_break_even_acceptance(c["k"]) == pytest.approx(c["value"], rel=1e-15)


def test_binding_requires_cuda_tensors():
    import torch

    x = torch.zeros(2, 3, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sv.spec_verify_greedy(x, torch.zeros(2, 2, dtype=torch.int32), workspace=torch.zeros(1 << 16, dtype=torch.uint8))


def test_best_gamma_matches_oracle(L):
    import oracle
    for alpha in (0.0, 0.3, 0.6, 0.8, 0.9, 0.97, 1.0):
        for c in (0.0, 0.01, 0.05, 0.1, 0.3, 1.0, 1.5):
            for gmax in (1, 5, 12):
                g, f = sv.spec_best_gamma(alpha, c, gmax)
                go, fo = oracle.best_gamma(alpha, c, gmax)
                assert g == go and f == pytest.approx(fo, rel=1e-15), (alpha, c, gmax)
    best = ctypes.c_double()
    for bad in ((-0.1, 0.1, 12), (1.1, 0.1, 12), (0.5, -1.0, 12), (0.5, 0.1, 0), (0.5, 0.1, 65)):
        assert L.spec_best_gamma(bad[0], bad[1], bad[2], ctypes.byref(best)) == sv.SPEC_ERR_INVALID_ARG
