"""GPU parity of sampling verification in the one-CTA-per-row launch
(SPEC_LAUNCH_ROWS) against the float64 oracle: the configuration, sweep and
edge cases of test_gpu_sample, run in that mode.  Same bar: identical accept
counts and tokens outside oracle boundary draws; p(x), q(x) within 1e-5."""
import numpy as np
import pytest

import workloads as W
from parity_utils import compare_sample, lib, q_support_mask, run_sample_gpu, run_sample_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def rows_mode():
    sv = lib()
    prev = sv.spec_sample_launch_mode(sv.SPEC_LAUNCH_ROWS)
    yield
    sv.spec_sample_launch_mode(prev)


def _check(case, seqs=None):
    gpu = run_sample_gpu(case)
    orc = run_sample_oracle(case, seqs)
    nb, draws = compare_sample(case, gpu, orc, seqs)
    return nb, draws


@pytest.mark.parametrize("per_seq", [False, True])
def test_rows_config3_full_size(per_seq):
    _check(W.config3(per_seq_temperature=per_seq))


def test_rows_config1_and_config2():
    _check(W.config1(B=8))
    _check(W.config2(mask_fn=q_support_mask(50, 1.0)))


@pytest.mark.parametrize("B,k,sigma", [(1, 1, 0.5), (16, 12, 2.0), (64, 8, 4.0), (256, 8, 0.5)])
def test_rows_config5_points(B, k, sigma):
    case = W.config5(B, k, sigma)
    _check(case, list(range(0, B, max(1, B // 32))))


EDGE = [
    (3, 1, 1, W.BF16, 0, 1.0, {}),
    (5, 2, 7, W.BF16, 0, 1.0, {}),
    (5, 3, 8, W.F32, 0, 1.0, {}),
    (6, 4, 9, W.BF16, 3, 1.0, {}),
    (8, 12, 1000, W.BF16, 20, 0.9, {}),
    (8, 31, 257, W.BF16, 0, 0.7, {"per_seq_temperature": True}),
    (4, 3, 70001, W.BF16, 0, 0.5, {"temperature": 0.6}),
    (6, 4, 2003, W.BF16, 7, 1.0, {"quantize": 0.5}),
    (6, 4, 2003, W.BF16, 0, 0.6, {"quantize": 0.5}),
    (4, 2, 5000, W.BF16, 1, 1.0, {}),
    (4, 2, 300, W.BF16, 300, 1.0, {}),
    (4, 2, 300, W.BF16, 0, 1e-4, {}),
    (3, 2, 100000, W.BF16, 0, 0.95, {"sigma": 0.05}),
]


@pytest.mark.parametrize("B,k,V,dtype,top_k,top_p,extra", EDGE,
                         ids=[f"B{e[0]}k{e[1]}V{e[2]}{e[3]}tk{e[4]}tp{e[5]}{''.join(e[6])}" for e in EDGE])
def test_rows_edge_shapes_and_filters(B, k, V, dtype, top_k, top_p, extra):
    extra = dict(extra)
    T = extra.pop("temperature", 1.0)
    case = W.random_sample_case(B, k, V, dtype=dtype, seed=V + k, top_k=top_k, top_p=top_p, temperature=T,
                                mask_fn=q_support_mask(top_k, top_p) if V <= 5000 else None, **extra)
    _check(case)


@pytest.mark.parametrize("top_k,top_p,spike", [(50, 1.0, 30.0), (0, 0.9, 12.0), (40, 0.98, 25.0),
                                               (40, 0.9999, 14.0), (3000, 1.0, 40.0), (0, 0.999, 12.0)])
def test_rows_cut_far_below_the_row_maximum(top_k, top_p, spike):
    _check(W.random_sample_case(4, 3, 50000, seed=13, sigma=1.0, noise=0.5, top_k=top_k, top_p=top_p, spike=spike))


def test_rows_repeat_calls_are_deterministic():
    case = W.random_sample_case(16, 6, 32000, seed=9, top_p=0.9)
    first = run_sample_gpu(case)
    for _ in range(3):
        for a, b in zip(first, run_sample_gpu(case)):
            assert np.array_equal(a, b)
