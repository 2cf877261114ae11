"""GPU parity of sampling verification in the three-launch split path
(SPEC_LAUNCH_SPLIT: stream, row, draw) against the float64 oracle: the
configuration, sweep and edge cases of test_gpu_sample, run in that mode,
plus cuts below the stream's window of values, ties at the cut, masked
entries, status bits and the workspace left for the other launch modes.
Same bar: identical accept counts and tokens outside oracle boundary draws;
p(x), q(x) within 1e-5."""
import numpy as np
import pytest

import workloads as W
from parity_utils import compare_sample, lib, q_support_mask, run_sample_gpu, run_sample_oracle, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def split_mode():
    sv = lib()
    prev = sv.spec_sample_launch_mode(sv.SPEC_LAUNCH_SPLIT)
    yield
    sv.spec_sample_launch_mode(prev)


def _check(case, seqs=None):
    gpu = run_sample_gpu(case)
    orc = run_sample_oracle(case, seqs)
    return compare_sample(case, gpu, orc, seqs)


@pytest.mark.parametrize("per_seq", [False, True])
def test_split_config3_full_size(per_seq):
    _check(W.config3(per_seq_temperature=per_seq))


def test_split_config1_and_config2():
    _check(W.config1(B=8))
    _check(W.config2(mask_fn=q_support_mask(50, 1.0)))


@pytest.mark.parametrize("B,k,sigma", [(1, 1, 0.5), (4, 12, 2.0), (16, 4, 4.0), (64, 8, 0.5), (64, 12, 4.0),
                                       (128, 2, 2.0), (256, 8, 2.0)])
def test_split_config5_points(B, k, sigma):
    case = W.config5(B, k, sigma)
    _check(case, list(range(0, B, max(1, B // 32))))


EDGE = [
    (3, 1, 8, W.BF16, 0, 1.0, {}),
    (5, 3, 8, W.F32, 0, 1.0, {}),
    (6, 4, 16, W.BF16, 3, 1.0, {}),
    (8, 12, 1000, W.BF16, 20, 0.9, {}),
    (8, 31, 256, W.BF16, 0, 0.7, {"per_seq_temperature": True}),
    (4, 3, 70000, W.BF16, 0, 0.5, {"temperature": 0.6}),
    (6, 4, 2000, W.BF16, 7, 1.0, {"quantize": 0.5}),
    (6, 4, 2000, W.BF16, 0, 0.6, {"quantize": 0.5}),
    (4, 2, 5000, W.BF16, 1, 1.0, {}),
    (4, 2, 304, W.BF16, 300, 1.0, {}),
    (4, 2, 304, W.BF16, 0, 1e-4, {}),
    (3, 2, 100000, W.BF16, 0, 0.95, {"sigma": 0.05}),
    (2, 5, 262144, W.BF16, 0, 0.9, {}),
    (7, 2, 4104, W.F32, 0, 1.0, {"per_seq_temperature": True}),
]


@pytest.mark.parametrize("B,k,V,dtype,top_k,top_p,extra", EDGE,
                         ids=[f"B{e[0]}k{e[1]}V{e[2]}{e[3]}tk{e[4]}tp{e[5]}{''.join(e[6])}" for e in EDGE])
def test_split_edge_shapes_and_filters(B, k, V, dtype, top_k, top_p, extra):
    extra = dict(extra)
    T = extra.pop("temperature", 1.0)
    case = W.random_sample_case(B, k, V, dtype=dtype, seed=V + k, top_k=top_k, top_p=top_p, temperature=T,
                                mask_fn=q_support_mask(top_k, top_p) if V <= 5000 else None, **extra)
    _check(case)


# the cut far below the row maximum: below the stream's 512 values (a search
# in the row), for top-k alone, top-p alone and both
@pytest.mark.parametrize("top_k,top_p,spike", [(50, 1.0, 30.0), (0, 0.9, 12.0), (40, 0.98, 25.0),
                                               (40, 0.9999, 14.0), (3000, 1.0, 40.0), (0, 0.999, 12.0),
                                               (20000, 0.95, 20.0), (0, 0.99, 3.0)])
def test_split_cut_far_below_the_row_maximum(top_k, top_p, spike):
    _check(W.random_sample_case(4, 3, 50000, seed=13, sigma=1.0, noise=0.5, top_k=top_k, top_p=top_p, spike=spike))


def test_split_all_equal_logits_ties_everywhere():
    B, k, V = 4, 3, 5000
    case = W.random_sample_case(B, k, V, seed=7, top_k=0, top_p=1.0)
    case.target[:] = W.bf16_bits(np.full((B, k + 1, V), 1.5, np.float32))
    d = np.full((B, k, V), 1.5, np.float32)
    d[..., :5] = 3.0
    case.draft[:] = W.bf16_bits(d)
    case.tokens[:, 0] = np.arange(B) % 7
    for top_k, top_p in ((0, 1.0), (17, 1.0), (0, 0.3), (100, 0.5)):
        case.top_k, case.top_p = top_k, top_p
        _check(case)


def test_split_masked_minus_inf_entries():
    case = W.random_sample_case(6, 4, 3000, seed=11, top_p=0.9)
    rng = np.random.default_rng(0)
    ninf = W.bf16_bits(np.array([-np.inf], np.float32))[0]
    case.target[rng.random(case.target.shape) < 0.3] = ninf
    case.draft[rng.random(case.draft.shape) < 0.3] = ninf
    _check(case)


def test_split_topk1_matches_greedy():
    case = W.random_sample_case(32, 5, 20000, seed=3, top_k=1)
    tok, n, _, _ = run_sample_gpu(case)
    g_tok, g_n = lib().spec_verify_greedy(to_dev(case.target), to_dev(case.tokens))
    assert np.array_equal(tok, g_tok.cpu().numpy()) and np.array_equal(n, g_n.cpu().numpy())


def test_split_bad_tokens_and_rows_set_status():
    sv = lib()
    case = W.random_sample_case(4, 3, 1000, seed=2)
    case.tokens[0, 0] = -1
    case.tokens[1, 1] = 1000
    ws = sv.Workspace()
    sv.spec_get_status(ws)
    out = sv.spec_verify_sample(to_dev(case.target), to_dev(case.draft), to_dev(case.tokens),
                                to_dev(case.uniforms), workspace=ws)
    assert sv.spec_get_status(ws) & sv.SPEC_STATUS_BAD_TOKEN
    orc = run_sample_oracle(case)
    assert np.array_equal(out[1].cpu().numpy(), orc["n"])
    assert np.array_equal(out[0].cpu().numpy(), orc["tokens"])
    nan = W.bf16_bits(np.array([np.nan], np.float32))[0]
    case.target[2, 0, 5] = nan
    out = sv.spec_verify_sample(to_dev(case.target), to_dev(case.draft), to_dev(case.tokens),
                                to_dev(case.uniforms), workspace=ws)
    assert sv.spec_get_status(ws) & sv.SPEC_STATUS_BAD_ROW
    n = out[1].cpu().numpy()
    assert n[2] == 0 and out[0].cpu().numpy()[2, 0] == -1  # a non-finite row at n: no token drawn
    assert sv.spec_get_status(ws) == 0


def test_split_repeat_calls_and_other_modes_share_the_workspace():
    sv = lib()
    case = W.random_sample_case(16, 6, 32000, seed=9, top_p=0.9)
    ws = sv.Workspace()
    first = run_sample_gpu(case, workspace=ws)
    for mode in (sv.SPEC_LAUNCH_FUSED, sv.SPEC_LAUNCH_ROWS, sv.SPEC_LAUNCH_SPLIT, sv.SPEC_LAUNCH_SEPARATE,
                 sv.SPEC_LAUNCH_SPLIT):
        sv.spec_sample_launch_mode(mode)
        again = run_sample_gpu(case, workspace=ws)
        for a, b in zip(first, again):
            assert np.array_equal(a, b) if a.dtype.kind in "iu" else np.allclose(a, b, rtol=1e-5, atol=1e-7)
    sv.spec_sample_launch_mode(sv.SPEC_LAUNCH_SPLIT)
    assert sv.spec_get_status(ws) == 0


# Calls the split launches do not take run the fused launch instead, with the
# same results: rows that are not whole 16-byte vectors, rows that do not start
# on a 16-byte boundary, f32 rows with a filter, rows over 512 KiB.
@pytest.mark.parametrize("B,k,V,dtype,top_k,top_p", [(5, 3, 1001, W.BF16, 0, 0.95), (4, 2, 4100, W.F32, 10, 0.9),
                                                     (2, 2, 270000, W.BF16, 0, 0.95)])
def test_split_falls_back_for_shapes_it_does_not_take(B, k, V, dtype, top_k, top_p):
    _check(W.random_sample_case(B, k, V, dtype=dtype, seed=V, top_k=top_k, top_p=top_p))


def test_split_unaligned_rows_fall_back():
    sv = lib()
    case = W.random_sample_case(4, 3, 4096, seed=5, top_p=0.95)
    t = to_dev(np.concatenate([np.zeros(1, np.uint16), case.target.ravel()]))[1:].view(case.target.shape)
    d = to_dev(np.concatenate([np.zeros(1, np.uint16), case.draft.ravel()]))[1:].view(case.draft.shape)
    assert t.data_ptr() % 16 == 2
    out = sv.spec_verify_sample(t, d, to_dev(case.tokens), to_dev(case.uniforms), 1.0, 0, 0.95)
    compare_sample(case, [o.cpu().numpy() for o in out], run_sample_oracle(case))
