"""Host logic of bench.py on the CPU: the DRAM-traffic record used only while
its kernel's sources are unchanged, the clock record taken during the timed
region (median SM clock, throttle reasons), and the algorithmic bytes of a
tree-sampling call (both rows of every node with a child to test, plus the
target row of a stop node without one)."""
import json
import os
import shutil
import types

import numpy as np

import bench


def _fake_root(tmp_path):
    csrc = tmp_path / "draft_token_verification_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "draft_token_verification_gb300", "csrc")
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            shutil.copy(os.path.join(src, f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_traffic_record_is_used_only_on_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    rec = {
        "tree_sample": {"kernel_source_hash": bench.kernel_source_hash("tree_sample"), "dram_bytes_per_launch": 123},
        "argmax_chain": {"kernel_source_hash": bench.kernel_source_hash("argmax"), "dram_bytes_per_launch": 456},
        "sample": {"kernel_source_hash": "0" * 16, "dram_bytes_per_launch": 789},
    }
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("tree_sample") == 123.0
    assert bench.recorded_traffic("argmax_chain") == 456.0
    assert bench.recorded_traffic("sample") is None  # taken on other sources
    assert bench.recorded_traffic("argmax_tree") is None  # no record
    # one changed byte in a file the kernel is compiled from voids its record
    f = root / "draft_token_verification_gb300" / "csrc" / "tree_sample_kernel.cu"
    f.write_bytes(f.read_bytes() + b"\n")
    assert bench.recorded_traffic("tree_sample") is None
    assert bench.recorded_traffic("argmax_chain") == 456.0
    # a header shared by every kernel voids them all
    h = root / "draft_token_verification_gb300" / "csrc" / "internal.h"
    h.write_bytes(h.read_bytes() + b"\n")
    assert bench.recorded_traffic("argmax_chain") is None


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_median_and_reasons():
    s = bench.ClockSampler(0)
    s.proc = _DoneProc()
    s.lines = [
        "2070, 2070, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "[N/A], 2070, 0x0, Not Active, Not Active, Not Active, Not Active",  # unreadable: skipped
        "truncated, line",
    ]
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    s.lines = ["1500, 2070, 0x08, Not Active, Active, Active, Not Active"] * 3
    c = s.stop()
    assert c["sm_mhz"] == 1500.0 and c["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_record_without_nvidia_smi():
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]


def _tree(parents, tokens, V, max_depth):
    return types.SimpleNamespace(B=1, N=len(parents), V=V, max_depth=max_depth,
                                 parents=np.array([parents], np.int32), node_tokens=np.array([tokens], np.int32))


def test_tree_sampling_algorithmic_bytes():
    # root 0 with children 1, 2; node 1 with children 3, 4
    case = _tree([-1, 0, 0, 1, 1], [0, 3, 4, 5, 6], V=10, max_depth=2)
    row = 10 * 2  # bf16
    # stop at leaf 3 (path 1, 3): nodes 0 and 1 test children, plus the leaf's target row
    assert bench.tree_sample_bytes(case, np.array([2]), np.array([[1, 3, -1]])) == (2 * 2 + 1) * row
    # stop at the root: its rows are already counted
    assert bench.tree_sample_bytes(case, np.array([0]), np.array([[-1, -1, -1]])) == 2 * 2 * row
    # children at max_depth are not tested: node 1 tests nothing, so its target row is read at the stop
    case1 = _tree([-1, 0, 0, 1, 1], [0, 3, 4, 5, 6], V=10, max_depth=1)
    assert bench.tree_sample_bytes(case1, np.array([1]), np.array([[1, -1]])) == (2 * 1 + 1) * row
    # a child whose token is out of range is not tested
    case2 = _tree([-1, 0, 0, 1, 1], [0, 3, 4, 10, -1], V=10, max_depth=2)
    assert bench.tree_sample_bytes(case2, np.array([1]), np.array([[1, -1, -1]])) == (2 * 1 + 1) * row


def test_job_rate_counts_every_rank():
    assert bench.job_rate(576, 4, 10, 2.0) == 576 * 4 * 10 / 2e-3
