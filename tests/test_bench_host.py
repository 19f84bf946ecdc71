"""bench.py's host-side helpers that feed the reported figures: the committed ncu traffic lookup
(a figure is used only for the kernel source it was taken from), the step-to-step selection
overlap, the clock summary that decides whether a run is kept, the fit of the host link's burst
cost, and that the profile summaries' commands run committed scripts.  Every expected value below
is worked out by hand."""
import hashlib
import importlib.util
import os
import re

import numpy as np
import pytest

import workload as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _fake_tree(tmp_path, sources, blocks):
    csrc = tmp_path / "sparse_kv_cache_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in sources.items():
        (csrc / name).write_text(text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text("# a summary\n\n" + "\n".join(f"```traffic\n{b}```\n" for b in blocks))
    return tmp_path


def test_profile_traffic_matches_only_the_source_it_was_taken_from(tmp_path):
    b = _bench()
    srcs = {"k_cache.cu": "fetch v1\n"}
    sha_v1 = hashlib.sha256(b"fetch v1\n").hexdigest()[:16]
    root = _fake_tree(tmp_path, srcs, [
        f"kernel: fetch\nworkload: wl_a\nsource_sha: {sha_v1}\ndram_bytes_per_launch: 1234\nnote: n\n",
        "kernel: fetch\nworkload: wl_b\nsource_sha: 0000000000000000\ndram_bytes_per_launch: 99\n",
    ])
    b.ROOT = str(root)
    b.KERNEL_SOURCES = {"fetch": ["k_cache.cu"]}
    got = b.profile_traffic("fetch", "wl_a")
    assert got == {"bytes": 1234, "profile": "profiles/k.md", "note": "n"}
    assert b.profile_traffic("fetch", "wl_b") is None          # taken from another source
    assert b.profile_traffic("fetch", "wl_c") is None          # no block for this workload
    (root / "sparse_kv_cache_decode_gb300" / "csrc" / "k_cache.cu").write_text("fetch v2\n")
    assert b.profile_traffic("fetch", "wl_a") is None          # the kernel changed since


def test_committed_traffic_blocks_name_known_kernels_and_workloads():
    b = _bench()
    pdir = os.path.join(ROOT, "profiles")
    n = 0
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        text = open(os.path.join(pdir, f)).read()
        for block in re.findall(r"```traffic\n(.*?)```", text, flags=re.S):
            kv = {k.strip(): v.strip() for k, v in (ln.split(":", 1) for ln in block.strip().splitlines() if ":" in ln)}
            assert kv["kernel"] in b.KERNEL_SOURCES, (f, kv["kernel"])
            assert W.get(kv["workload"]).name == kv["workload"], (f, kv["workload"])
            assert re.fullmatch(r"[0-9a-f]{16}", kv["source_sha"]), (f, kv["source_sha"])
            assert int(kv["dram_bytes_per_launch"]) > 0
            n += 1
    assert n >= 1


def test_selection_overlap_counts_only_the_valid_entries():
    b = _bench()
    prev = np.array([[[1, 2, 3, 4, 9], [7, 8, 0, 0, 0]]], dtype=np.int32)   # [B=1][H=2][K=5]
    prev_n = np.array([[4, 2]], dtype=np.int32)
    cur = np.array([[[3, 4, 5, 6, 1], [8, 0, 0, 0, 0]]], dtype=np.int32)
    cur_n = np.array([[4, 1]], dtype=np.int32)
    # unit 0: {3,4,5,6} & {1,2,3,4} = {3,4} -> 2/4 (the 9 and 1 past the counts do not count);
    # unit 1: {8} & {7,8} -> 1/1
    assert b.selection_overlap(prev, prev_n, cur, cur_n) == [0.5, 1.0]
    cur_n0 = np.array([[4, 0]], dtype=np.int32)                               # empty selections skipped
    assert b.selection_overlap(prev, prev_n, cur, cur_n0) == [0.5]


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


class _Thread:
    def join(self, timeout=None):
        pass


def test_clock_summary_median_max_and_reasons():
    b = _bench()
    c = b.ClockSampler(0)
    c.proc, c.t = _Proc(), _Thread()
    c.lines = [
        "0, 2070, 2070, 950.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    got = c.stop()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c2 = b.ClockSampler(0)
    c2.proc, c2.t = _Proc(), _Thread()
    c2.lines = ["0, 1500, 2070, 700.0, 0x8, Active, Not Active, Active, Not Active"]
    assert c2.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_nvidia_smi():
    b = _bench()
    c = b.ClockSampler(0)
    assert c.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}


def test_burst_fit_recovers_fixed_cost_and_rate():
    b = _bench()
    # exact points of t = 14 us + bytes / 210.5 GB/s (210.5e3 bytes per us)
    pts = [(n, 14.0 + n / 210.5e3) for n in (2.28e6, 4.01e6, 16.4e6, 536.9e6)]
    fixed, rate = b.burst_fit(pts)
    assert fixed == pytest.approx(14.0, abs=1e-6)
    assert rate == pytest.approx(210.5, rel=1e-9)


def test_profile_commands_run_committed_files_only():
    """Each ncu summary under profiles/ gives the command that made it; the scripts it runs must
    be files of this repository (not scratch copies)."""
    pdir = os.path.join(ROOT, "profiles")
    seen = 0
    for f in sorted(os.listdir(pdir)):
        text = open(os.path.join(pdir, f)).read()
        assert "_work/" not in text, f
        for script in re.findall(r"python3?\s+([\w./-]+\.py)", text):
            assert os.path.isfile(os.path.join(ROOT, script)), (f, script)
            seen += 1
    assert seen >= 5
