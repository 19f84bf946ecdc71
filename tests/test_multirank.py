"""The N > 1 path of bench.py on CPU, as two gloo ranks on 127.0.0.1: the barrier and the max over
ranks that bound the timed region, the per-rank request shard (each rank its own seed), and the
reference arm, which rank 0 alone runs and prints.  The decode path itself has no collective:
requests are independent, so ranks exchange only the timing."""
import json
import os
import socket
import subprocess
import sys

import numpy as np

import workload as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DIST_SNIPPET = r"""
import importlib.util, json, os, sys
spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(sys.argv[1], "bench.py"))
b = importlib.util.module_from_spec(spec); spec.loader.exec_module(b)
d = b.Dist(int(os.environ["WORLD_SIZE"]))
d.barrier()
m = d.max(1.5 + d.rank)          # each rank reports its own elapsed time
d.barrier()
print(json.dumps({"rank": d.rank, "world": d.world, "max": m}), flush=True)
d.close()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(args, world=2, timeout=300):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                   LOCAL_WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable] + args, cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=timeout)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_barrier_and_max_over_two_gloo_ranks():
    outs = _launch(["-c", DIST_SNIPPET, ROOT])
    got = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(g["rank"] for g in got) == [0, 1]
    assert all(g["world"] == 2 and g["max"] == 2.5 for g in got)


def test_reference_arm_prints_on_rank_zero_only():
    outs = _launch(["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1"])
    lines = [o.strip() for o in outs]
    assert lines[1] == ""
    j = json.loads(lines[0].splitlines()[-1])
    assert j["impl"] == "reference" and j["value"] > 0 and j["cpu_baseline"]["kind"] == "oracle"
    cov = j["dense_softmax_coverage"]
    assert 0.0 < cov["min"] <= cov["value"] <= 1.0


def test_ranks_serve_different_requests():
    """bench.py gives rank r the seed seed + r: the ranks' histories differ (weak scaling)."""
    w = W.TINY
    k0, _ = W.kv_numpy(w)
    k1, _ = W.kv_numpy(w.with_(seed=w.seed + 1))
    assert k0.shape == k1.shape and not np.array_equal(k0, k1)
