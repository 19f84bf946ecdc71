"""bench.py's algorithmic byte counts (the numerators of every roofline figure), pinned against
values worked out by hand from the shapes: index scan N_b * d_k * 2 per unit, attention reads of the
selected rows |S| * bs * (d_k + d_v, or d_k alone when V shares the K row) * 2, queries and drafts,
fp32 outputs, plus the fetched bytes written to the slots."""
import importlib.util
import os

import workload as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_llama8b_lookahead_bytes():
    b = _bench()
    w = W.LLAMA8B_32K
    lens = [w.ctx0] * w.n_req
    hbm, link, per_layer = b.algorithmic_bytes(w, lens, 589_656_637)
    idx = 8 * 8 * 2048 * 128 * 2                  # units x blocks x d_k x bf16
    attn = 8 * 8 * (128 * 16) * (128 + 128) * 2   # units x selected tokens x (K + V) x bf16
    q = 8 * 32 * 128 * 2                          # current queries
    drafts = 8 * 32 * 128 * 2 * 4
    out = 8 * 32 * 128 * 4
    assert per_layer["index"] == idx == 33_554_432
    assert per_layer["attn"] == attn + q + out == 67_305_472
    assert link == 589_656_637
    assert hbm == 32 * (idx + attn + q + drafts + out) + link


def test_mla_bytes_share_the_latent_row():
    b = _bench()
    w = W.MLA_128K
    lens = [w.ctx0] * w.n_req
    hbm, _, per_layer = b.algorithmic_bytes(w, lens, 0)
    assert per_layer["index"] == 16 * 131072 * 576 * 2 == 2_415_919_104
    attn = 16 * 2048 * 576 * 2                    # V is the first 512 dims of the same row
    assert per_layer["attn"] == attn + 16 * 128 * 576 * 2 + 16 * 128 * 512 * 4
    assert hbm == 16 * (per_layer["index"] + attn + 16 * 128 * 576 * 2 + 16 * 128 * 512 * 4)


def test_short_contexts_read_only_present_rows():
    b = _bench()
    w = W.TINY.with_(n_req=3)
    lens = [4096, 1000, 17]
    _, _, per_layer = b.algorithmic_bytes(w, lens, 0)
    # budget 16 blocks of 16 tokens = 256 rows, capped by the context (17 tokens -> 17 rows)
    rows = (256 + 256 + 17) * w.n_kv_head
    assert per_layer["attn"] == rows * 256 * 2 + 3 * 8 * 128 * 2 + 3 * 8 * 128 * 4
    assert per_layer["index"] == (256 + 63 + 2) * 2 * 128 * 2


def test_host_memory_guard(monkeypatch):
    b = _bench()
    b.check_host_memory(1 << 20)                                  # 1 MiB always fits
    monkeypatch.setenv("LOCAL_WORLD_SIZE", "4")
    import pytest
    with pytest.raises(RuntimeError, match="host memory"):
        b.check_host_memory(1 << 50)


def test_prefetch_report():
    import numpy as np
    b = _bench()
    assert b.prefetch_report(W.LLAMA8B_32K, np.zeros(7), 10) is None          # no layer prefetch
    w = W.MLA_128K
    dstat = np.array([0, 0, 0, 5000, 2500, 0, 0], dtype=np.int64)            # over 10 steps
    r = b.prefetch_report(w, dstat, 10)
    assert r["blocks_per_step"] == 500 and r["used_per_step"] == 250 and r["used_fraction"] == 0.5
    assert r["hidden_miss_bytes_per_step"] == 250 * 576 * 2                  # token blocks of the latent row


def test_fp8_rows_and_bound_index_widths():
    """E4M3 rows move one byte per element; [max | min] summaries make the index scan twice as wide."""
    b = _bench()
    w = W.LLAMA8B_32K
    lens = [w.ctx0] * w.n_req
    _, _, base = b.algorithmic_bytes(w, lens, 0)
    _, _, f8 = b.algorithmic_bytes(w.with_(kv_dtype="fp8"), lens, 0)
    _, _, bd = b.algorithmic_bytes(w.with_(score_mode="bound"), lens, 0)
    rows = 8 * 8 * 128 * 16                        # units x selected tokens
    assert base["attn"] - f8["attn"] == rows * 256  # 512 B of bf16 K + V per token vs 256 B of E4M3
    assert bd["index"] == 2 * base["index"] and f8["index"] == base["index"]
