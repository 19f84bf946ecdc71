"""Pins for oracle.kv_size: the worked figures the pages print.

The tuntang.top survey's introduction puts the Llama3.1-8B KV cache at 32K context at about
4 GB; the KV-cache overview's section 1.1 gives the formula and a table whose columns scale
by 8x per context step and halve per precision step; section 2 gives the MHA/MQA/GQA/MLA
ratios h, h/g and d/d_c (d = 4096, d_c = 512 -> 8x)."""
import pytest

from oracle import kv_cache_bytes, kv_cache_bytes_variant


def test_llama8b_32k_about_4gb():
    b = kv_cache_bytes(32768, 32, 8, 128, 2)
    assert b == 4_294_967_296          # 4.0 GiB = 4.29 GB, "about 4GB"
    assert 4.0e9 < b < 4.5e9


def test_long_context_host_history_64gib():
    # 128K context, batch 4 (the host-resident workload): 64 GiB
    assert 4 * kv_cache_bytes(131072, 32, 8, 128, 2) == 64 * 2**30


def test_table_scaling():
    base = kv_cache_bytes(16 * 1024, 65, 64, 128, 2)
    assert kv_cache_bytes(128 * 1024, 65, 64, 128, 2) == 8 * base            # 16K -> 128K
    assert kv_cache_bytes(16 * 1024, 65, 64, 128, 1) == base / 2             # FP16 -> FP8
    assert kv_cache_bytes(16 * 1024, 65, 64, 128, 0.5) == base / 4           # FP16 -> INT4
    assert 32 * 6.8 == pytest.approx(217.6)                                  # batch 32 column: 217 GB
    assert kv_cache_bytes(1024 * 1024, 65, 64, 128, 2) == 64 * base          # 16K -> 1M: 6.8 -> 435.2


def test_architecture_ratios():
    L, nl, h, d = 4096, 32, 64, 128
    mha = kv_cache_bytes_variant("mha", L, nl, h, d, 2)
    assert mha / kv_cache_bytes_variant("mqa", L, nl, h, d, 2) == h
    assert mha / kv_cache_bytes_variant("gqa", L, nl, h, d, 2, n_groups=8) == h / 8
    # MLA: d = 4096 compressed to d_c = 512 is an 8x reduction of the 2Ld term
    assert kv_cache_bytes_variant("mha", L, nl, 1, 4096, 2) / kv_cache_bytes_variant("mla", L, nl, 1, 4096, 2, d_latent=512) == 8
