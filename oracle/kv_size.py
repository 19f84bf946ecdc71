"""KV-cache size formulas (oracle; test-only).

Source: "当上下文冲破百万：KV-Cache压缩技术的工程原理与2026年工业实践", section 1.1
(precise model of KV memory): bytes = 2 * L * N_layer * N_kv_head * D_head * P, the factor 2
counting K and V; and section 2 (MHA 2LhD, MQA 2LD, GQA 2LgD, MLA 2Ld_c per layer).

Pinned by tests/test_oracle_kv_size.py against the figure the tuntang.top survey gives
for Llama3.1-8B at 32K ("about 4GB", introduction) and the section 1.1 table's scaling.
"""


def kv_cache_bytes(seq_len: int, n_layer: int, n_kv_head: int, d_head: int, bytes_per_elem: float) -> float:
    return 2 * seq_len * n_layer * n_kv_head * d_head * bytes_per_elem


def kv_cache_bytes_variant(kind: str, seq_len: int, n_layer: int, n_q_head: int, d_head: int,
                           bytes_per_elem: float, n_groups: int = 1, d_latent: int = 0) -> float:
    """Per-architecture cache size: MHA keeps h heads, MQA one, GQA g groups, MLA a d_c latent."""
    per_layer_elems = {
        "mha": 2 * seq_len * n_q_head * d_head,
        "mqa": 2 * seq_len * d_head,
        "gqa": 2 * seq_len * n_groups * d_head,
        "mla": 2 * seq_len * d_latent,
    }[kind]
    return per_layer_elems * n_layer * bytes_per_elem
