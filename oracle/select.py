"""Block selection (oracle; test-only).

With nb = ceil(L / bs) blocks and a budget of K_b blocks:
  * nb <= K_b: every block is selected;
  * otherwise the forced set F = [0, n_sink) U [nb - n_recent, nb) (sink and recent
    blocks) is always kept, and the remaining K_b - |F| slots go to the other blocks with
    the highest scores, ties going to the lower block index; NaN ranks below -inf, and
    -0.0 equals +0.0.
The result is returned in ascending block order.

Sources: tuntang.top survey, section 2.3 (SparseSpec-L keeps sink + recent + historical top
tokens) and section 3 step 1 (`topk(k=kv_budget)` per decode step); tie-break by lower index
is this build's reading (deterministic, so the GPU set is checkable bit for bit).

Pinned by tests/test_oracle_select.py: rank-by-counting brute force, all-equal ties, NaN,
+-0 and infinities, and the |S| = min(K_b, nb), F in S properties.
"""
import numpy as np


def forced_blocks(nb: int, budget: int, n_sink: int, n_recent: int) -> np.ndarray:
    if nb <= budget:
        return np.arange(nb)
    sink = np.arange(min(n_sink, nb))
    recent = np.arange(max(0, nb - n_recent), nb)
    return np.union1d(sink, recent)


def select_blocks(scores: np.ndarray, nb: int, budget: int, n_sink: int, n_recent: int) -> np.ndarray:
    """scores: (>= nb,) fp32 block scores; returns the selected block ids, ascending (int64)."""
    if nb <= budget:
        return np.arange(nb, dtype=np.int64)
    forced = forced_blocks(nb, budget, n_sink, n_recent)
    is_forced = np.zeros(nb, bool)
    is_forced[forced] = True
    rest = np.nonzero(~is_forced)[0]
    s = scores[rest].astype(np.float64)
    # sort by (score descending, index ascending); numpy places NaN after every number
    order = np.lexsort((rest, -s))
    top = rest[order[: budget - forced.size]]
    return np.sort(np.concatenate([forced, top])).astype(np.int64)
