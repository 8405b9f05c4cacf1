"""Parity rules between a candidate (the CUDA path) and the oracle (TEST INFRASTRUCTURE).

Top-K: the selected set is unique except where scores tie or nearly tie at the K-th value.
With tau the oracle's K-th largest score and eps = 1e-3 * max(|tau|, 1e-30), a candidate set
passes when (i) it holds min(K, n) distinct positions in [0, n) and -1 in the other slots,
(ii) it holds every position scoring above tau + eps and (iii) no position scoring below
tau - eps.  Positions inside the band are free: fp32 scoring on the GPU and fp64 here may order
them differently.

Attention: the oracle's attention over the candidate's own indices is compared element-wise
(max-abs) with the candidate's output, which isolates the attention error from band swaps.
"""
from __future__ import annotations

import numpy as np

REL_BAND = 1e-3


def check_topk(cand_idx, scores: np.ndarray, K: int) -> dict:
    """Check one query's candidate index row against the oracle scores of its n visible
    positions.  Returns a report dict; raises AssertionError with a reason on failure."""
    cand = np.asarray(cand_idx, dtype=np.int64)
    n = scores.shape[0]
    m = min(K, n)
    assert cand.shape == (K,), f"index row has shape {cand.shape}, want ({K},)"
    valid = cand[cand >= 0]
    assert np.all(cand[cand < 0] == -1), "padding must be -1"
    assert valid.shape[0] == m, f"{valid.shape[0]} valid indices, want {m}"
    assert np.all(valid < n), "index beyond the visible range"
    assert np.unique(valid).shape[0] == m, "duplicate indices"
    if m == 0:
        return {"band": 0, "swaps": 0, "tau": None}
    tau = np.sort(scores)[::-1][m - 1]
    eps = REL_BAND * max(abs(tau), 1e-30)
    chosen = np.zeros(n, dtype=bool)
    chosen[valid] = True
    must = scores > tau + eps
    never = scores < tau - eps
    missing = np.flatnonzero(must & ~chosen)
    wrong = np.flatnonzero(never & chosen)
    assert missing.size == 0, f"{missing.size} positions above the band not selected, e.g. {missing[:5]}"
    assert wrong.size == 0, f"{wrong.size} positions below the band selected, e.g. {wrong[:5]}"
    band = ~must & ~never
    # swaps: band positions chosen by the candidate that the oracle's own order leaves out
    order = np.lexsort((np.arange(n), -scores))
    oracle_set = np.zeros(n, dtype=bool)
    oracle_set[order[:m]] = True
    swaps = int(np.count_nonzero(chosen & ~oracle_set))
    return {"band": int(band.sum()), "swaps": swaps, "tau": float(tau)}


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))
