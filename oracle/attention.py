"""Decode attention over the decoded cache (oracle; test infrastructure only).

One query row per head attends over all cached positions with an exact,
max-subtracted softmax in FP64.  Grouped-query attention: query head h reads
KV head floor(h / G), G = n_q / n_kv, with no head expansion (summary page,
"전제와 한계").  Split-KV (summary page, "무엇과 다른가": long contexts are
split and reduced) is restated as per-chunk (max, sum-exp, weighted sum)
partials merged by rescaling to the common maximum -- the standard reading,
exact in real arithmetic.
"""
import numpy as np


def attend(q, k_hat, v_hat) -> np.ndarray:
    """q [d], k_hat/v_hat [n, d] -> softmax(k_hat q / sqrt(d)) @ v_hat, FP64."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    s = (np.asarray(k_hat, np.float64) @ q) / np.sqrt(d)
    s = s - np.max(s)
    p = np.exp(s)
    p = p / np.sum(p)
    return p @ np.asarray(v_hat, np.float64)


def _partial(q, k_hat, v_hat):
    d = q.shape[-1]
    s = (k_hat @ q) / np.sqrt(d)
    if s.size == 0:
        return -np.inf, 0.0, np.zeros(v_hat.shape[-1])
    m = np.max(s)
    e = np.exp(s - m)
    return m, float(np.sum(e)), e @ v_hat


def merge_partials(parts) -> np.ndarray:
    """Merge (m, l, acc) partials: rescale each to the global maximum."""
    m_all = max(p[0] for p in parts)
    l_tot = 0.0
    acc = 0.0
    for m, l, a in parts:
        if m == -np.inf:
            continue
        w = np.exp(m - m_all)
        l_tot += l * w
        acc = acc + a * w
    return acc / l_tot


def attend_split(q, k_hat, v_hat, n_split: int) -> np.ndarray:
    """Split the positions into n_split contiguous chunks, attend, merge."""
    q = np.asarray(q, dtype=np.float64)
    k_hat = np.asarray(k_hat, np.float64)
    v_hat = np.asarray(v_hat, np.float64)
    n = k_hat.shape[0]
    bounds = np.linspace(0, n, n_split + 1).round().astype(int)
    parts = [_partial(q, k_hat[a:b], v_hat[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
    return merge_partials(parts)
