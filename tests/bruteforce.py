"""Independent brute-force references used to pin the CPU oracle on tiny inputs.

Nothing here shares code with the oracle (``oracle/h2o_oracle.c``) or the CUDA path. Each function
computes a quantity the H2O pages fix by plain definition, in a different way than the oracle does:
dense causal attention with no cache at all, a sliding window with no scores at all, and
accumulated scores recomputed from scratch out of the history of attended sets.
"""

from __future__ import annotations

import math

import numpy as np


def widen(x: np.ndarray) -> np.ndarray:
    """Stored values (float32, or bf16 as uint16 bits) -> float64, exactly."""
    if x.dtype == np.float32:
        return x.astype(np.float64)
    assert x.dtype == np.uint16
    return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def attention_weights(q: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """softmax(q . K^T / sqrt(D)) for one query (float64)."""
    D = q.shape[-1]
    logits = keys @ q / math.sqrt(D)
    e = np.exp(logits - logits.max())
    return e / e.sum()


def attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """softmax(q . K^T / sqrt(D)) V for one query (float64). Returns (output, weights)."""
    w = attention_weights(q, keys)
    return w @ values, w


def dense_causal_attention(q_seq, k_seq, v_seq, t: int) -> np.ndarray:
    """The Full-KV-cache baseline: query t attends every position 0..t."""
    return attention(q_seq[t], k_seq[: t + 1], v_seq[: t + 1])[0]


def window_attention(q_seq, k_seq, v_seq, t: int, window: int) -> np.ndarray:
    """The Local (sliding window) baseline: query t attends positions max(0, t - window) .. t."""
    lo = max(0, t - window)
    return attention(q_seq[t], k_seq[lo: t + 1], v_seq[lo: t + 1])[0]


def causal_column_sums(q_seq, k_seq) -> np.ndarray:
    """c_j = sum_i softmax_row_i(j) of the causal prompt attention matrix, via a masked dense matrix."""
    P, D = q_seq.shape
    logits = (q_seq @ k_seq.T) / math.sqrt(D)
    mask = np.tril(np.ones((P, P), dtype=bool))
    logits = np.where(mask, logits, -np.inf)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    a = e / e.sum(axis=1, keepdims=True)
    return a.sum(axis=0)


def heavy_selection(c: np.ndarray, budget: int, k_heavy: int, k_local: int) -> list[int]:
    """Kept prompt positions (ascending) by a full sort: last k_local, plus the k_heavy largest
    column sums among the rest, equal sums keeping the later position."""
    P = len(c)
    if P <= budget:
        return list(range(P))
    older = sorted(range(P - k_local), key=lambda j: (-c[j], -j))
    return sorted(older[:k_heavy] + list(range(P - k_local, P)))


def recomputed_scores(q_seq, k_seq, prompt_len: int, history: list[tuple[int, list[int]]],
                      positions: list[int]) -> dict[int, float]:
    """Accumulated attention of each position in ``positions`` recomputed from raw Q/K:
    its prompt column sum (if it is a prompt position) plus, for every decode step (t, attended
    positions) in ``history`` that attended it, its softmax weight in that step."""
    total = {p: 0.0 for p in positions}
    c = causal_column_sums(q_seq[:prompt_len], k_seq[:prompt_len])
    for p in positions:
        if p < prompt_len:
            total[p] += c[p]
    for t, attended in history:
        w = attention_weights(q_seq[t], k_seq[attended])
        for idx, p in enumerate(attended):
            if p in total:
                total[p] += w[idx]
    return total


def harmonic(n: int) -> float:
    return math.fsum(1.0 / i for i in range(1, n + 1))
