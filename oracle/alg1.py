"""H2O greedy eviction in its plain form (test infrastructure only).

Restates what the H2O page ("H2O 完全拆解：抓住 KV Cache 里的「重击者」", sections
问题形式化 and 贪心驱逐算法) defines, for one head and tiny inputs, in float64
numpy.  State is kept per token position: an accumulated-attention array and a
membership mask of the cache.  At step i:

1. the query of token i attends to the cached tokens only (the new token does
   not see itself): a softmax over their logits;
2. every cached token's accumulated score gains the probability it received;
3. token i enters the cache with accumulated score 0;
4. when the cache then holds more than ``budget`` tokens, exactly one leaves: the
   member with the smallest accumulated score, the lowest position among equal
   scores (positions enter in increasing order, so this is also the earliest
   cached).

The page's softmax carries no scale; ``scale`` defaults to 1 so that this
reading is the default.
"""
from __future__ import annotations

import numpy as np


def h2o_greedy_literal(Q: np.ndarray, K: np.ndarray, budget: int, scale: float = 1.0):
    """Run the greedy eviction over len(Q) steps.

    Q, K: float arrays [n, d] (one head; token i has query Q[i] and key K[i]).
    Returns (kept, evicted, acc): ``kept`` the cached positions at the end in
    ascending order, ``evicted[i]`` the position that left at step i (-1 when
    none), and ``acc`` a float64 array over positions holding each kept token's
    accumulated score (NaN for tokens no longer cached).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    n = Q.shape[0]
    score = np.zeros(n, dtype=np.float64)
    cached = np.zeros(n, dtype=bool)
    evicted = [-1] * n
    for i in range(n):
        members = np.flatnonzero(cached)  # ascending positions
        if members.size:
            logits = scale * (K[members] @ Q[i])
            w = np.exp(logits - logits.max())
            score[members] += w / w.sum()
        cached[i] = True  # score[i] is still 0
        if np.count_nonzero(cached) > budget:
            members = np.flatnonzero(cached)
            victim = int(members[np.argmin(score[members])])  # first minimum = lowest position
            cached[victim] = False
            evicted[i] = victim
    acc = np.where(cached, score, np.nan)
    return np.flatnonzero(cached).tolist(), evicted, acc
