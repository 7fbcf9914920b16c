"""Literal H2O greedy eviction (test infrastructure only).

Follows the H2O page ("H2O 完全拆解：抓住 KV Cache 里的「重击者」", section
贪心驱逐算法, Algorithm 1) step for step, in float64 numpy, for tiny inputs:
each new query attends (softmax, no self term) to the tokens currently cached,
every cached token's accumulated score gains its probability, the new token
joins the cache with score 0, and once the cache holds more than ``budget``
tokens the one with the lowest accumulated score leaves.  Among equal scores the
earliest-cached token (the first in cache order) leaves, which is what taking
the minimum over the cache in its insertion order does.

The page prints no scale inside the softmax; ``scale`` defaults to 1 so that the
literal reading is the default.  The function returns the final cache, the
per-step evicted token (or -1) and the accumulated scores.
"""
from __future__ import annotations

import numpy as np


def h2o_greedy_literal(Q: np.ndarray, K: np.ndarray, budget: int, scale: float = 1.0):
    """Run the greedy eviction loop over len(Q) steps.

    Q, K: float arrays [n, d] (one head).  Returns (cache, evicted, acc) where
    ``cache`` is the list of token positions kept at the end (in cache order),
    ``evicted[i]`` the token removed at step i (-1 when none) and ``acc`` a dict
    position -> accumulated attention of the tokens still cached.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    cache: list[int] = []
    acc: dict[int, float] = {}
    evicted: list[int] = []
    for i in range(Q.shape[0]):
        if cache:
            logits = scale * (K[cache] @ Q[i])
            e = np.exp(logits - logits.max())
            probs = e / e.sum()
            for tok, p in zip(cache, probs):
                acc[tok] += float(p)
        cache.append(i)
        acc[i] = 0.0
        gone = -1
        if len(cache) > budget:
            lowest = cache[0]
            for tok in cache[1:]:
                if acc[tok] < acc[lowest]:
                    lowest = tok
            cache.remove(lowest)
            del acc[lowest]
            gone = lowest
        evicted.append(gone)
    return cache, evicted, acc
