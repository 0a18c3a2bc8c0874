"""Importance scores and victim selection (oracle).

FADE-zh §驱逐策略: when the INT4 budget is reached, tokens are evicted.
FADE-zh §四种驱逐策略详解: (1) H2O keeps the tokens with the highest accumulated attention;
(2) EMA tracks attention with an exponential moving average during decode; (3) position
evicts older tokens first and needs no attention. (4) the learned MLP policy needs a trained
checkpoint and is not part of this path.
KVLong §1.3.1 H2O: the score of a token is its accumulated attention (the attention matrix
summed by column); the lowest-scoring tokens are evicted.

Readings:
  * decisions are per (layer, row, KV head); the score of a token sums the probabilities of
    all G query heads of its group;
  * H2O: sigma_j += sum_h p[h, j]; EMA: sigma_j = delta*sigma_j + (1-delta)*sum_h p[h, j];
    every held token accumulates (sinks and recent too), only middle tokens are candidates;
  * victims are the ``k`` candidates with the smallest key (sigma_j, j); equal sigma evicts
    the lower (older) index first; the position policy uses the index alone.
Pinned by: brute force over every victim subset of small caches, the StreamingLLM kept-set
closed form for the position policy, the EMA closed form sigma_n = p(1 - delta^n) for a
constant p, and the H2O mass sum.
"""

from __future__ import annotations

import numpy as np


def h2o_update(sigma: np.ndarray, p: np.ndarray) -> np.ndarray:
    """sigma [N] + column sums of p [G, N]."""
    return sigma + p.sum(axis=0)


def ema_update(sigma: np.ndarray, p: np.ndarray, decay: float) -> np.ndarray:
    """decay * sigma + (1 - decay) * column sums of p [G, N]."""
    return decay * sigma + (1.0 - decay) * p.sum(axis=0)


def select_victims(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices (ascending) of the ``k`` smallest entries of ``keys`` by (value, index).

    ``keys`` is a 1-D array of candidate scores in index order (None: position policy)."""
    keys = np.asarray(keys)
    n = keys.shape[0]
    if not 0 <= k <= n:
        raise ValueError("cannot evict more tokens than there are candidates")
    idx = np.arange(n)
    order = np.lexsort((idx, keys))       # primary: value, secondary: index
    return np.sort(order[:k])


def select_victims_position(n: int, k: int) -> np.ndarray:
    """Position policy: the ``k`` oldest candidates."""
    if not 0 <= k <= n:
        raise ValueError("cannot evict more tokens than there are candidates")
    return np.arange(k)
