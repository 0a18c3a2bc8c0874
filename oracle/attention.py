"""Single-query softmax attention over the held tokens, and prefill attention mass (oracle).

KVLong §1.2 (重要性): attention scores a query against every key (Q K^T), normalises the
scores with softmax and takes the weighted average of V.
FADE-zh §项目结构与代码质量 (kernels/: fused INT4 dequant + SDPA): attention runs directly on
the dequantised tiers.
FADE-zh §四种驱逐策略详解 1 (H2O needs prefill attention) and KVLong §1.3.1 H2O (the token
importance is the column sum of the attention matrix): the prefill mass of key j is the sum,
over the query heads of its group and over the causal queries i >= j, of p[h, i, j].

Readings: scale 1/sqrt(d); no soft-cap, ALiBi bias or extra mask (the held set is already
causal); every query head of a GQA group attends to the group's one KV head; fp64 throughout.
Pinned by: torch scaled_dot_product_attention in float64 on CPU (a library routine), direct
summation on tiny caches, rows of p summing to one, and the prefill mass summing to the
number of query rows times heads.
"""

from __future__ import annotations

import numpy as np


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """q [G, d], k [N, d], v [N, d] (any float) -> (out [G, d], p [G, N], logits [G, N]),
    all float64. logits are the scaled scores (q . k) / sqrt(d)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    d = q.shape[-1]
    s = (q @ k.T) / np.sqrt(np.float64(d))
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=-1, keepdims=True)
    return p @ v, p, s


def prefill_mass(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """Causal attention mass per key for one (row, KV head).

    q [G, P, d] (query heads of the group, RoPE'd at 0..P-1), k [P, d] (RoPE'd) ->
    mass [P] float64 = sum_h sum_{i >= j} softmax_j(q_{h,i} . k_j / sqrt(d) over j <= i)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    G, P, d = q.shape
    s = np.einsum("gid,jd->gij", q, k) / np.sqrt(np.float64(d))
    causal = np.tril(np.ones((P, P), bool))
    s = np.where(causal[None], s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.where(causal[None], np.exp(s - m), 0.0)
    p = e / e.sum(axis=-1, keepdims=True)
    return p.sum(axis=(0, 1))
