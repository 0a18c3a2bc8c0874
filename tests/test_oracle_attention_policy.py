"""Pins of the oracle's attention, prefill mass and victim selection."""

import itertools
import math

import numpy as np
import pytest
import torch

from oracle import attention, policy
from synth import draw_scores


def _sdpa64(q, k, v):
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, None]
    kt = torch.from_numpy(np.asarray(k, np.float64))[None, None]
    vt = torch.from_numpy(np.asarray(v, np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, 0].numpy()


def test_attend_matches_torch_sdpa_float64():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((4, 128))
    k = rng.standard_normal((777, 128)) * 3
    v = rng.standard_normal((777, 128))
    out, p, s = attention.attend(q, k, v)
    assert np.allclose(out, _sdpa64(q, k, v), atol=1e-12, rtol=1e-12)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14)


def test_attend_direct_summation_tiny():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 4))
    k = rng.standard_normal((5, 4))
    v = rng.standard_normal((5, 4))
    out, p, _ = attention.attend(q, k, v)
    for h in range(2):
        w = [math.exp(sum(q[h, c] * k[j, c] for c in range(4)) / 2.0) for j in range(5)]
        z = sum(w)
        for c in range(4):
            assert math.isclose(out[h, c], sum(w[j] * v[j, c] for j in range(5)) / z,
                                rel_tol=1e-12, abs_tol=1e-12)


def test_prefill_mass_against_library_softmax_and_sum():
    rng = np.random.default_rng(2)
    G, P, d = 4, 96, 64
    q = rng.standard_normal((G, P, d))
    k = rng.standard_normal((P, d))
    m = attention.prefill_mass(q, k)
    # library routine: torch softmax with a causal mask in float64, then column sums
    s = torch.from_numpy(q) @ torch.from_numpy(k).T / math.sqrt(d)
    mask = torch.ones(P, P, dtype=torch.bool).tril()
    pt = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1)
    assert np.allclose(m, pt.sum(dim=(0, 1)).numpy(), atol=1e-12)
    # each causal query row sums to one: the mass of the prompt is G*P
    assert math.isclose(m.sum(), G * P, rel_tol=1e-12)
    # the first query row puts all its mass on token 0, the last key only sees the last row
    assert m[0] >= G - 1e-12


def test_prefill_mass_brute_force_tiny():
    rng = np.random.default_rng(3)
    G, P, d = 2, 5, 4
    q = rng.standard_normal((G, P, d))
    k = rng.standard_normal((P, d))
    want = np.zeros(P)
    for h in range(G):
        for i in range(P):
            w = [math.exp(float(q[h, i] @ k[j]) / 2.0) for j in range(i + 1)]
            for j in range(i + 1):
                want[j] += w[j] / sum(w)
    assert np.allclose(attention.prefill_mass(q, k), want, atol=1e-13)


def _dominates(a, b):
    return all(x <= y for x, y in zip(a, b))


@pytest.mark.parametrize("seed", range(12))
def test_select_victims_brute_force(seed):
    keys = draw_scores(8, seed, tie_fraction=0.5, levels=np.array([0.0, 1.0], np.float32))
    items = [(float(keys[i]), i) for i in range(8)]
    for k in range(9):
        chosen = policy.select_victims(keys, k)
        assert len(chosen) == k and np.all(np.diff(chosen) > 0)
        mine = sorted(items[i] for i in chosen)
        # the k smallest (value, index) pairs dominate every other k-subset element-wise
        for other in itertools.combinations(range(8), k):
            assert _dominates(mine, sorted(items[i] for i in other))


def test_select_prefers_lower_index_on_ties():
    keys = np.array([0.5, 0.2, 0.2, 0.2, 0.9], np.float32)
    assert policy.select_victims(keys, 2).tolist() == [1, 2]
    assert policy.select_victims(np.zeros(6), 3).tolist() == [0, 1, 2]
    assert policy.select_victims_position(10, 4).tolist() == [0, 1, 2, 3]


def test_ema_closed_form_constant_input():
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(30), size=4)              # G=4 heads, constant over steps
    sigma = np.zeros(30)
    delta = 0.9
    for n in range(1, 41):
        sigma = policy.ema_update(sigma, p, delta)
        assert np.allclose(sigma, p.sum(0) * (1 - delta ** n), atol=1e-14)


def test_h2o_sum_counts_heads_times_steps():
    rng = np.random.default_rng(6)
    sigma = np.zeros(50)
    for n in range(1, 21):
        sigma = policy.h2o_update(sigma, rng.dirichlet(np.ones(50), size=8))
        assert math.isclose(sigma.sum(), 8 * n, rel_tol=1e-12)
