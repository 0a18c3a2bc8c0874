"""Pins of the oracle's tiered cache (step order, tiers, eviction, accounting)."""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import accounting, quant
from oracle.cache import Params, UnitCache
from oracle.rope import RopeTable
from synth import Workload, draw_decode_tokens, draw_prompt, get_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def _unit(S, W, budget, policy, d=64, G=4, kb=4, vb=2, max_pos=8192, rope_kind="default"):
    p = Params(d, G, S, W, budget, policy, kb, vb, 0.9)
    return UnitCache(p, RopeTable(rope_kind, d, max_pos, base=10000.0))


def _tiny_wl(**kw):
    base = dict(name="tiny", layers=1, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64,
                n_sink=2, recent_window=4, int4_budget=-1, policy="none", middle_k_bits=4,
                middle_v_bits=2, prompt_len=0, steps=0, seed=7)
    base.update(kw)
    return Workload(**base)


def test_safe_mode_all_fp16_equals_sdpa():
    # sinks + window hold every token: attention must be plain attention over rotated keys
    u = _unit(S=4, W=64, budget=-1, policy="none")
    wl = _tiny_wl(n_sink=4, recent_window=64)
    pr = draw_prompt(wl, 0, 20)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0])
    assert u.n_mid == 0
    keys = [u.rope.apply(pr["k"][0, 0], np.arange(20))]
    vals = [pr["v"][0, 0]]
    for step in range(30):
        t = draw_decode_tokens(wl, 0, step)
        out, p, _, pos = u.step(t["q"][0], t["k"][0, 0], t["v"][0, 0])
        assert pos == 20 + step
        keys.append(u.rope.apply(t["k"][0, 0][None], pos))
        vals.append(t["v"][0, 0][None])
        q = u.rope.apply(t["q"][0], pos)
        qt = torch.from_numpy(q.astype(np.float64))[None]
        kt = torch.from_numpy(np.concatenate(keys).astype(np.float64))[None, None]
        vt = torch.from_numpy(np.concatenate(vals).astype(np.float64))[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt[:, :, None], kt.expand(1, 4, -1, -1),
                                                               vt.expand(1, 4, -1, -1))
        assert np.allclose(out, ref[0, :, 0].numpy(), atol=1e-12)
        assert math.isclose(p.sum(), 4.0, rel_tol=1e-12)


def test_tier_arithmetic_single_layer_workload():
    # 511-token prompt + one decode step = 4 sinks + 444 middle + 64 recent = 512 held
    wl = get_workload(1)
    u = UnitCache(Params.from_workload(wl), RopeTable.from_workload(wl, 1024))
    pr = draw_prompt(wl, 0)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0])
    t = draw_decode_tokens(wl, 0, 0)
    u.step(t["q"][0, :wl.group], t["k"][0, 0], t["v"][0, 0])
    assert (u.n_sink, u.n_mid, u.n_recent) == (4, 444, 64)


def test_position_policy_keeps_streaming_llm_set():
    # StreamingLLM closed form: sinks plus the newest (budget + window) tokens
    S, W, budget = 2, 4, 6
    u = _unit(S, W, budget, "position")
    wl = _tiny_wl(n_sink=S, recent_window=W)
    P = 30
    pr = draw_prompt(wl, 0, P)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0])
    total = P
    for step in range(25):
        t = draw_decode_tokens(wl, 0, step)
        u.step(t["q"][0], t["k"][0, 0], t["v"][0, 0])
        total += 1
        want = list(range(S)) + list(range(total - budget - W, total))
        assert u.orig_pos.tolist() == want
        assert u.n_mid == budget


def test_h2o_mass_sum_without_eviction():
    u = _unit(S=2, W=4, budget=-1, policy="h2o")
    wl = _tiny_wl()
    P = 16
    pr = draw_prompt(wl, 0, P)
    mass = np.full(P, 4.0)                  # any prefill mass; G*P in total = 64
    u.prefill(pr["k"][0, 0], pr["v"][0, 0], mass=mass)
    for step in range(10):
        t = draw_decode_tokens(wl, 0, step)
        u.step(t["q"][0], t["k"][0, 0], t["v"][0, 0])
        assert math.isclose(u.sigma.sum(), 4 * P + 4 * (step + 1), rel_tol=1e-12)


def test_h2o_mass_sum_with_eviction_drops_evicted_mass():
    u = _unit(S=2, W=4, budget=3, policy="h2o")
    wl = _tiny_wl()
    pr = draw_prompt(wl, 0, 9)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0], mass=np.zeros(9))
    total = 0.0
    for step in range(20):
        before = u.sigma.copy()
        s0 = u.n_sink
        t = draw_decode_tokens(wl, 0, step)
        u.demote()
        vic = u.choose_victims()
        dropped = before[s0 + vic].sum()
        u.evict(vic)
        pos = u.n_held
        u.append(u.rope.apply(t["k"][0, 0][None], pos), t["v"][0, 0])
        _, p, _ = u.attend(u.rope.apply(t["q"][0], pos))
        u.accumulate(p)
        total += 4.0 - dropped
        assert math.isclose(u.sigma.sum(), total, rel_tol=1e-12, abs_tol=1e-12)


def test_brute_force_eight_token_cache():
    # tiny H2O cache: every eviction is the brute-force minimum, and attention is direct
    # summation over the dequantised held tokens
    u = _unit(S=1, W=2, budget=3, policy="h2o")
    wl = _tiny_wl(n_sink=1, recent_window=2)
    pr = draw_prompt(wl, 0, 6)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0], mass=np.arange(6, dtype=float)[::-1].copy())
    for step in range(12):
        t = draw_decode_tokens(wl, 0, step)
        u.demote()
        s0, n_mid = u.n_sink, u.n_mid
        keys = u.sigma[s0:s0 + n_mid]
        k = max(0, n_mid - 3)
        vic = u.choose_victims()
        best = min(itertools.combinations(range(n_mid), k),
                   key=lambda c: sorted((keys[i], i) for i in c)[::-1] if c else ())
        assert sorted(vic.tolist()) == sorted(best)
        u.evict(vic)
        pos = u.n_held
        u.append(u.rope.apply(t["k"][0, 0][None], pos), t["v"][0, 0])
        q = u.rope.apply(t["q"][0], pos).astype(np.float64)
        out, p, _ = u.attend(q)
        K, V = u.keys(), u.values()
        for h in range(4):
            w = [math.exp(float(q[h] @ K[j]) / 8.0) for j in range(K.shape[0])]
            ref = sum(w[j] * V[j] for j in range(len(w))) / sum(w)
            assert np.allclose(out[h], ref, atol=1e-12)
        u.accumulate(p)
        assert u.n_held <= 1 + 3 + 2


def test_eviction_keeps_relative_positions_of_recent_tokens():
    # recent tokens are FP16 (no re-quantisation): after an eviction shifts them by one,
    # their logits against the next query match the fp64 rotation by original distance
    u = _unit(S=2, W=4, budget=2, policy="position", d=64)
    wl = _tiny_wl()
    pr = draw_prompt(wl, 0, 8)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0])
    for step in range(3):
        t = draw_decode_tokens(wl, 0, step)
        _, _, logits, pos = u.step(t["q"][0], t["k"][0, 0], t["v"][0, 0])
    raw_k = {i: pr["k"][0, 0][i] for i in range(8)}
    for s in range(3):
        raw_k[8 + s] = draw_decode_tokens(wl, 0, s)["k"][0, 0]
    inv = u.rope.inv_freq.astype(np.float64)
    from oracle.rope import rotate64
    q_raw = t["q"][0].astype(np.float64)
    n_rec = u.n_recent
    for r in range(n_rec):
        j = u.n_sink + u.n_mid + r
        orig = u.orig_pos[j]
        dist = (u.seen - 1) - orig                      # query is the newest token
        want = rotate64(q_raw, dist * inv) @ raw_k[orig].astype(np.float64) / 8.0
        assert np.allclose(logits[:, j], want, atol=0.05, rtol=0.02)


def test_compression_accounting_matches_pages_figures():
    g = json.load(open(GOLDEN))
    # safe preset on the Qwen2.5-3B shape (K4/V4, 4096 tokens): inside the stated 3-4x
    wl = get_workload(2)
    n_fp16 = wl.n_sink + wl.recent_window
    comp = accounting.compressed_bytes(wl.layers, wl.num_kv_heads, 128, wl.n_sink,
                                       wl.recent_window, 4096 - n_fp16, 4, 4)
    base = accounting.fp16_bytes(wl.layers, wl.num_kv_heads, 128, 4096)
    lo, hi = g["preset_compression"]["safe"]
    assert lo <= base / comp <= hi
    assert math.isclose(base / comp, 3.41, abs_tol=0.005)
    # INT2 V: about 30% more compression than INT4 V at d=128
    gain = accounting.middle_token_bytes(128, 4, 4) / accounting.middle_token_bytes(128, 4, 2)
    assert abs((gain - 1) - g["int2_v_extra_compression_about"]["value"]) < 0.05
    # Llama-3.2-1B: 29.9 MiB of FP16 at 32 KiB per token; about 29% evicted; K4/V2 middle
    ll = g["llama-3.2-1b"]
    per_tok = accounting.fp16_bytes(ll["layers"], ll["kv_heads"], ll["head_dim"], 1)
    assert per_tok == 32 * 1024
    seen = round(ll["baseline_mib"] * 2 ** 20 / per_tok)
    kept = round(seen * (1 - ll["eviction_rate_about"]))
    tiered = accounting.compressed_bytes(ll["layers"], ll["kv_heads"], ll["head_dim"], 4, 64,
                                         kept - 68, 4, 2)
    assert abs(tiered / 2 ** 20 - ll["tiered_mib"]) < 0.05


def test_custom_config_example_is_the_balanced_workload():
    g = json.load(open(GOLDEN))["custom_config_example"]
    wl = get_workload(3)
    assert (wl.n_sink, wl.recent_window, wl.int4_budget, wl.policy, wl.middle_k_bits,
            wl.middle_v_bits) == (g["n_sink"], g["recent_window"], g["int4_budget"],
                                  g["eviction_policy"], g["middle_k_bits"], g["middle_v_bits"])


def test_demoted_token_keeps_its_index_and_codes_are_its_quantisation():
    u = _unit(S=2, W=4, budget=-1, policy="none")
    wl = _tiny_wl()
    pr = draw_prompt(wl, 0, 6)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0])
    assert (u.n_sink, u.n_mid, u.n_recent) == (2, 0, 4)
    oldest = u.rec_k[0].copy()
    u.demote()
    q, s = quant.quantize(oldest[None], 4)
    assert np.array_equal(u.mid_kq[0], q[0]) and np.array_equal(u.mid_ks[0], s[0])
    assert u.orig_pos[2] == 2


def _units_with_scores(rows_sigma, S=2, W=4, budget=3, policy="h2o"):
    """Units of one (layer, KV head) whose middle tiers hold len(sigma) tokens with the given
    scores (one unit per row)."""
    from oracle.cache import choose_shared_victims  # noqa: F401  (imported by the tests)
    units = []
    wl = _tiny_wl(n_sink=S, recent_window=W)
    n_mid = len(rows_sigma[0])
    pr = draw_prompt(wl, 0, S + n_mid + W)
    for sig in rows_sigma:
        u = _unit(S=S, W=W, budget=-1, policy="none")
        u.prefill(pr["k"][0, 0], pr["v"][0, 0])
        u.p = Params(64, 4, S, W, budget, policy, 4, 2, 0.9)
        u.sigma = np.concatenate([np.zeros(S), np.asarray(sig, np.float64), np.zeros(W)])
        units.append(u)
    return units


def test_shared_victims_reduce_to_one_row_and_to_identical_rows():
    from oracle.cache import choose_shared_victims

    rng = np.random.default_rng(11)
    sig = rng.random(9)
    one = _units_with_scores([sig])
    assert np.array_equal(choose_shared_victims(one), one[0].choose_victims())
    same = _units_with_scores([sig] * 4)           # identical rows: the same choice
    assert np.array_equal(choose_shared_victims(same), one[0].choose_victims())


def test_shared_victims_follow_the_row_sum_not_any_row():
    from oracle.cache import choose_shared_victims

    # row 0 alone would drop index 0, row 1 alone index 2; their sums [10, 6, 10, ...] drop 1
    rows = [[1.0, 3.0, 9.0, 20.0, 20.0], [9.0, 3.0, 1.0, 20.0, 20.0]]
    units = _units_with_scores(rows, budget=4)
    assert list(units[0].choose_victims()) == [0] and list(units[1].choose_victims()) == [2]
    assert list(choose_shared_victims(units)) == [1]
    # equal sums: the lower index goes first, as for one row
    tie = _units_with_scores([[1.0, 5.0, 9.0], [9.0, 5.0, 1.0]], budget=2)
    assert list(choose_shared_victims(tie)) == [0]
    # rows with different tier counts cannot share decisions
    bad = _units_with_scores([[1.0, 2.0, 3.0]]) + _units_with_scores([[1.0, 2.0, 3.0, 4.0]])
    with pytest.raises(ValueError):
        choose_shared_victims(bad)
