"""Pins of the oracle's re-positioning of keys (FADE-zh §驱逐策略, §RoPE重计算; KVLong §1.2.2
StreamingLLM: a key held at cache index j carries the rotation of position j).

Each pin compares the oracle's stored keys with an independent fp64 statement of what they
must be: the rotation of a key by exact angles j * base^(-2i/d), computed here in fp64 from
the definition of RoPE (not from the oracle's fp32 table), with a tolerance derived from the
arithmetic the pages fix:
  * a middle key is stored quantised: |x - q s| <= s/2 per channel (s: its group's scale);
  * every fp32 -> fp16 cast adds at most 2^-11 |x| (half an fp16 ulp, relative);
  * the fp32 table angle RN32(j * RN32(inv_i)) differs from j * inv_i by at most
    ~2^-23 * j * inv_i, and each fp32 rotation adds a few 2^-24 |x|.
Mutation tests plant the plausible mistakes in the oracle (a re-positioning to the wrong index,
a skipped rotation, a skipped re-quantisation) and check that a pin fails.
"""

import numpy as np
import pytest

from oracle import quant
from oracle.cache import Params, UnitCache
from oracle.rope import RopeTable
from synth import Workload, draw_decode_tokens, draw_prompt

BASE = 10000.0
D = 64


RD = {"r": D}   # rotated width (proportional RoPE); the tests set it


def _inv64(r=None, base=BASE):
    r = RD["r"] if r is None else r
    i = np.arange(r // 2, dtype=np.float64)
    return base ** (-2.0 * i / r)


def _rot64(x, pos):
    """fp64 rotate-half rotation of the first r channels of x [..., D] to position(s) pos
    (exact angles); the other channels pass through."""
    x = np.asarray(x, np.float64)
    r = RD["r"]
    ang = np.asarray(pos, np.float64)[..., None] * _inv64()
    c, s = np.cos(ang), np.sin(ang)
    h = r // 2
    x1, x2, rest = x[..., :h], x[..., h:r], x[..., r:]
    rest = np.broadcast_to(rest, x1.shape[:-1] + rest.shape[-1:]) if rest.ndim < x1.ndim else rest
    y1, y2 = x1 * c - x2 * s, x2 * c + x1 * s
    rest = np.broadcast_to(rest, y1.shape[:-1] + rest.shape[-1:])
    return np.concatenate([y1, y2, rest], axis=-1)


def _pair_norm(x):
    r = RD["r"]
    h = r // 2
    n = np.sqrt(x[..., :h] ** 2 + x[..., h:r] ** 2)
    return np.concatenate([n, n, np.abs(x[..., r:])], axis=-1)


def _angle_tol(x, positions):
    """Rotation error allowance per channel: fp32 table angles at `positions` (summed) plus
    fp32 rounding of the rotations, on the pair magnitude (none on pass-through channels)."""
    r = RD["r"]
    inv = np.concatenate([_inv64(), _inv64(), np.zeros(D - r)])
    rot = np.concatenate([np.ones(r), np.zeros(D - r)])
    ptot = np.asarray(positions, np.float64)[..., None]
    return _pair_norm(x) * (2.0 ** -22 * (ptot + 1.0) * inv + 2.0 ** -20 * rot)


def _scales_per_channel(ks):
    return np.repeat(ks.astype(np.float64), quant.GROUP, axis=-1)


def _wl(S, W):
    return Workload(name="pin", layers=1, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=D,
                    n_sink=S, recent_window=W, int4_budget=-1, policy="none", middle_k_bits=4,
                    middle_v_bits=2, prompt_len=0, steps=0, k_outlier_channels=2,
                    outlier_scale=10.0, seed=31)


def _unit(S, W, budget, policy):
    p = Params(D, 4, S, W, budget, policy, 4, 2, 0.9)
    return UnitCache(p, RopeTable("default", D, 8192, base=BASE, rotary_dim=RD["r"]))


@pytest.fixture(params=[64, 32, 48], ids=["full", "rotary32", "rotary48"], autouse=True)
def rotary(request):
    """Every pin runs with full RoPE and with proportional RoPE over 32 channels (one whole
    quantisation group rotates) and 48 (the rotated width splits the second group)."""
    RD["r"] = request.param
    yield request.param
    RD["r"] = D


def _prefilled(policy, S=4, W=8, budget=40, P=120, seed=5):
    wl = _wl(S, W)
    pr = draw_prompt(wl, 0, P)
    u = _unit(S, W, budget, policy)
    rng = np.random.default_rng(seed)
    mass = rng.gamma(0.5, 2.0, P) if policy == "h2o" else None
    u.prefill(pr["k"][0, 0], pr["v"][0, 0], mass=mass)
    return wl, u, pr["k"][0, 0]


# ---------------------------------------------------------------------------- the pins
def decode_eviction_violations(u, wl, steps=6):
    """Run `steps` decode steps that evict; at each, compare every surviving middle key after
    the eviction with the fp64 rotation of its dequantised value before it, by the exact angle
    of its index change, and the logit of every survivor whose distance to the query did not
    change. Returns (number of checked keys, number of violations)."""
    checked = bad = 0
    for step in range(steps):
        t = draw_decode_tokens(wl, 0, step)
        u.demote()
        s0 = u.n_sink
        k_before = u.keys()                      # fp64, cache order, after the demotion
        op_before = u.orig_pos.copy()
        n_held_before = u.n_held
        vic = u.choose_victims()
        assert vic.size > 0, "the pin needs a step that evicts"
        u.evict(vic)
        k_after = u.keys()
        j_old_of = {int(o): j for j, o in enumerate(op_before)}
        mid = range(s0, s0 + u.n_mid)
        for j_new in mid:
            j_old = j_old_of[int(u.orig_pos[j_new])]
            x_old = k_before[j_old]
            want = _rot64(x_old, j_new - j_old)
            sc = _scales_per_channel(u.mid_ks[j_new - s0])
            if j_old == j_new:
                ok = np.array_equal(k_after[j_new], x_old)   # unmoved: untouched
            else:
                tol = sc / 2 + 2.0 ** -11 * np.abs(want) + _angle_tol(x_old, j_old + j_new)
                ok = np.all(np.abs(k_after[j_new] - want) <= tol * (1 + 1e-9))
            checked += 1
            bad += not ok
        # logits at unchanged distance: the next query sits at n_held (after the eviction)
        P_new = u.n_held
        P_old = n_held_before
        q = _rot64(t["q"][0].astype(np.float64), P_new)
        q_old = _rot64(t["q"][0].astype(np.float64), P_old)
        last_victim = s0 + int(vic.max())
        for j_new in mid:
            j_old = j_old_of[int(u.orig_pos[j_new])]
            if j_old <= last_victim:                 # before a victim: its distance changed
                continue
            assert P_old - j_old == P_new - j_new
            sc = _scales_per_channel(u.mid_ks[j_new - s0])
            x_old = k_before[j_old]
            ktol = sc / 2 + 2.0 ** -11 * np.abs(k_after[j_new]) + _angle_tol(x_old, j_old + j_new)
            lt = np.abs(q) @ ktol + np.abs(q).sum(1) * 1e-9
            diff = np.abs(q @ k_after[j_new] - q_old @ x_old)
            checked += 1
            bad += not np.all(diff <= lt * (1 + 1e-9))
        pos = u.n_held
        u.append(u.rope.apply(t["k"][0, 0][None], pos), t["v"][0, 0])
        _, p, _ = u.attend(u.rope.apply(t["q"][0], pos))
        u.accumulate(p)
    return checked, bad


def prefill_violations(u, k_raw):
    """Every key held after a prefill with evictions against the fp64 rotation of its raw
    key to its cache index: FP16 tiers within two fp16 roundings (rotation at the original
    position, then re-positioning), middle keys within s/2 more."""
    K = u.keys()
    s0, n_mid = u.n_sink, u.n_mid
    checked = bad = 0
    for j in range(u.n_held):
        o = int(u.orig_pos[j])
        x = k_raw[o].astype(np.float64)
        want = _rot64(x, j)
        tol = 2 * 2.0 ** -11 * _pair_norm(x) + _angle_tol(x, o + j)
        if s0 <= j < s0 + n_mid:
            tol = tol + _scales_per_channel(u.mid_ks[j - s0]) / 2
        checked += 1
        bad += not np.all(np.abs(K[j] - want) <= tol * (1 + 1e-9))
    return checked, bad


@pytest.mark.parametrize("policy", ["position", "h2o"])
def test_moved_middle_keys_are_rotations_by_their_index_change(policy):
    wl, u, _ = _prefilled(policy)
    checked, bad = decode_eviction_violations(u, wl)
    assert checked > 200 and bad == 0


@pytest.mark.parametrize("policy", ["position", "h2o", "ema"])
def test_prefill_survivors_are_rotated_to_their_cache_index(policy):
    _, u, k_raw = _prefilled(policy)
    assert u.n_mid == 40 and np.any(u.orig_pos != np.arange(u.n_held))
    checked, bad = prefill_violations(u, k_raw)
    assert checked == u.n_held and bad == 0


def test_h2o_eviction_moves_keys_on_both_sides_of_a_victim():
    # the pin above covers unmoved keys (before the first victim) and moved ones
    wl, u, _ = _prefilled("h2o")
    u.demote()
    vic = u.choose_victims()
    assert 0 < vic.min() < u.n_mid - 1


# ---------------------------------------------------------------------------- mutations
def _plant(monkeypatch, kind):
    """Plant a mistake in the oracle's re-positioning (on the CPU)."""
    orig = RopeTable.reposition

    def wrong_index(self, x, old_pos, new_pos):
        return orig(self, x, old_pos, np.asarray(new_pos) + 4)   # off by the sink count

    def skipped_rotation(self, x, old_pos, new_pos):
        return np.asarray(x, np.float32).astype(np.float16)

    def inverse_only(self, x, old_pos, new_pos):
        return orig(self, x, old_pos, np.zeros_like(np.asarray(new_pos)))

    monkeypatch.setattr(RopeTable, "reposition",
                        {"index": wrong_index, "skip": skipped_rotation,
                         "inverse": inverse_only}[kind])


@pytest.mark.parametrize("kind", ["index", "skip", "inverse"])
@pytest.mark.parametrize("policy", ["position", "h2o"])
def test_decode_pin_catches_a_planted_repositioning_mistake(monkeypatch, kind, policy):
    wl, u, _ = _prefilled(policy)
    _plant(monkeypatch, kind)
    _, bad = decode_eviction_violations(u, wl, steps=2)
    assert bad > 0


@pytest.mark.parametrize("kind", ["index", "skip", "inverse"])
def test_prefill_pin_catches_a_planted_repositioning_mistake(monkeypatch, kind):
    _plant(monkeypatch, kind)
    _, u, k_raw = _prefilled("position")
    _, bad = prefill_violations(u, k_raw)
    assert bad > 0


def test_decode_pin_catches_a_skipped_requantisation(monkeypatch):
    # moved keys keep their old codes and scales (the rotation is computed but not stored)
    wl, u, _ = _prefilled("position")
    orig_evict = UnitCache.evict

    def evict_without_requant(self, victims=None):
        kq, ks = self.mid_kq.copy(), self.mid_ks.copy()
        v = orig_evict(self, victims)
        keep = np.ones(kq.shape[0], bool)
        keep[v] = False
        self.mid_kq, self.mid_ks = kq[keep], ks[keep]
        return v

    monkeypatch.setattr(UnitCache, "evict", evict_without_requant)
    _, bad = decode_eviction_violations(u, wl, steps=2)
    assert bad > 0
