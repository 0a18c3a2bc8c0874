"""Lockstep runner for parity tests: the CUDA path (through the C ABI) and the oracle step the
same seeded workload and are compared after every call.

Both sides start from the same raw fp16 draws (``synth``). The oracle never reads anything the
CUDA path produced; the only value passed from the oracle to the CUDA path is the H2O prefill
mass, an input of the prefill call that the oracle computes (rounded to fp32 and given to both
sides so their selections see identical keys).
"""

from __future__ import annotations

import numpy as np

from oracle import attention, quant
from oracle.cache import Params, UnitCache
from oracle.rope import RopeTable
from synth import draw_decode_tokens, draw_prompt, ragged_context_lengths
from synth.draws import pq_calibration

ATOL, RTOL = 2e-3, 1e-2          # the spec's attention / score tolerance (allclose form)
TIE_RTOL = 1e-5                  # fp32-vs-fp64 score noise that may flip a near-tie


def allclose_report(got, ref, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    return (not bad.any()), float(err.max(initial=0.0)), int(bad.sum())


def victims_from_bits(words, n_mid):
    """Victim middle indices from a unit's selection bitmap words (bit i = index i)."""
    words = np.ascontiguousarray(words[:(n_mid + 31) // 32], np.uint32)
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:n_mid]
    return np.nonzero(bits)[0]


def oracle_unit_step(u, t, b, h, G, policy, gpu_words=None, evict=True):
    """One decode step of oracle unit ``u`` (layer row b, KV head h) on the raw draws ``t``
    (q [B][Hq][d], k, v [B][Hkv][d]): demote, evict, append, attend, accumulate. Under H2O /
    EMA the oracle's own fp64 selection is compared with the GPU's victims (``gpu_words``, the
    unit's selection bitmap); where they differ they must be a near-tie, and the oracle then
    adopts the GPU's victims (R10) and the unit stays under comparison.
    Returns (attention output [G, d] fp64, whether a near-tie was adopted)."""
    u.demote()
    n_mid = u.n_mid
    vic = u.choose_victims() if evict else np.zeros(0, np.int64)
    tie = False
    if vic.size and policy in ("h2o", "ema") and gpu_words is not None:
        gpu_vic = victims_from_bits(gpu_words, n_mid)
        if not np.array_equal(np.sort(gpu_vic), np.sort(vic)):
            keys = u.sigma[u.n_sink:u.n_sink + n_mid]
            a, g = np.sort(keys[vic]), np.sort(keys[gpu_vic])
            assert gpu_vic.size == vic.size and np.allclose(a, g, rtol=TIE_RTOL, atol=1e-7), (
                f"selection differs beyond a near-tie at row {b} head {h}: oracle {vic} {a}, "
                f"gpu {gpu_vic} {g}")
            vic = gpu_vic
            tie = True
    if evict:
        u.evict(vic)
    pos = u.n_held
    u.append(u.rope.apply(t["k"][b, h][None], pos), t["v"][b, h])
    out, p, _ = u.attend(u.rope.apply(t["q"][b, h * G:(h + 1) * G], pos))
    u.accumulate(p)
    return out, tie


def compare_unit_state(g, u, where):
    """A unit's GPU tiers (``g``, cache order) against the oracle unit: counts, FP16 tiers,
    packed codes and scales bit for bit; scores within the tolerance."""
    assert (g["n_sink"], g["n_mid"], g["n_recent"]) == (u.n_sink, u.n_mid, u.n_recent), \
        f"tier counts differ at {where}: gpu {(g['n_sink'], g['n_mid'], g['n_recent'])} " \
        f"oracle {(u.n_sink, u.n_mid, u.n_recent)}"
    eq16 = lambda a, r: np.array_equal(np.asarray(a).view(np.uint16), np.asarray(r).view(np.uint16))
    assert eq16(g["sink_k"], u.sink_k) and eq16(g["sink_v"], u.sink_v), f"sinks differ at {where}"
    assert eq16(g["recent_v"], u.rec_v), f"recent V differs at {where}"
    if not eq16(g["recent_k"], u.rec_k):
        d = np.nonzero(np.asarray(g["recent_k"]).view(np.uint16) != u.rec_k.view(np.uint16))
        raise AssertionError(f"recent K differs at {where}: {len(d[0])} entries, first {d[0][:5]}")
    kc = quant.pack(u.mid_kq, u.p.k_bits)
    vc = u.mid_vq if u.p.v_codec == "pq" else quant.pack(u.mid_vq, u.p.v_bits)
    for name, got, ref in (("mid K codes", g["mid_k_codes"], kc),
                           ("mid V codes", g["mid_v_codes"], vc)):
        if not np.array_equal(got, ref):
            rows = np.nonzero((got != ref).any(-1))[0]
            raise AssertionError(f"{name} differ at {where}: rows {rows[:8]} of {len(rows)}")
    assert eq16(g["mid_k_scales"], u.mid_ks), f"mid K scales differ at {where}"
    assert eq16(g["mid_v_scales"], u.mid_vs), f"mid V scales differ at {where}"
    if u.p.policy in ("h2o", "ema"):
        ok, err, nbad = allclose_report(g["scores"], u.sigma)
        assert ok, f"scores differ at {where}: max err {err}, {nbad} bad"


class Lockstep:
    """Drives ``FadeCache`` and per-unit oracle caches over a workload."""

    def __init__(self, wl, layers=None, steps=None, device="cuda", mid_capacity=None,
                 shared_rows=False, v_codec="int"):
        import dataclasses

        import torch

        from tiered_mixed_precision_gb300 import Config
        from tiered_mixed_precision_gb300.model import FadeCache

        self.torch = torch
        self.wl = wl
        self.L = wl.layers if layers is None else layers
        self.steps = wl.steps if steps is None else steps
        self.lens = ragged_context_lengths(wl)
        self.maxP = int(self.lens.max())
        self.max_pos = self.maxP + self.steps + 8
        self.shared = shared_rows   # the rows share their tier decisions (row-summed scores)
        self.cfg = dataclasses.replace(Config.from_workload(wl, mid_capacity=mid_capacity),
                                       shared_rows=shared_rows, v_codec=v_codec)
        self.fc = FadeCache(self.cfg, self.L, self.maxP, self.max_pos, device)
        self.params = dataclasses.replace(Params.from_workload(wl), v_codec=v_codec)
        self.codebook = None
        if v_codec == "pq":
            # a codebook made of 256 V-like draws (centroid c of sub-space s = channels
            # 4s..4s+3 of draw c), the same array on both sides
            d = wl.head_dim
            rows = pq_calibration(wl, 256)
            self.codebook = np.ascontiguousarray(rows.reshape(256, d // 4, 4).transpose(1, 0, 2))
            self.fc.set_pq_codebook(torch.from_numpy(self.codebook).to(self.fc.device))
        self.rope = RopeTable.from_workload(wl, self.max_pos)
        B, H = wl.batch, wl.num_kv_heads
        self.units = [[[UnitCache(self.params, self.rope, codebook=self.codebook)
                        for _ in range(H)] for _ in range(B)] for _ in range(self.L)]
        self.near_ties = 0               # unit-steps whose fp64 selection differed at a near-tie
        self.unit_steps = 0              # (layer, row, KV head) decode steps compared
        self.prefill_near_ties = 0       # GPU-mass prefills whose fp64 selection differed
        self.step_index = 0

    # -------------------------------------------------------------------- prefill
    def prefill_mass32(self, pr, b, h):
        """fp32 H2O prefill mass of unit (b, h), computed by the oracle."""
        wl, G, P = self.wl, self.wl.group, int(self.lens[b])
        pos = np.arange(P)
        q = np.stack([self.rope.apply(pr["q"][b, h * G + g, :P], pos) for g in range(G)])
        k = self.rope.apply(pr["k"][b, h, :P], pos)
        return attention.prefill_mass(q.astype(np.float64), k.astype(np.float64)).astype(np.float32)

    def prefill(self, layer, gpu_mass=False):
        """Prefill one layer on both sides. gpu_mass (H2O): the GPU computes the prefill mass
        itself (the product path) instead of taking the oracle's; see _prefill_gpu_mass."""
        torch = self.torch
        wl = self.wl
        h2o = wl.policy == "h2o" and wl.int4_budget >= 0
        pr = draw_prompt(wl, layer, self.maxP, with_q=h2o)
        if gpu_mass and h2o:
            return self._prefill_gpu_mass(layer, pr)
        mass = None
        if h2o:
            mass = np.zeros((wl.batch, wl.num_kv_heads, self.maxP), np.float32)
            for b in range(wl.batch):
                for h in range(wl.num_kv_heads):
                    mass[b, h, :self.lens[b]] = self.prefill_mass32(pr, b, h)
        dev = self.fc.device
        k = torch.from_numpy(pr["k"]).to(dev)
        v = torch.from_numpy(pr["v"]).to(dev)
        md = torch.from_numpy(mass).to(dev) if mass is not None else None
        self.fc.prefill(layer, k, v, self.lens, md)
        sel = None
        if mass is not None and self.shared:  # rows sharing decisions select by the row sum
            sel = mass.astype(np.float64).sum(axis=0)
        for b in range(wl.batch):
            P = int(self.lens[b])
            for h in range(wl.num_kv_heads):
                u = self.units[layer][b][h]
                u.prefill(pr["k"][b, h, :P], pr["v"][b, h, :P],
                          mass=None if mass is None else mass[b, h, :P].astype(np.float64),
                          select_mass=None if sel is None else sel[h, :P])

    def _prefill_gpu_mass(self, layer, pr):
        """H2O prefill with the mass computed on the GPU (fade_prefill_mass) and used there.
        Checks: the GPU mass is within 1e-5 + 1e-4|ref| of the oracle's fp64 mass, a second
        computation gives the same bits, the oracle's selection rule applied to the GPU's fp32
        mass picks the GPU's victims (the whole prefilled state is then compared bit for bit),
        and the rule applied to the oracle's own mass picks the same victims except at fp32
        near-ties (counted in prefill_near_ties). The oracle's scores start from its own
        mass."""
        from oracle import policy as pol
        from tiered_mixed_precision_gb300 import fade as F

        torch, wl = self.torch, self.wl
        assert not self.shared, "rows sharing decisions: use the oracle's mass"
        dev = self.fc.device
        k = torch.from_numpy(pr["k"]).to(dev)
        v = torch.from_numpy(pr["v"]).to(dev)
        q = torch.from_numpy(pr["q"]).to(dev)
        mass_d = self.fc.prefill(layer, k, v, self.lens, None, q_raw=q)
        again = torch.full_like(mass_d, float("nan"))
        F.fade_prefill_mass(self.cfg, q, k, self.maxP, self.lens, again)  # q, k now rotated
        g32 = mass_d.cpu().numpy()
        assert np.array_equal(again.cpu().numpy().view(np.uint32), g32.view(np.uint32)), \
            "prefill mass differs between two runs"
        n_s, W, budget = wl.n_sink, wl.recent_window, wl.int4_budget
        for b in range(wl.batch):
            P = int(self.lens[b])
            for h in range(wl.num_kv_heads):
                m64 = self.prefill_mass32(pr, b, h).astype(np.float64)
                ok, err, nbad = allclose_report(g32[b, h, :P], m64, atol=1e-5, rtol=1e-4)
                assert ok, f"prefill mass of {(layer, b, h)}: max err {err}, {nbad} bad"
                ns = min(n_s, P)
                n_m = P - ns - min(W, P - ns)
                if n_m > budget:
                    cand = slice(ns, ns + n_m)
                    mine = pol.select_victims(m64[cand], n_m - budget)
                    gpu = pol.select_victims(g32[b, h, cand].astype(np.float64), n_m - budget)
                    if not np.array_equal(mine, gpu):
                        a, g = np.sort(m64[cand][mine]), np.sort(m64[cand][gpu])
                        assert np.allclose(a, g, rtol=TIE_RTOL, atol=1e-6), (
                            f"prefill selection differs beyond a near-tie at {(layer, b, h)}")
                        self.prefill_near_ties += 1
                u = self.units[layer][b][h]
                u.prefill(pr["k"][b, h, :P], pr["v"][b, h, :P], mass=m64,
                          select_mass=g32[b, h, :P].astype(np.float64))

    # -------------------------------------------------------------------- decode
    def step(self, check_state=True, evict=True):
        """One decode step of every layer; returns the max attention error seen. evict=False
        leaves out the eviction call on both sides (the middle tier then grows past its budget
        and a later step evicts every pending token at once)."""
        torch = self.torch
        wl, G = self.wl, self.wl.group
        if evict:
            pos = self.fc.next_positions()
            for b in range(wl.batch):
                want = self.units[0][b][0].next_position()
                assert pos[b] == want, f"row {b}: next position {pos[b]} != oracle {want}"
        else:  # no eviction: the new token's position is the number of tokens held
            L0 = self.fc.layers[0]
            pos = (L0.h_n_sink + L0.h_n_mid + L0.h_n_recent).astype(np.int32)
            for b in range(wl.batch):
                want = self.units[0][b][0].n_held
                assert pos[b] == want, f"row {b}: held {pos[b]} != oracle {want}"
        self.fc.set_positions(pos)
        worst = 0.0
        for layer in range(self.L):
            t = draw_decode_tokens(wl, layer, self.step_index)
            dev = self.fc.device
            q = torch.from_numpy(t["q"].copy()).to(dev)
            k = torch.from_numpy(t["k"].copy()).to(dev)
            v = torch.from_numpy(t["v"].copy()).to(dev)
            out = torch.empty_like(q)
            if evict:
                self.fc.step_layer(layer, q, k, v, out)
            else:
                from tiered_mixed_precision_gb300 import fade as F
                F.fade_cache_demote(self.fc.layers[layer])
                self.fc.attend_layer(layer, q, k, v, out)
            victims_gpu = self._gpu_victims(layer)
            if evict and wl.policy in ("h2o", "ema"):
                self._replay_selection(layer, victims_gpu)
            out_h = out.float().cpu().numpy()
            shared_vic = {}
            if self.shared and evict:
                for h in range(wl.num_kv_heads):
                    shared_vic[h] = self._shared_victims(layer, h, victims_gpu)
            for b in range(wl.batch):
                for h in range(wl.num_kv_heads):
                    key = (layer, b, h)
                    u = self.units[layer][b][h]
                    o_ref, tie = self._oracle_step(u, t, b, h, victims_gpu, key, evict,
                                                   shared_vic.get(h))
                    self.unit_steps += 1
                    ok, err, nbad = allclose_report(out_h[b, h * G:(h + 1) * G], o_ref)
                    worst = max(worst, err)
                    assert ok, (f"attention mismatch at step {self.step_index} layer {layer} "
                                f"row {b} head {h}: max err {err}, {nbad} bad")
            if check_state:
                self.check_layer_state(layer)
        self.step_index += 1
        return worst

    def _replay_selection(self, layer, bm):
        """Selection replay: the selection rule (smallest key, lower index first on ties; the
        oracle's) applied to the very fp32 keys the GPU compared must give the GPU's victims
        bit for bit. The keys are the middle scores in the buffer the step compacted from
        (eviction writes the survivors to the other buffer); rows sharing their decisions
        compare the fp32 sum over the rows in ascending row order."""
        from oracle import policy as pol

        L = self.fc.layers[layer]
        meta = L.meta.cpu().numpy()
        scores = [t.cpu().numpy() for t in L.mid_scores]   # both ping-pong buffers
        wl = self.wl
        for h in range(wl.num_kv_heads):
            rows = []
            for b in range(wl.batch):
                u = self.units[layer][b][h]   # oracle state before this step
                n_mid = u.n_mid + (1 if u._ring_full() else 0)
                k = n_mid - u.p.int4_budget if u.p.evicts else 0
                if k <= 0:
                    continue
                prev = 1 - int(meta[b, h, 4])   # the buffer the selection read
                keys = scores[prev][b, h, :n_mid].astype(np.float32)
                words = bm[b, h, :(n_mid + 31) // 32]
                gpu = np.nonzero(np.unpackbits(words.view(np.uint8), bitorder="little")[:n_mid])[0]
                rows.append((b, keys, k, gpu))
            if not rows:
                continue
            if self.shared:
                total = rows[0][1].copy()
                for _, keys, _, _ in rows[1:]:
                    total = (total + keys).astype(np.float32)
                want = np.sort(pol.select_victims(total.astype(np.float64), rows[0][2]))
                for b, _, _, gpu in rows:
                    assert np.array_equal(gpu, want), f"shared selection replay at {layer, b, h}"
            else:
                for b, keys, k, gpu in rows:
                    want = np.sort(pol.select_victims(keys.astype(np.float64), k))
                    assert np.array_equal(gpu, want), (
                        f"selection replay differs at layer {layer} row {b} head {h}: "
                        f"gpu {gpu}, rule on the gpu keys {want}")

    def _gpu_victims(self, layer):
        """Victim middle indices chosen by the CUDA path in this step (per unit), read from
        its selection bitmap, or None for units without an eviction."""
        return self.fc.layers[layer].victims.cpu().numpy().view(np.uint32)

    def _shared_victims(self, layer, h, bm):
        """Rows sharing their decisions: demote every row of (layer, h), choose the victims
        once by the row-summed scores, check that the GPU gave every row the same set and that
        it equals this one (up to an fp32-vs-fp64 near-tie, which the oracle then adopts)."""
        from oracle.cache import choose_shared_victims

        units = [self.units[layer][b][h] for b in range(self.wl.batch)]
        for u in units:
            u.demote()
        vic = choose_shared_victims(units)
        n_mid = units[0].n_mid
        if vic.size == 0 or self.wl.policy == "position":  # no bitmap: the oldest go
            return vic
        words = [bm[b, h, :(n_mid + 31) // 32] for b in range(self.wl.batch)]
        assert all(np.array_equal(w, words[0]) for w in words), "rows got different victims"
        bits = np.unpackbits(words[0].view(np.uint8), bitorder="little")[:n_mid]
        gpu_vic = np.nonzero(bits)[0]
        if not np.array_equal(np.sort(gpu_vic), np.sort(vic)):
            s0 = units[0].n_sink
            keys = np.sum([u.sigma[s0:s0 + n_mid] for u in units], axis=0)
            a, g = np.sort(keys[vic]), np.sort(keys[gpu_vic])
            assert gpu_vic.size == vic.size and np.allclose(a, g, rtol=TIE_RTOL, atol=1e-7), (
                f"shared selection differs beyond a near-tie at layer {layer} head {h}")
            self.near_ties += 1
            vic = gpu_vic
        return vic

    def _oracle_step(self, u, t, b, h, bm, key, evict=True, shared_vic=None):
        G = self.wl.group
        if shared_vic is not None:  # demoted and chosen for all rows by _shared_victims
            u.evict(shared_vic)
            pos = u.n_held
            u.append(u.rope.apply(t["k"][b, h][None], pos), t["v"][b, h])
            out, p, _ = u.attend(u.rope.apply(t["q"][b, h * G:(h + 1) * G], pos))
            u.accumulate(p)
            return out, False
        out, tie = oracle_unit_step(u, t, b, h, G, self.wl.policy, bm[b, h], evict)
        self.near_ties += tie
        return out, tie

    def check_near_ties(self, frac=0.01, floor=1):
        """Print how many unit-steps were compared and how many took the GPU's victims at
        a near-tie; the latter must stay within ``frac`` of the former (at least ``floor``)."""
        print(f"lockstep {self.wl.name}: {self.unit_steps} unit-steps compared, "
              f"{self.near_ties} near-tie selections adopted")
        assert self.near_ties <= max(floor, frac * self.unit_steps), (
            f"{self.near_ties} near-ties in {self.unit_steps} unit-steps")

    # -------------------------------------------------------------------- state
    def check_layer_state(self, layer):
        wl = self.wl
        for b in range(wl.batch):
            for h in range(wl.num_kv_heads):
                self.check_unit_state(layer, b, h)

    def check_unit_state(self, layer, b, h):
        compare_unit_state(self.fc.unit_state(layer, b, h), self.units[layer][b][h],
                           f"layer {layer} row {b} head {h} step {self.step_index}")
