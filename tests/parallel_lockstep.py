"""Lockstep at a workload's stated size: the CUDA path steps every layer of the full workload
(all rows and KV heads) exactly as in ``harness.Lockstep``, while the oracle's units are
spread over worker processes (one per host core, started with ``spawn``), each holding its
share of the (layer, row, KV head) units for the whole run.

Per decode step the main process runs every layer on the GPU, replays each H2O / EMA
selection on the GPU's own fp32 keys (the selection rule must give the GPU's victims bit for
bit), and sends every worker its units' attention outputs and selection bitmaps; the workers
step their oracle units (adopting the GPU's victims at an fp32-vs-fp64 near-tie, R10) and
compare the outputs within 2e-3 + 1e-2|ref|. Every ``check_every`` steps and after the last
one the whole cache of every layer is copied to the host and each worker compares its units'
tiers bit for bit (scores within the tolerance). Units may be a sample (``units``) when the
workload's rows are too long for the oracle to step every unit.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import sys

import numpy as np

from harness import TIE_RTOL, allclose_report, compare_unit_state, oracle_unit_step


# ------------------------------------------------------------------------------ worker side
def _worker(conn, paths, wl, units, max_pos):
    sys.path[:0] = paths
    from oracle.cache import Params, UnitCache
    from oracle.rope import RopeTable
    from synth import draw_decode_tokens
    from oracle import attention, policy as pol

    rope = RopeTable.from_workload(wl, max_pos)
    params = Params.from_workload(wl)
    caches = {key: UnitCache(params, rope) for key in units}
    G = wl.group
    h2o = wl.policy == "h2o" and wl.int4_budget >= 0
    try:
        while True:
            cmd, arg = conn.recv()
            if cmd == "close":
                conn.send(("ok", None))
                return
            if cmd == "prefill":   # arg: {key: (raw k [P][d], v, q [G][P][d] or None, mass)}
                ties = 0
                for key, (kr, vr, qr, g32) in arg.items():
                    P = kr.shape[0]
                    mass = sel = None
                    if h2o:
                        pos = np.arange(P)
                        q = np.stack([rope.apply(qr[g], pos) for g in range(G)])
                        k = rope.apply(kr, pos)
                        mass = attention.prefill_mass(q.astype(np.float64), k.astype(np.float64))
                        ok, err, nbad = allclose_report(g32, mass, atol=1e-5, rtol=1e-4)
                        assert ok, f"prefill mass of {key}: max err {err}, {nbad} bad"
                        sel = g32.astype(np.float64)
                        n_s = min(wl.n_sink, P)
                        n_m = P - n_s - min(wl.recent_window, P - n_s)
                        if n_m > wl.int4_budget:
                            c = slice(n_s, n_s + n_m)
                            mine_v = pol.select_victims(mass[c], n_m - wl.int4_budget)
                            gpu_v = pol.select_victims(sel[c], n_m - wl.int4_budget)
                            if not np.array_equal(mine_v, gpu_v):
                                a, g = np.sort(mass[c][mine_v]), np.sort(mass[c][gpu_v])
                                assert np.allclose(a, g, rtol=TIE_RTOL, atol=1e-6), (
                                    f"prefill selection differs beyond a near-tie at {key}")
                                ties += 1
                    caches[key].prefill(kr, vr, mass=mass, select_mass=sel)
                conn.send(("ok", ties))
            elif cmd == "step":    # arg: step index, positions, {key: (out [G][d], bitmap)}
                step, pos, data = arg
                worst, ties, n = 0.0, 0, 0
                cache_t = {}
                for key, (out, words) in data.items():
                    layer, b, h = key
                    u = caches[key]
                    want = u.next_position()
                    assert pos[b] == want, f"{key}: next position {pos[b]} != oracle {want}"
                    if layer not in cache_t:
                        cache_t[layer] = draw_decode_tokens(wl, layer, step)
                    ref, tie = oracle_unit_step(u, cache_t[layer], b, h, G, wl.policy, words)
                    ok, err, nbad = allclose_report(out, ref)
                    assert ok, (f"attention mismatch at step {step} unit {key}: max err {err}, "
                                f"{nbad} bad")
                    worst = max(worst, err)
                    ties += tie
                    n += 1
                conn.send(("ok", (worst, ties, n)))
            elif cmd == "state":   # arg: step index, {key: GPU unit state}
                step, states = arg
                for key, g in states.items():
                    compare_unit_state(g, caches[key], f"unit {key} after step {step}")
                conn.send(("ok", len(states)))
    except BaseException as e:  # report to the main process, which raises it
        import traceback

        conn.send(("error", f"{type(e).__name__}: {e}\n{traceback.format_exc()}"))


# ------------------------------------------------------------------------------ main side
def _layer_host(fc, layer):
    """Every buffer of a layer copied to the host once (numpy)."""
    L = fc.layers[layer]
    g = lambda t: t.cpu().numpy()
    return {"meta": g(L.meta), "sink_k": g(L.sink_k), "sink_v": g(L.sink_v),
            "recent_k": g(L.recent_k), "recent_v": g(L.recent_v),
            "mid_k_codes": [g(t) for t in L.mid_k_codes],
            "mid_k_scales": [g(t) for t in L.mid_k_scales],
            "mid_v_codes": [g(t) for t in L.mid_v_codes],
            "mid_v_scales": [g(t) for t in L.mid_v_scales],
            "sink_scores": g(L.sink_scores), "mid_scores": [g(t) for t in L.mid_scores],
            "recent_scores": g(L.recent_scores)}


def _unit_from_host(H, b, h, W):
    """One unit's tiers in cache order from a host copy of its layer."""
    m = H["meta"][b, h]
    n_sink, n_mid, n_rec, head, cur = (int(m[i]) for i in range(5))
    ring = [(head + i) % W for i in range(n_rec)]
    return {
        "n_sink": n_sink, "n_mid": n_mid, "n_recent": n_rec,
        "sink_k": H["sink_k"][b, h, :n_sink], "sink_v": H["sink_v"][b, h, :n_sink],
        "mid_k_codes": H["mid_k_codes"][cur][b, h, :n_mid],
        "mid_k_scales": H["mid_k_scales"][cur][b, h, :n_mid],
        "mid_v_codes": H["mid_v_codes"][cur][b, h, :n_mid],
        "mid_v_scales": H["mid_v_scales"][cur][b, h, :n_mid],
        "recent_k": H["recent_k"][b, h, ring], "recent_v": H["recent_v"][b, h, ring],
        "scores": np.concatenate([H["sink_scores"][b, h, :n_sink],
                                  H["mid_scores"][cur][b, h, :n_mid],
                                  H["recent_scores"][b, h, ring]]),
    }


class ParallelLockstep:
    """Full-size lockstep with the oracle's units in worker processes."""

    def __init__(self, wl, steps=None, units=None, workers=None, device="cuda"):
        import torch

        from synth import ragged_context_lengths
        from tiered_mixed_precision_gb300 import Config
        from tiered_mixed_precision_gb300.model import FadeCache

        self.torch = torch
        self.wl = wl
        self.steps = wl.steps if steps is None else steps
        self.lens = ragged_context_lengths(wl)
        self.maxP = int(self.lens.max())
        self.max_pos = self.maxP + self.steps + 8
        self.cfg = Config.from_workload(wl)
        self.fc = FadeCache(self.cfg, wl.layers, self.maxP, self.max_pos, device)
        if units is None:
            units = [(l, b, h) for l in range(wl.layers) for b in range(wl.batch)
                     for h in range(wl.num_kv_heads)]
        self.units = list(units)
        n = max(1, min(workers or os.cpu_count() or 1, len(self.units)))
        shares = [self.units[i::n] for i in range(n)]
        ctx = mp.get_context("spawn")
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        paths = [root, os.path.join(root, "tests")]
        self.conns, self.procs, self.owner = [], [], {}
        # one process per core, each single-threaded (a spawned child reads these at start)
        threads = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in threads}
        os.environ.update({k: "1" for k in threads})
        try:
            for i, share in enumerate(shares):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_worker, args=(b, paths, wl, share, self.max_pos),
                                daemon=True)
                p.start()
                self.conns.append(a)
                self.procs.append(p)
                for key in share:
                    self.owner[key] = i
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.step_index = 0
        self.unit_steps = 0
        self.near_ties = 0
        self.prefill_near_ties = 0
        self.worst = 0.0

    # -------------------------------------------------------------------- plumbing
    def _all(self, msgs):
        """Send msgs[i] to worker i (None: nothing) and gather the replies."""
        for c, m in zip(self.conns, msgs):
            if m is not None:
                c.send(m)
        out = []
        for c, m in zip(self.conns, msgs):
            if m is None:
                out.append(None)
                continue
            tag, val = c.recv()
            if tag == "error":
                self.close()
                raise AssertionError(f"oracle worker failed:\n{val}")
            out.append(val)
        return out

    def close(self):
        for c in self.conns:
            try:
                c.send(("close", None))
                c.recv()
            except (EOFError, OSError, BrokenPipeError):
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()

    # -------------------------------------------------------------------- prefill
    def prefill(self):
        """Every layer's prompt (seeded numpy draws, the same arrays on both sides) on the GPU
        (H2O: the GPU computes the prefill mass and evicts by it, the product path); each
        worker gets its units' rows and prefills its oracle units."""
        from synth import draw_prompt

        torch, wl, G = self.torch, self.wl, self.wl.group
        h2o = wl.policy == "h2o" and wl.int4_budget >= 0
        dev = self.fc.device
        for layer in range(wl.layers):
            pr = draw_prompt(wl, layer, self.maxP, with_q=h2o)
            k = torch.from_numpy(pr["k"]).to(dev)
            v = torch.from_numpy(pr["v"]).to(dev)
            q = torch.from_numpy(pr["q"]).to(dev) if h2o else None
            mass = self.fc.prefill(layer, k, v, self.lens, None, q_raw=q)
            g32 = mass.cpu().numpy() if mass is not None else None
            del k, v, q
            msgs = [dict() for _ in self.conns]
            for key in self.units:
                if key[0] == layer:
                    _, b, h = key
                    P = int(self.lens[b])
                    msgs[self.owner[key]][key] = (
                        pr["k"][b, h, :P].copy(), pr["v"][b, h, :P].copy(),
                        pr["q"][b, h * G:(h + 1) * G, :P].copy() if h2o else None,
                        None if g32 is None else g32[b, h, :P].copy())
            del pr
            replies = self._all([("prefill", m) if m else None for m in msgs])
            self.prefill_near_ties += sum(r for r in replies if r)
        self.check_state()

    # -------------------------------------------------------------------- decode
    def _replay(self, layer, n_mid_pre, words):
        """The selection rule on the very fp32 keys the GPU compared must give its victims."""
        from oracle import policy as pol

        L = self.fc.layers[layer]
        meta = L.meta.cpu().numpy()
        scores = [t.cpu().numpy() for t in L.mid_scores]
        wl = self.wl
        for b in range(wl.batch):
            k = int(n_mid_pre[b]) - wl.int4_budget
            if k <= 0:
                continue
            n = int(n_mid_pre[b])
            for h in range(wl.num_kv_heads):
                keys = scores[1 - int(meta[b, h, 4])][b, h, :n].astype(np.float64)
                want = np.sort(pol.select_victims(keys, k))
                got = np.sort(np.nonzero(np.unpackbits(
                    np.ascontiguousarray(words[b, h, :(n + 31) // 32]).view(np.uint8),
                    bitorder="little")[:n])[0])
                assert np.array_equal(got, want), (
                    f"selection replay differs at layer {layer} row {b} head {h}")

    def step(self):
        from synth import draw_decode_tokens

        torch, wl, G = self.torch, self.wl, self.wl.group
        pos = self.fc.next_positions()
        self.fc.set_positions(pos)
        dev = self.fc.device
        msgs = [dict() for _ in self.conns]
        for layer in range(wl.layers):
            L = self.fc.layers[layer]
            n_mid_pre = L.h_n_mid + (L.h_n_recent == wl.recent_window)
            t = draw_decode_tokens(wl, layer, self.step_index)
            q, k, v = (torch.from_numpy(t[x].copy()).to(dev) for x in ("q", "k", "v"))
            out = torch.empty_like(q)
            self.fc.step_layer(layer, q, k, v, out)
            words = L.victims.cpu().numpy().view(np.uint32)
            if wl.policy in ("h2o", "ema") and wl.int4_budget >= 0:
                self._replay(layer, n_mid_pre, words)
            out_h = out.float().cpu().numpy()
            for key in self.units:
                if key[0] == layer:
                    _, b, h = key
                    msgs[self.owner[key]][key] = (out_h[b, h * G:(h + 1) * G].copy(),
                                                  words[b, h].copy())
        replies = self._all([("step", (self.step_index, pos, m)) if m else None for m in msgs])
        for worst, ties, n in (r for r in replies if r is not None):
            self.worst = max(self.worst, worst)
            self.near_ties += ties
            self.unit_steps += n
        self.step_index += 1

    def check_state(self):
        W = self.wl.recent_window
        msgs = [dict() for _ in self.conns]
        for layer in range(self.wl.layers):
            keys = [key for key in self.units if key[0] == layer]
            if len(keys) > 8:   # most of the layer: one copy of every buffer
                H = _layer_host(self.fc, layer)
                for key in keys:
                    msgs[self.owner[key]][key] = _unit_from_host(H, key[1], key[2], W)
                del H
            else:               # a sample: only those units' rows
                for key in keys:
                    msgs[self.owner[key]][key] = self.fc.unit_state(*key)
        self._all([("state", (self.step_index, m)) if m else None for m in msgs])

    def run(self, check_every=64):
        self.prefill()
        for s in range(self.steps):
            self.step()
            if (s + 1) % check_every == 0 or s + 1 == self.steps:
                self.check_state()
        self.torch.cuda.synchronize()
        for L in self.fc.layers:
            assert int(L.status.abs().sum()) == 0, "a kernel gave up a bounded wait"
        print(f"full-size lockstep {self.wl.name}: {len(self.units)} units x {self.steps} steps, "
              f"{self.unit_steps} unit-steps compared, {self.near_ties} near-tie selections "
              f"adopted, {self.prefill_near_ties} prefill near-ties, max |attention error| "
              f"{self.worst:.2e}")
        self.close()
        assert self.near_ties <= max(1, 0.01 * self.unit_steps)
        assert self.prefill_near_ties <= max(1, 0.01 * len(self.units))
