"""Parity at the full per-layer sizes of the throughput workloads, in the launch configuration
the benchmark times (full batch, heads and context of one layer): sampled (row, KV head)
units are replayed by the oracle from the same raw draws and compared after prefill and after
each of 16 decode steps (every step evicts and re-positions the whole middle tier)."""

import numpy as np
import pytest

from harness import allclose_report
from oracle import quant
from oracle.cache import Params, UnitCache
from oracle.rope import RopeTable
from synth import draw_prompt, draw_vectors, get_workload, ragged_context_lengths

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _compare_unit(fc, u, b, h, where):
    g = fc.unit_state(0, b, h)
    assert (g["n_sink"], g["n_mid"], g["n_recent"]) == (u.n_sink, u.n_mid, u.n_recent), where
    eq16 = lambda a, r: np.array_equal(np.asarray(a).view(np.uint16), np.asarray(r).view(np.uint16))
    assert eq16(g["sink_k"], u.sink_k) and eq16(g["recent_k"], u.rec_k), f"fp16 K differs {where}"
    assert eq16(g["sink_v"], u.sink_v) and eq16(g["recent_v"], u.rec_v), f"fp16 V differs {where}"
    assert np.array_equal(g["mid_k_codes"], quant.pack(u.mid_kq, u.p.k_bits)), f"K codes {where}"
    assert np.array_equal(g["mid_v_codes"], quant.pack(u.mid_vq, u.p.v_bits)), f"V codes {where}"
    assert eq16(g["mid_k_scales"], u.mid_ks) and eq16(g["mid_v_scales"], u.mid_vs), where
    if u.p.policy in ("h2o", "ema"):
        ok, err, _ = allclose_report(g["scores"], u.sigma)
        assert ok, f"scores differ {where}: {err}"


@pytest.mark.parametrize("key", [4, 5])
def test_full_size_layer_sampled_units(key):
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    wl = get_workload(key)
    steps = 16
    cfg = T.Config.from_workload(wl)
    lens = ragged_context_lengths(wl)
    maxP = int(lens.max())
    max_pos = maxP + steps + 16
    dev = torch.device("cuda")
    fc = FadeCache(cfg, 1, maxP, max_pos, dev)
    pr = draw_prompt(wl, 0, maxP, backend="torch", device=dev)
    rng = np.random.default_rng(key)
    sample = sorted({(int(rng.integers(wl.batch)), int(rng.integers(wl.num_kv_heads)))
                     for _ in range(4)} | {(wl.batch - 1, wl.num_kv_heads - 1)})
    raw = {(b, h): (pr["k"][b, h, :lens[b]].cpu().numpy(), pr["v"][b, h, :lens[b]].cpu().numpy())
           for b, h in sample}
    fc.prefill(0, pr["k"], pr["v"], lens, None)
    del pr
    rope = RopeTable.from_workload(wl, max_pos)
    units = {}
    for (b, h), (k, v) in raw.items():
        u = UnitCache(Params.from_workload(wl), rope)
        u.prefill(k, v)
        units[(b, h)] = u
        _compare_unit(fc, u, b, h, f"after prefill, unit {(b, h)}")
    G, d = wl.group, wl.head_dim
    out = torch.empty((wl.batch, wl.num_q_heads, d), dtype=torch.float16, device=dev)
    for step in range(steps):
        q = draw_vectors(wl, "q", (wl.batch, wl.num_q_heads, d), "full", step, backend="torch", device=dev)
        k = draw_vectors(wl, "k", (wl.batch, wl.num_kv_heads, d), "full", step, backend="torch", device=dev)
        v = draw_vectors(wl, "v", (wl.batch, wl.num_kv_heads, d), "full", step, backend="torch", device=dev)
        fc.set_positions(fc.next_positions())
        fc.step_layer(0, q, k, v, out)
        oh = out.float().cpu().numpy()
        qh, kh, vh = q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy()
        for (b, h), u in units.items():
            o_ref, _, _, _ = u.step(qh[b, h * G:(h + 1) * G], kh[b, h], vh[b, h])
            ok, err, nbad = allclose_report(oh[b, h * G:(h + 1) * G], o_ref)
            assert ok, f"step {step} unit {(b, h)}: max err {err}, {nbad} bad"
            _compare_unit(fc, u, b, h, f"after step {step}, unit {(b, h)}")
    torch.cuda.synchronize()
    assert int(fc.layers[0].status.abs().sum()) == 0


@pytest.mark.parametrize("key", [4, 5])
def test_full_size_pipelined_graph_sampled_units(key):
    """The benchmark's own launch configuration at full layer size: the pipelined step (each
    layer's maintenance for the next step on side streams) captured once as a CUDA graph and
    replayed. The oracle follows the same order: maintenance first (demote, evict), then per
    step append, attention, accumulation and the next step's maintenance."""
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    wl = get_workload(key)
    steps = 16
    cfg = T.Config.from_workload(wl)
    lens = ragged_context_lengths(wl)
    maxP = int(lens.max())
    max_pos = maxP + steps + 16
    dev = torch.device("cuda")
    fc = FadeCache(cfg, 1, maxP, max_pos, dev)
    pr = draw_prompt(wl, 0, maxP, backend="torch", device=dev)
    rng = np.random.default_rng(100 + key)
    sample = sorted({(int(rng.integers(wl.batch)), int(rng.integers(wl.num_kv_heads)))
                     for _ in range(4)} | {(0, 0)})
    raw = {(b, h): (pr["k"][b, h, :lens[b]].cpu().numpy(), pr["v"][b, h, :lens[b]].cpu().numpy())
           for b, h in sample}
    fc.prefill(0, pr["k"], pr["v"], lens, None)
    del pr
    rope = RopeTable.from_workload(wl, max_pos)
    units = {}
    for (b, h), (k, v) in raw.items():
        u = UnitCache(Params.from_workload(wl), rope)
        u.prefill(k, v)
        u.demote()                      # the prologue's maintenance
        u.evict(u.choose_victims())
        units[(b, h)] = u
    G, d = wl.group, wl.head_dim
    q = [draw_vectors(wl, "q", (1, wl.batch, wl.num_q_heads, d), "pipe", s, backend="torch",
                      device=dev) for s in range(steps)]
    k = [draw_vectors(wl, "k", (1, wl.batch, wl.num_kv_heads, d), "pipe", s, backend="torch",
                      device=dev) for s in range(steps)]
    v = [draw_vectors(wl, "v", (1, wl.batch, wl.num_kv_heads, d), "pipe", s, backend="torch",
                      device=dev) for s in range(steps)]
    out = torch.empty((1, wl.batch, wl.num_q_heads, d), dtype=torch.float16, device=dev)
    side = [torch.cuda.Stream(), torch.cuda.Stream()]
    fc.maintain_all()
    qb, kb, vb = q[0].clone(), k[0].clone(), v[0].clone()
    graph = fc.capture_step(qb, kb, vb, out, side)
    for step in range(steps):
        qb.copy_(q[step])
        kb.copy_(k[step])
        vb.copy_(v[step])
        graph.replay()
        torch.cuda.synchronize()
        oh = out[0].float().cpu().numpy()
        qh, kh, vh = q[step][0].cpu().numpy(), k[step][0].cpu().numpy(), v[step][0].cpu().numpy()
        for (b, h), u in units.items():
            pos = u.n_held
            u.append(rope.apply(kh[b, h][None], pos), vh[b, h])
            o_ref, p, _ = u.attend(rope.apply(qh[b, h * G:(h + 1) * G], pos))
            u.accumulate(p)
            ok, err, nbad = allclose_report(oh[b, h * G:(h + 1) * G], o_ref)
            assert ok, f"step {step} unit {(b, h)}: max err {err}, {nbad} bad"
            u.demote()                  # the next step's maintenance, as the graph did
            u.evict(u.choose_victims())
            _compare_unit(fc, u, b, h, f"after pipelined step {step}, unit {(b, h)}")
    assert int(fc.layers[0].status.abs().sum()) == 0
