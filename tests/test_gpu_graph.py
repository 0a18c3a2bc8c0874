"""A decode step captured once as a CUDA graph and replayed gives, step after step, the same
bytes as launching every call (steady state: the cache sits at its budget, so each step
demotes one token, evicts one and appends one)."""

import numpy as np
import pytest

from synth import draw_prompt, draw_vectors, get_workload
from synth.draws import pq_calibration

pytestmark = pytest.mark.gpu


def _masses(wl):
    """H2O prefill masses computed once on the GPU and given to both caches of a comparison."""
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    if wl.policy != "h2o":
        return [None] * wl.layers
    cfg = T.Config.from_workload(wl)
    fc = FadeCache(cfg, 1, wl.prompt_len, wl.prompt_len + 64, "cuda")
    B, P = wl.batch, wl.prompt_len
    out = []
    for layer in range(wl.layers):
        pr = draw_prompt(wl, layer, with_q=True)
        q = torch.from_numpy(pr["q"]).cuda()
        k = torch.from_numpy(pr["k"]).cuda()
        fc.rope_(q, B * wl.num_q_heads, P, None, 1)
        fc.rope_(k, B * wl.num_kv_heads, P, None, 1)
        m = torch.empty((B, wl.num_kv_heads, P), dtype=torch.float32, device="cuda")
        T.fade_prefill_mass(cfg, q, k, P, np.full(B, P, np.int32), m)
        out.append(m)
    return out


def _make(wl, masses, v_codec="int"):
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    cfg = T.Config.from_workload(wl)
    cfg.v_codec = v_codec
    fc = FadeCache(cfg, wl.layers, wl.prompt_len, wl.prompt_len + 64, "cuda")
    if v_codec == "pq":   # a codebook made of 256 V-like draws
        rows = pq_calibration(wl, 256)
        cb = rows.reshape(256, wl.head_dim // 4, 4).transpose(1, 0, 2).copy()
        fc.set_pq_codebook(torch.from_numpy(cb).cuda())
    for layer in range(wl.layers):
        pr = draw_prompt(wl, layer)
        fc.prefill(layer, torch.from_numpy(pr["k"]).cuda(), torch.from_numpy(pr["v"]).cuda(),
                   mass=masses[layer])
    return fc


@pytest.mark.parametrize("policy", ["position", "h2o"])
def test_graph_replay_matches_eager_steps(policy):
    import torch

    wl = get_workload(4).scaled(layers=2, batch=2, num_q_heads=8, num_kv_heads=2,
                                prompt_len=1200, int4_budget=500, policy=policy)
    if policy == "h2o":
        wl = wl.scaled(rope=get_workload(3).rope)
    masses = _masses(wl)
    eager, graphed = _make(wl, masses), _make(wl, masses)
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    steps = 4
    q = torch.from_numpy(draw_vectors(wl, "q", (steps, L, B, Hq, d), "graph")).cuda()
    k = torch.from_numpy(draw_vectors(wl, "k", (steps, L, B, Hkv, d), "graph")).cuda()
    v = torch.from_numpy(draw_vectors(wl, "v", (steps, L, B, Hkv, d), "graph")).cuda()
    out_e = torch.empty((L, B, Hq, d), dtype=torch.float16, device="cuda")
    out_g = torch.empty_like(out_e)
    qb, kb, vb = q[0].clone(), k[0].clone(), v[0].clone()
    g = graphed.capture_step(qb, kb, vb, out_g)
    for s in range(steps):
        eager.step_all(q[s], k[s], v[s], out_e)
        qb.copy_(q[s])
        kb.copy_(k[s])
        vb.copy_(v[s])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_e.view(torch.int16), out_g.view(torch.int16)), f"step {s}"
    for layer in range(L):
        for b in range(B):
            for h in range(Hkv):
                a_, b_ = eager.unit_state(layer, b, h), graphed.unit_state(layer, b, h)
                for key in a_:
                    if isinstance(a_[key], np.ndarray):
                        assert np.array_equal(a_[key], b_[key]), (layer, b, h, key)
                    else:
                        assert a_[key] == b_[key], (layer, b, h, key)


@pytest.mark.parametrize("policy,n_side,v_codec", [("position", 1, "int"), ("position", 2, "int"),
                                                   ("h2o", 2, "int"), ("position", 2, "pq")])
def test_pipelined_graph_matches_eager_steps(policy, n_side, v_codec):
    """Pipelined steps (each layer's maintenance for the next step on a side stream, right
    after its attention; with two side streams the layers take them in turn) give the same
    outputs as the method's step order, and after one more maintenance pass the same cache."""
    import torch

    wl = get_workload(4).scaled(layers=3, batch=2, num_q_heads=8, num_kv_heads=2,
                                prompt_len=1200, int4_budget=500, policy=policy)
    if policy == "h2o":
        wl = wl.scaled(rope=get_workload(3).rope)
    masses = _masses(wl)
    eager, piped = _make(wl, masses, v_codec), _make(wl, masses, v_codec)
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    steps = 4
    q = torch.from_numpy(draw_vectors(wl, "q", (steps, L, B, Hq, d), "pipe")).cuda()
    k = torch.from_numpy(draw_vectors(wl, "k", (steps, L, B, Hkv, d), "pipe")).cuda()
    v = torch.from_numpy(draw_vectors(wl, "v", (steps, L, B, Hkv, d), "pipe")).cuda()
    out_e = torch.empty((L, B, Hq, d), dtype=torch.float16, device="cuda")
    out_p = torch.empty_like(out_e)
    side = [torch.cuda.Stream() for _ in range(n_side)]
    piped.maintain_all()
    qb, kb, vb = q[0].clone(), k[0].clone(), v[0].clone()
    g = piped.capture_step(qb, kb, vb, out_p, side)
    for s in range(steps):
        eager.step_all(q[s], k[s], v[s], out_e)
        qb.copy_(q[s])
        kb.copy_(k[s])
        vb.copy_(v[s])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_e.view(torch.int16), out_p.view(torch.int16)), f"step {s}"
    eager.maintain_all()
    torch.cuda.synchronize()
    for layer in range(L):
        for b in range(B):
            for h in range(Hkv):
                a_, b_ = eager.unit_state(layer, b, h), piped.unit_state(layer, b, h)
                for key in a_:
                    if isinstance(a_[key], np.ndarray):
                        assert np.array_equal(a_[key], b_[key]), (layer, b, h, key)
                    else:
                        assert a_[key] == b_[key], (layer, b, h, key)


@pytest.mark.parametrize("kb,vb,prompt", [(4, 4, 700), (2, 2, 700), (4, 4, 322), (4, 2, 322),
                                          (2, 4, 322)])
def test_growing_graph_matches_eager_steps(kb, vb, prompt):
    """Without eviction the cache grows by one token a step; a captured step replayed with the
    positions copied in and the host mirror advanced (growing_step) gives the same bytes as
    launching every call. The tensor-core attention kernel's schedule follows the tile counts,
    so the step is captured again when a row's middle tier reaches a new 256-token tile:
    prompt 322 leaves 254 middle tokens, so the third step crosses one."""
    import torch

    wl = get_workload(2).scaled(layers=2, batch=2, num_q_heads=8, num_kv_heads=2,
                                prompt_len=prompt, middle_k_bits=kb, middle_v_bits=vb, steps=6)
    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    def make():
        cfg = T.Config.from_workload(wl, mid_capacity=700)
        fc = FadeCache(cfg, wl.layers, wl.prompt_len, wl.prompt_len + 64, "cuda")
        for layer in range(wl.layers):
            pr = draw_prompt(wl, layer)
            fc.prefill(layer, torch.from_numpy(pr["k"]).cuda(), torch.from_numpy(pr["v"]).cuda())
        return fc

    eager, grown = make(), make()
    assert grown.growing_graph_ok()
    tiled = T.fade.fade_attention_tiled(grown.cfg)
    assert tiled
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    steps = 6
    q = torch.from_numpy(draw_vectors(wl, "q", (steps, L, B, Hq, d), "grow")).cuda()
    k = torch.from_numpy(draw_vectors(wl, "k", (steps, L, B, Hkv, d), "grow")).cuda()
    v = torch.from_numpy(draw_vectors(wl, "v", (steps, L, B, Hkv, d), "grow")).cuda()
    out_e = torch.empty((L, B, Hq, d), dtype=torch.float16, device="cuda")
    out_g = torch.empty_like(out_e)
    qb, kb_, vb_ = q[0].clone(), k[0].clone(), v[0].clone()
    for s in range(steps):
        eager.step_all(q[s], k[s], v[s], out_e)
        qb.copy_(q[s])
        kb_.copy_(k[s])
        vb_.copy_(v[s])
        grown.growing_step(qb, kb_, vb_, out_g)
        torch.cuda.synchronize()
        assert torch.equal(out_e.view(torch.int16), out_g.view(torch.int16)), f"step {s}"
        assert all((a == b).all() for x, y in zip(eager.mirror(), grown.mirror())
                   for a, b in zip(x, y))
    assert grown.growing_captures == (2 if prompt == 322 else 1)
    for layer in range(L):
        for b in range(B):
            for h in range(Hkv):
                a_, b_ = eager.unit_state(layer, b, h), grown.unit_state(layer, b, h)
                for key in a_:
                    if isinstance(a_[key], np.ndarray):
                        assert np.array_equal(a_[key], b_[key]), (layer, b, h, key)
                    else:
                        assert a_[key] == b_[key], (layer, b, h, key)


@pytest.mark.parametrize("policy", ["position", "h2o"])
def test_host_fed_pipeline_matches_eager_steps(policy):
    """run_from_host (two captured graphs taking the steps in turn, inputs copied in from
    pinned host memory while the previous step runs, outputs copied out while the next one
    runs, maintenance on side streams) gives every step's outputs, and the cache after the
    last step, bit for bit as launching every call."""
    import torch

    wl = get_workload(4).scaled(layers=2, batch=2, num_q_heads=8, num_kv_heads=2,
                                prompt_len=1200, int4_budget=500, policy=policy)
    if policy == "h2o":
        wl = wl.scaled(rope=get_workload(3).rope)
    masses = _masses(wl)
    eager, fed = _make(wl, masses), _make(wl, masses)
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    steps = 5
    qh = torch.from_numpy(draw_vectors(wl, "q", (steps, L, B, Hq, d), "host")).pin_memory()
    kh = torch.from_numpy(draw_vectors(wl, "k", (steps, L, B, Hkv, d), "host")).pin_memory()
    vh = torch.from_numpy(draw_vectors(wl, "v", (steps, L, B, Hkv, d), "host")).pin_memory()
    oh = torch.full((steps, L, B, Hq, d), float("nan"), dtype=torch.float16).pin_memory()
    side = [torch.cuda.Stream(), torch.cuda.Stream()]
    fed.maintain_all()                    # the pipelined schedule's prologue
    fed.run_from_host(qh, kh, vh, oh, side)
    torch.cuda.synchronize()
    out_e = torch.empty((L, B, Hq, d), dtype=torch.float16, device="cuda")
    for s in range(steps):
        eager.step_all(qh[s].cuda(), kh[s].cuda(), vh[s].cuda(), out_e)
        torch.cuda.synchronize()
        assert torch.equal(oh[s].view(torch.int16), out_e.cpu().view(torch.int16)), f"step {s}"
    eager.maintain_all()                  # the fed cache already ran the next maintenance
    torch.cuda.synchronize()
    for a, b in zip(eager.layers, fed.layers):
        assert torch.equal(a.meta, b.meta)
        cur = int(a.meta[0, 0, 4])
        assert torch.equal(a.mid_k_codes[cur], b.mid_k_codes[cur])
        assert torch.equal(a.recent_k, b.recent_k)
        assert np.array_equal(a.h_n_mid, b.h_n_mid)
