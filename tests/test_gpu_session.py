"""Session persistence (page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §会话持久化): a cache
saved mid-stream (cache_state_dict, torch.save) and restored into a fresh cache
(torch.load, load_cache_state_dict) continues bit for bit like the uninterrupted one."""

import io

import numpy as np
import pytest

from synth import draw_prompt, draw_vectors, get_workload, ragged_context_lengths
from synth.draws import pq_calibration, pq_init_indices

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy,v_codec", [("position", "int"), ("h2o", "int"), ("ema", "int"),
                                            ("position", "pq")])
def test_state_dict_round_trip_continues_bit_identically(policy, v_codec):
    """With PQ-coded V the layers' codebooks travel in the state too."""
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    base = {"position": 4, "h2o": 3, "ema": 5}[policy]
    wl = get_workload(base).scaled(layers=2, batch=2, num_q_heads=8, num_kv_heads=2,
                                   prompt_len=700, int4_budget=200, ragged=None, steps=6)
    cfg = T.Config.from_workload(wl)
    cfg.v_codec = v_codec
    lens = ragged_context_lengths(wl)
    maxP = int(lens.max())
    max_pos = maxP + 32
    a = FadeCache(cfg, wl.layers, maxP, max_pos)
    if v_codec == "pq":   # a trained codebook per layer (different per layer)
        for layer in range(wl.layers):
            calib = pq_calibration(wl.scaled(seed=wl.seed + layer), 600, backend="torch",
                                   device="cuda")
            a.train_pq_codebook(calib, pq_init_indices(600, layer), 2, layer=layer)
    for layer in range(wl.layers):
        pr = draw_prompt(wl, layer, maxP, with_q=policy == "h2o", backend="torch", device="cuda")
        a.prefill(layer, pr["k"], pr["v"], lens, None, q_raw=pr.get("q"))
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q = draw_vectors(wl, "q", (6, L, B, Hq, d), "session", backend="torch", device="cuda")
    k = draw_vectors(wl, "k", (6, L, B, Hkv, d), "session", backend="torch", device="cuda")
    v = draw_vectors(wl, "v", (6, L, B, Hkv, d), "session", backend="torch", device="cuda")
    out_a = torch.empty((L, B, Hq, d), dtype=torch.float16, device="cuda")
    out_b = torch.empty_like(out_a)
    for s in range(3):
        a.step_all(q[s], k[s], v[s], out_a)
    sd = a.cache_state_dict()
    buf = io.BytesIO()
    torch.save(sd, buf)
    buf.seek(0)
    b = FadeCache(cfg, L, maxP, max_pos)
    b.load_cache_state_dict(torch.load(buf, weights_only=True))
    for s in range(3, 6):
        a.step_all(q[s], k[s], v[s], out_a)
        b.step_all(q[s], k[s], v[s], out_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16)), f"step {s}"
    for layer in range(L):
        for row in range(B):
            for h in range(Hkv):
                sa, sb = a.unit_state(layer, row, h), b.unit_state(layer, row, h)
                for key in sa:
                    if isinstance(sa[key], np.ndarray):
                        assert np.array_equal(sa[key], sb[key]), (layer, row, h, key)
                    else:
                        assert sa[key] == sb[key], (layer, row, h, key)
    # a cache of another configuration refuses the state
    other = FadeCache(T.Config.from_workload(wl.scaled(int4_budget=150)), L, maxP, max_pos)
    with pytest.raises(ValueError):
        other.load_cache_state_dict(sd)
