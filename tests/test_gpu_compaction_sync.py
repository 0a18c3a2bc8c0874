"""Compaction under a selection policy skips the middle tokens that both ping-pong buffers
already hold alike (below the agreement index in the unit's metadata and before the step's
first victim): it copies only their scores. Two checks on the GPU:

* the invariant itself: after every step, the two buffers' K/V codes and scales agree byte
  for byte below each unit's agreement index, which never exceeds the middle count;
* the skip changes nothing: a cache whose agreement index is cleared before every step
  (so every compaction copies every token) gives the same outputs and the same live state,
  bit for bit.
"""

import numpy as np
import pytest

from synth import draw_prompt, draw_vectors, get_workload
from synth.draws import ragged_context_lengths

pytestmark = pytest.mark.gpu

SYNC = 6  # FADE_META_SYNC


def _workload(policy):
    if policy == "ema":
        return get_workload(5).scaled(layers=2, batch=3, num_q_heads=8, num_kv_heads=2,
                                      ragged=(700, 1200), prompt_len=1200, int4_budget=500,
                                      steps=8)
    return get_workload(3).scaled(layers=2, batch=2, num_q_heads=8, num_kv_heads=2,
                                  prompt_len=900, int4_budget=300, steps=8)


def _make(wl):
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    lens = ragged_context_lengths(wl)
    P = int(lens.max())
    cfg = T.Config.from_workload(wl)
    fc = FadeCache(cfg, wl.layers, P, P + wl.steps + 8, "cuda")
    h2o = wl.policy == "h2o"
    for layer in range(wl.layers):
        pr = draw_prompt(wl, layer, P, with_q=h2o)
        q = torch.from_numpy(pr["q"]).cuda() if h2o else None   # GPU prefill mass (H2O)
        fc.prefill(layer, torch.from_numpy(pr["k"]).cuda(), torch.from_numpy(pr["v"]).cuda(),
                   lens, q_raw=q)
    return fc


def _check_agreement(fc):
    """Both buffers agree below every unit's agreement index; returns the largest index."""
    top = 0
    for L in fc.layers:
        meta = L.meta.cpu().numpy()
        bufs = [[t.cpu().numpy() for t in getattr(L, n)]
                for n in ("mid_k_codes", "mid_k_scales", "mid_v_codes", "mid_v_scales")]
        for b in range(meta.shape[0]):
            for h in range(meta.shape[1]):
                sync, n_mid = int(meta[b, h, SYNC]), int(meta[b, h, 1])
                assert 0 <= sync <= n_mid, (b, h, sync, n_mid)
                for pair in bufs:
                    assert np.array_equal(pair[0][b, h, :sync], pair[1][b, h, :sync]), (b, h)
                top = max(top, sync)
    return top


@pytest.mark.parametrize("policy", ["ema", "h2o"])
def test_skipped_compaction_matches_full_copies(policy):
    import torch

    wl = _workload(policy)
    fast, full = _make(wl), _make(wl)
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q = torch.from_numpy(draw_vectors(wl, "q", (wl.steps, L, B, Hq, d), "sync")).cuda()
    k = torch.from_numpy(draw_vectors(wl, "k", (wl.steps, L, B, Hkv, d), "sync")).cuda()
    v = torch.from_numpy(draw_vectors(wl, "v", (wl.steps, L, B, Hkv, d), "sync")).cuda()
    out_f = torch.empty((L, B, Hq, d), dtype=torch.float16, device="cuda")
    out_c = torch.empty_like(out_f)
    top = 0
    for s in range(wl.steps):
        for layer in full.layers:
            layer.meta[:, :, SYNC] = 0
        fast.step_all(q[s], k[s], v[s], out_f)
        full.step_all(q[s], k[s], v[s], out_c)
        torch.cuda.synchronize()
        assert torch.equal(out_f.view(torch.int16), out_c.view(torch.int16)), f"step {s}"
        top = max(top, _check_agreement(fast))
        for layer in range(L):
            for b in range(B):
                for h in range(Hkv):
                    a_, b_ = fast.unit_state(layer, b, h), full.unit_state(layer, b, h)
                    for key in a_:
                        if isinstance(a_[key], np.ndarray):
                            assert np.array_equal(a_[key], b_[key]), (s, layer, b, h, key)
                        else:
                            assert a_[key] == b_[key], (s, layer, b, h, key)
    assert top > 0, "no compaction skipped any token: the test does not exercise the skip"
