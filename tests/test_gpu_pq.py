"""Parity of product-quantised V (FADE-zh §产品量化) on the GPU with the oracle: the codec and
the codebook training bit for bit, and the whole decode step with PQ-coded middle V in
lockstep."""

import numpy as np
import pytest

from harness import Lockstep
from oracle import pq
from synth import draw_codec_cases, get_workload
from synth.draws import pq_calibration, pq_codebook, pq_init_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch  # noqa: F401

    import tiered_mixed_precision_gb300 as T

    T.lib()
    return T


def _tie_heavy_inputs(dim, n, seed):
    """A drawn codebook with duplicated centroids, and rows that sit exactly on centroids
    (so the duplicates tie) besides the codec edge cases (zeros, subnormals, near 65504)."""
    rng = np.random.default_rng(seed)
    cb = pq_codebook(rng, dim)
    cb[:, 200] = cb[:, 3]
    cb[:, 255] = cb[:, 0]
    x = draw_codec_cases(n, dim, seed)
    S = dim // 4
    for r in range(0, n, 5):  # every fifth row: each sub-vector on a (possibly tied) centroid
        pick = rng.integers(0, 256, S)
        x[r] = cb[np.arange(S), pick].reshape(dim)
    return cb, x


@pytest.mark.parametrize("dim", [64, 128])
@pytest.mark.parametrize("n", [1, 7, 1029])
def test_pq_encode_decode_bit_exact(T, dim, n):
    import torch

    cb, x = _tie_heavy_inputs(dim, n, seed=dim * 7 + n)
    cbd, xd = torch.from_numpy(cb).cuda(), torch.from_numpy(x).cuda()
    codes = torch.zeros((n, dim // 4), dtype=torch.uint8, device="cuda")
    T.fade_pq_encode(cbd, xd, n, dim, codes)
    want = pq.encode(x, cb)
    assert np.array_equal(codes.cpu().numpy(), want)
    out = torch.empty((n, dim), dtype=torch.float16, device="cuda")
    T.fade_pq_decode(cbd, codes, n, dim, out)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), pq.decode(want, cb).view(np.uint16))


@pytest.mark.parametrize("key,n,iters", [(4, 1500, 4), (3, 300, 3), (4, 200, 0)])
def test_pq_train_bit_exact(T, key, n, iters):
    """n = 200 < 256 draws repeated start rows: their duplicates lose every tie and keep
    their value (the empty-centroid rule)."""
    import torch

    from tiered_mixed_precision_gb300.model import FadeCache

    wl = get_workload(key)
    calib = pq_calibration(wl, n)
    idx = pq_init_indices(n, seed=key)
    want = pq.train(calib, idx, iters)
    cfg = T.Config(batch=1, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                   head_dim=wl.head_dim, mid_capacity=64, v_codec="pq")
    fc = FadeCache(cfg, 2, 16, 64)
    got = fc.train_pq_codebook(torch.from_numpy(calib).cuda(), idx, iters)
    assert np.array_equal(got.cpu().numpy().view(np.uint16), want.view(np.uint16))
    for L in fc.layers:   # installed in every layer
        assert np.array_equal(L.pq_codebook.cpu().numpy().view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("key,policy,kbits", [(4, "position", 4), (3, "h2o", 4), (5, "ema", 4),
                                             (1, "none", 4), (4, "h2o", 2), (3, "ema", 2)])
def test_pq_lockstep(T, key, policy, kbits):
    """The whole step with PQ-coded middle V: prefill tiering, demotion (encode), eviction
    and compaction (codes move as bytes), tensor-core attention (centroids decoded through
    shared memory; INT4 or INT2 K) and score accumulation, compared with the oracle after
    every call."""
    over = dict(layers=1, batch=2, ragged=None, prompt_len=600, int4_budget=200, steps=6,
                policy=policy, middle_k_bits=kbits)
    if key == 5:
        over.update(num_q_heads=8, num_kv_heads=2)
    if policy == "none":
        over.update(int4_budget=-1)
    wl = get_workload(key).scaled(**over)
    ls = Lockstep(wl, v_codec="pq")
    ls.prefill(0)
    ls.check_layer_state(0)
    for _ in range(ls.steps):
        ls.step()
    ls.check_near_ties()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 8])
def test_pq_lockstep_query_groups(T, d, G):
    """PQ-coded V on the tensor-core kernel for every query-group size it is built for."""
    wl = get_workload(4).scaled(layers=1, batch=2, num_q_heads=2 * G, num_kv_heads=2,
                                head_dim=d, ragged=None, prompt_len=700, int4_budget=300,
                                steps=4, policy="h2o" if G == 2 else "position")
    ls = Lockstep(wl, v_codec="pq")
    ls.prefill(0)
    ls.check_layer_state(0)
    for _ in range(ls.steps):
        ls.step()
    ls.check_near_ties()
