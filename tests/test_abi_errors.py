"""Host-side failure detection of the C ABI, without a GPU: every capacity and argument error
is returned before anything is enqueued, so these calls run on a layer whose buffers are host
memory (no kernel is ever launched)."""

import numpy as np
import pytest


@pytest.fixture(scope="module")
def T():
    import torch  # noqa: F401

    from tiered_mixed_precision_gb300 import build

    build.build()
    import tiered_mixed_precision_gb300 as T

    return T


class _S:  # a stream handle that is never used (no launch happens)
    cuda_stream = 0


def _layer(T, **kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=64, n_sink=2,
                recent_window=4, int4_budget=3, middle_k_bits=4, middle_v_bits=2,
                mid_capacity=4, policy="h2o")
    base.update(kw)
    cfg = T.Config(**base)
    return T.TieredLayer(cfg, 32, device="cpu")


def _expect(T, status, fn, *args, **kw):
    with pytest.raises(T.FadeError) as e:
        fn(*args, stream=_S(), **kw)
    assert e.value.status == status, str(e.value)
    return str(e.value)


def test_append_into_a_full_window_is_a_capacity_error(T):
    L = _layer(T)
    L.h_n_sink[:] = 2
    L.h_n_recent[:] = 4
    import torch
    k = torch.zeros((2, 2, 64), dtype=torch.float16)
    msg = _expect(T, 3, T.fade_cache_append, L, k, k)
    assert "recent window full" in msg
    # the host mirror is untouched by a rejected call
    assert L.h_n_recent.tolist() == [4, 4]


def test_demote_into_a_full_middle_tier_is_a_capacity_error(T):
    L = _layer(T, mid_capacity=4)
    L.h_n_recent[:] = 4
    L.h_n_mid[:] = 4
    _expect(T, 3, T.fade_cache_demote, L)


def test_prefill_errors(T):
    import torch
    L = _layer(T)
    k = torch.zeros((2, 2, 16, 64), dtype=torch.float16)
    # H2O needs the prefill mass
    _expect(T, 1, T.fade_cache_prefill, L, k, k, 16, np.array([16, 16]), None, k, 64)
    # a row longer than the prompt buffer
    m = torch.zeros((2, 2, 16), dtype=torch.float32)
    _expect(T, 1, T.fade_cache_prefill, L, k, k, 16, np.array([17, 3]), m, k, 64)
    # the cache must be empty
    L.h_n_sink[:] = 1
    _expect(T, 1, T.fade_cache_prefill, L, k, k, 16, np.array([16, 16]), m, k, 64)
    L.h_n_sink[:] = 0
    # too many middle survivors for the capacity (no eviction)
    L2 = _layer(T, policy="none", int4_budget=-1, mid_capacity=4)
    _expect(T, 3, T.fade_cache_prefill, L2, k, k, 16, np.array([16, 16]), None, k, 64)
    # a RoPE table too short for the prompt positions
    _expect(T, 3, T.fade_cache_prefill, L, k, k, 16, np.array([16, 16]), m, k, 8)


def test_attention_workspace_and_empty_cache_errors(T):
    import torch
    L = _layer(T)
    q = torch.zeros((2, 8, 64), dtype=torch.float16)
    ml = torch.zeros(32, dtype=torch.float32)
    ws = torch.zeros(16, dtype=torch.uint8)
    _expect(T, 1, T.fade_decode_attention, L, q, q, None, ml, ws)      # empty cache
    L.h_n_sink[:] = 2
    L.h_n_recent[:] = 4
    L.h_n_mid[:] = 3
    msg = _expect(T, 3, T.fade_decode_attention, L, q, q, None, ml, ws)
    assert "workspace" in msg


def test_rope_apply_position_and_null_errors(T):
    import torch
    cfg = T.Config(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, mid_capacity=16)
    x = torch.zeros((1, 40, 64), dtype=torch.float16)
    tab = torch.zeros(32 * 64, dtype=torch.float32)
    _expect(T, 3, T.fade_rope_apply, cfg, tab, 32, x, x, 1, 40, None, 1)
    _expect(T, 1, T.fade_rope_apply, cfg, tab, 32, None, x, 1, 40, None, 1)
    _expect(T, 1, T.fade_rope_table_init, T.Config(batch=1, num_q_heads=4, num_kv_heads=1,
                                                   head_dim=64, mid_capacity=16,
                                                   rope_kind="none"), tab, 32)


def test_layer_with_missing_buffers_is_rejected(T):
    L = _layer(T)
    L.c.status = None
    _expect(T, 1, T.fade_cache_demote, L)


def test_pq_argument_errors(T):
    import torch

    cb = torch.zeros((32, 256, 4), dtype=torch.float16)
    x = torch.zeros((8, 128), dtype=torch.float16)
    codes = torch.zeros((8, 32), dtype=torch.uint8)
    ws = torch.zeros(T.fade.pq_train_ws_bytes(128), dtype=torch.uint8)
    _expect(T, 1, T.fade_pq_encode, cb, x, 8, 126, codes)          # dim not a multiple of 4
    _expect(T, 1, T.fade_pq_encode, None, x, 8, 128, codes)
    _expect(T, 1, T.fade_pq_decode, cb, None, 8, 128, x)
    idx = np.arange(256)
    _expect(T, 1, T.fade_pq_train, x, 8, 128, idx, 3, cb, ws)       # indices beyond 8 rows
    _expect(T, 1, T.fade_pq_train, x, 0, 128, np.zeros(256), 3, cb, ws)
    _expect(T, 1, T.fade_pq_train, x, 9000, 128, np.zeros(256), 3, cb, ws)
    _expect(T, 3, T.fade_pq_train, x, 8, 128, np.zeros(256), 3, cb, ws[:100])
    with pytest.raises(ValueError):
        T.fade_pq_train(x, 8, 128, np.zeros(255), 3, cb, ws, stream=_S())


def test_pq_layer_without_codebook_is_rejected(T):
    """The C side refuses a PQ layer whose codebook pointer is NULL."""
    import torch

    L = _layer(T, v_codec="pq")
    L.set_pq_codebook(torch.ones_like(L.pq_codebook))
    L.c.pq_codebook = None
    msg = _expect(T, 1, T.fade_cache_demote, L)
    assert "codebook" in msg


def test_pq_layer_refuses_to_encode_before_its_codebook_is_set(T):
    import torch

    L = _layer(T, v_codec="pq")
    with pytest.raises(ValueError):
        T.fade_cache_demote(L, stream=_S())
    L.set_pq_codebook(torch.ones_like(L.pq_codebook))
    assert L.pq_codebook_set
    L.c.status = None   # now the C side runs its own checks (and refuses this layer)
    _expect(T, 1, T.fade_cache_demote, L)


def test_advance_host_layers_matches_per_layer_calls_and_is_all_or_nothing(T):
    """fade_cache_advance_host_layers advances every layer's mirror as per-layer calls would;
    when one layer's row would overflow, no layer's mirror changes."""
    def layers(n):
        out = [_layer(T) for _ in range(n)]
        for i, L in enumerate(out):
            L.h_n_sink[:] = [2, i % 2]      # row 0: sinks full; row 1: the append adds a sink
            L.h_n_recent[:] = [4, 0]        # row 0: the window is full, a demotion is due
            L.h_n_mid[:] = [i % 4, 0]       # some rows then exceed the budget (3) and evict
        return out

    def expect(status, *args):
        with pytest.raises(T.FadeError) as e:
            T.fade_cache_advance_host_layers(*args)
        assert e.value.status == status, str(e.value)

    a, b = layers(5), layers(5)
    for L in a:
        T.fade_cache_advance_host(L)
    T.fade_cache_advance_host_layers(b[0].cfg, T.fade.layer_pointer_array(b), len(b))
    for x, y in zip(a, b):
        for name in ("h_n_sink", "h_n_mid", "h_n_recent"):
            assert np.array_equal(getattr(x, name), getattr(y, name)), name
    # the last layer's first row has a full window and a full middle tier: nothing is stored
    c = layers(3)
    c[2].h_n_mid[0] = c[2].cfg.mid_capacity
    before = [(L.h_n_sink.copy(), L.h_n_mid.copy(), L.h_n_recent.copy()) for L in c]
    expect(3, c[0].cfg, T.fade.layer_pointer_array(c), 3)
    for L, (s_, m_, r_) in zip(c, before):
        assert np.array_equal(L.h_n_sink, s_) and np.array_equal(L.h_n_mid, m_)
        assert np.array_equal(L.h_n_recent, r_)
    # an empty list is a no-op; a negative count is rejected
    T.fade_cache_advance_host_layers(c[0].cfg, None, 0)
    expect(1, c[0].cfg, None, -1)
