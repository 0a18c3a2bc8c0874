"""The C ABI without a GPU: the library builds and loads, every declared entry point is
exported, host-side validation returns the documented errors, and the host-only queries agree
with the oracle's accounting and step schedule."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fade.h")


@pytest.fixture(scope="module")
def T():
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)

    from tiered_mixed_precision_gb300 import build

    build.build()
    import tiered_mixed_precision_gb300 as T

    return T


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fade_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(T):
    names = declared_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(T.fade.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def _cfg(T, **kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, n_sink=4,
                recent_window=64, int4_budget=400, middle_k_bits=4, middle_v_bits=2,
                mid_capacity=401, policy="h2o")
    base.update(kw)
    return T.Config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2),
    (dict(num_q_heads=6), 2),
    (dict(num_q_heads=7), 1),
    (dict(middle_v_bits=3), 2),
    (dict(mid_capacity=400), 3),
    (dict(ema_decay=1.0), 1),
    (dict(recent_window=0), 1),
    (dict(batch=0), 1),
    (dict(batch=257), 1),
    (dict(rope_base=1.0), 1),
    (dict(rope_rotary_dim=6), 1),
    (dict(rope_rotary_dim=132), 1),
    (dict(rope_rotary_dim=2), 1),
    (dict(rope_kind="llama3", rope_low_freq_factor=4.0, rope_high_freq_factor=1.0), 1),
    (dict(v_codec="pq", middle_v_bits=4), 1),
    (dict(rope_kind="dynamic", rope_factor=0.5), 1),
])
def test_invalid_configs_are_rejected_on_the_host(T, kw, status):
    with pytest.raises(T.FadeError) as e:
        T.fade_layout(_cfg(T, **kw), 1024)
    assert e.value.status == status
    assert T.fade_last_error()


def test_layout_sizes(T):
    c = _cfg(T)
    lay = T.fade_layout(c, 2048)
    units = 2 * 2
    C = lay.mid_stride
    assert C == 448 and C % 64 == 0 and C >= 401          # capacity rounded up to 64 slots
    assert lay.mid_k_codes == units * C * 64
    assert lay.mid_v_codes == units * C * 32
    assert lay.mid_k_scales == units * C * 4 * 2
    assert lay.sink_k == units * 4 * 128 * 2
    assert lay.recent_k == units * 64 * 128 * 2
    assert lay.logits_ws == 2 * 8 * (4 + C + 64) * 4
    assert lay.victim_words >= 2048 // 32 + 1


def test_null_pointers_rejected_before_any_launch(T):
    class S:  # a stream object whose handle is never used
        cuda_stream = 0
    with pytest.raises(T.FadeError) as e:
        T.fade_quantize_pack(None, 4, 64, 4, None, None, stream=S())
    assert e.value.status == 1
    with pytest.raises(T.FadeError):
        T.fade_dequantize(None, None, 4, 64, 2, None, stream=S())


def test_next_position_and_compressed_bytes_follow_the_oracle(T):
    """Host mirror queries, on a layer object holding host memory only."""
    from oracle import accounting
    from oracle.cache import Params, UnitCache
    from oracle.rope import RopeTable
    from synth import Workload, draw_decode_tokens, draw_prompt

    wl = Workload(name="t", layers=1, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64,
                  n_sink=2, recent_window=4, int4_budget=3, policy="position", middle_k_bits=4,
                  middle_v_bits=2, prompt_len=9, steps=12, seed=3)
    cfg = T.Config.from_workload(wl)
    layer = T.TieredLayer(cfg, 16, device="cpu")
    u = UnitCache(Params.from_workload(wl), RopeTable.from_workload(wl, 64))
    u.prefill(draw_prompt(wl, 0)["k"][0, 0], draw_prompt(wl, 0)["v"][0, 0])
    for step in range(12):
        layer.h_n_sink[0], layer.h_n_mid[0], layer.h_n_recent[0] = u.n_sink, u.n_mid, u.n_recent
        assert T.fade_next_position(layer, 0) == u.next_position()
        want = accounting.unit_bytes(64, u.n_sink + u.n_recent, u.n_mid, 4, 2)
        assert T.fade_compressed_bytes(layer) == want
        t = draw_decode_tokens(wl, 0, step)
        u.step(t["q"][0], t["k"][0, 0], t["v"][0, 0])
    with pytest.raises(T.FadeError):
        T.fade_next_position(layer, 5)


def test_pq_compressed_bytes_follow_the_oracle(T):
    """A PQ middle token stores K codes and scales plus d/4 code bytes, no V scale."""
    from oracle import accounting

    for d in (64, 128):
        cfg = _cfg(T, head_dim=d, v_codec="pq", batch=1, num_q_heads=4, num_kv_heads=1)
        layer = T.TieredLayer(cfg, 16, device="cpu")
        layer.h_n_sink[0], layer.h_n_mid[0], layer.h_n_recent[0] = 4, 300, 64
        want = accounting.unit_bytes(d, 68, 0, 4, 2) + 300 * accounting.middle_token_bytes(
            d, 4, 2, v_codec="pq")
        assert T.fade_compressed_bytes(layer) == want
        assert layer.pq_codebook.shape == (d // 4, 256, 4)


def test_missing_library_fails_loudly(monkeypatch):
    import tiered_mixed_precision_gb300.fade as F

    monkeypatch.setattr(F, "_lib", None)
    monkeypatch.setattr(F, "LIB_PATH", "/nonexistent/libfade.so")
    with pytest.raises(ImportError):
        F.lib()


def test_config_struct_is_cached_and_rebuilt_on_change(T):
    """Config.c() builds the C struct once per set of field values (every entry point takes
    it); setting a field, or dataclasses.replace, gives a fresh struct."""
    import dataclasses

    cfg = _cfg(T)
    a = cfg.c()
    assert cfg.c() is a
    cfg.policy = "ema"
    assert cfg.c() is not a and cfg.c().policy == 2
    pq = dataclasses.replace(cfg, v_codec="pq")
    assert pq.c().v_codec == 1 and cfg.c().v_codec == 0
    assert dataclasses.replace(cfg) == cfg


@pytest.mark.parametrize("policy,budget", [("none", -1), ("position", 3), ("h2o", 5)])
def test_advance_host_follows_the_oracle_counts(T, policy, budget):
    """fade_cache_advance_host moves the host mirror exactly as one decode step moves the
    oracle's tier counts (demote, evict, append), and a step that would overflow the middle
    tier is refused with the mirror unchanged."""
    from oracle.cache import Params, UnitCache
    from oracle.rope import RopeTable
    from synth import Workload, draw_decode_tokens, draw_prompt

    wl = Workload(name="t", layers=1, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64,
                  n_sink=2, recent_window=4, int4_budget=budget, policy=policy,
                  middle_k_bits=4, middle_v_bits=2, prompt_len=3, steps=14, seed=5)
    cfg = T.Config.from_workload(wl)
    layer = T.TieredLayer(cfg, 16, device="cpu")
    u = UnitCache(Params.from_workload(wl), RopeTable.from_workload(wl, 64))
    pr = draw_prompt(wl, 0)
    u.prefill(pr["k"][0, 0], pr["v"][0, 0], mass=np.ones(3) if policy == "h2o" else None)
    layer.h_n_sink[0], layer.h_n_mid[0], layer.h_n_recent[0] = u.n_sink, u.n_mid, u.n_recent
    for step in range(14):
        t = draw_decode_tokens(wl, 0, step)
        u.step(t["q"][0], t["k"][0, 0], t["v"][0, 0])
        T.fade_cache_advance_host(layer)
        assert (layer.h_n_sink[0], layer.h_n_mid[0], layer.h_n_recent[0]) == \
            (u.n_sink, u.n_mid, u.n_recent), step
    if policy == "none":   # the middle tier is at its capacity: the next demotion is refused
        full = T.TieredLayer(T.Config.from_workload(wl, mid_capacity=layer.h_n_mid[0]), 16,
                             device="cpu")
        full.h_n_sink[0], full.h_n_mid[0], full.h_n_recent[0] = 2, layer.h_n_mid[0], 4
        with pytest.raises(T.FadeError) as e:
            T.fade_cache_advance_host(full)
        assert e.value.status == 3
        assert (full.h_n_sink[0], full.h_n_mid[0], full.h_n_recent[0]) == (2, layer.h_n_mid[0], 4)


def test_tier_counts_query_reads_the_host_mirror(T):
    cfg = _cfg(T, batch=3)
    layer = T.TieredLayer(cfg, 16, device="cpu")
    for b, (s, m, r) in enumerate([(4, 0, 10), (4, 350, 64), (2, 0, 0)]):
        layer.h_n_sink[b], layer.h_n_mid[b], layer.h_n_recent[b] = s, m, r
    got = T.fade.fade_tier_counts(layer)
    assert got.tolist() == [[4, 0, 10], [4, 350, 64], [2, 0, 0]]


def test_debug_build_compiles_and_exports_every_symbol():
    """The FADE_DEBUG=1 variant (device index checks on the hot paths) builds in its own
    directory and exports the same entry points."""
    import torch  # noqa: F401

    from tiered_mixed_precision_gb300 import build

    path = build.build(debug=True)
    assert path.endswith(os.path.join("_build_debug", "libfade.so"))
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported by the debug build: {missing}"


@pytest.mark.parametrize("kw,tiled", [
    (dict(), True),                                          # INT4 K, INT2 V
    (dict(middle_v_bits=4), True),                           # INT4 V (safe preset)
    (dict(v_codec="pq"), True),                              # PQ-coded V
    (dict(head_dim=64, middle_v_bits=4, num_q_heads=16), True),
    (dict(middle_k_bits=2, middle_v_bits=2), True),          # INT2 K
    (dict(middle_k_bits=2, middle_v_bits=4), True),
    (dict(middle_k_bits=2, middle_v_bits=2, v_codec="pq"), True),
])
def test_attention_tiled_query(T, kw, tiled):
    """fade_attention_tiled names the configurations whose attention runs the tensor-core
    kernel (scheduled by middle tiles); an invalid configuration is an error."""
    assert T.fade.fade_attention_tiled(_cfg(T, **kw)) is tiled


def test_attention_tiled_query_rejects_invalid_config(T):
    with pytest.raises(T.FadeError):
        T.fade.fade_attention_tiled(_cfg(T, head_dim=96))


def test_tile_constant_matches_the_header(T):
    m = re.search(r"#define\s+FADE_ATTN_TILE_TOKENS\s+(\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == T.fade.ATTN_TILE_TOKENS


def test_growing_graph_key_follows_the_tile_counts(T):
    """The growing-step graph is keyed on every layer's and row's count of middle tiles at the
    coming attention call (one more middle token than the mirror holds): the counts the
    tensor-core kernel's schedule is built from, for INT4 and INT2 K alike."""
    from types import SimpleNamespace

    from tiered_mixed_precision_gb300.model import FadeCache

    t = T.fade.ATTN_TILE_TOKENS

    def key(cfg, mids):
        layers = [SimpleNamespace(h_n_mid=np.array(m, np.int32)) for m in mids]
        return FadeCache.growing_graph_key(SimpleNamespace(cfg=cfg, layers=layers))

    tiled = _cfg(T, middle_v_bits=4, batch=2)
    assert key(tiled, [[t - 2, 0], [3 * t - 1, 5]]) == ((1, 1), (3, 1))
    assert key(tiled, [[t - 1, 0], [3 * t, 5]]) == ((1, 1), (4, 1))   # the second layer crosses
    assert key(tiled, [[t - 1, 0]]) != key(tiled, [[t, 0]])          # 256 -> 257 at the call
    k2 = _cfg(T, middle_k_bits=2, middle_v_bits=2, batch=2)
    assert key(k2, [[10, 20]]) == ((1, 1),)


def test_rope_append_validates_before_any_launch(T):
    """fade_rope_append rejects NULL inputs and both capacity overflows (the recent window full
    without demotion; the middle tier full with it) on the host, leaving the mirror as it was."""
    import torch

    cfg = _cfg(T, batch=2)   # mid_capacity 401
    layer = T.TieredLayer(cfg, 16, device="cpu")
    x = torch.zeros(4, dtype=torch.float16)
    layer.h_n_sink[:] = 4
    layer.h_n_recent[:] = [64, 10]
    layer.h_n_mid[:] = [401, 3]

    class S:  # a stream object whose handle is never used
        cuda_stream = 0
    with pytest.raises(T.FadeError) as e:
        T.fade.fade_rope_append(layer, None, 10, None, x, x, x, x, stream=S())
    assert e.value.status == 1
    with pytest.raises(T.FadeError) as e:   # row 0's ring is full and nothing demotes
        T.fade.fade_rope_append(layer, x, 10, x, x, x, x, x, demote=False, stream=S())
    assert e.value.status == 3
    with pytest.raises(T.FadeError) as e:   # row 0 would demote into a full middle tier
        T.fade.fade_rope_append(layer, x, 10, x, x, x, x, x, demote=True, stream=S())
    assert e.value.status == 3
    assert layer.h_n_recent.tolist() == [64, 10] and layer.h_n_mid.tolist() == [401, 3]
