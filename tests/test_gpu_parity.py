"""Parity of the CUDA path (through the C ABI) with the oracle on seeded inputs."""

import numpy as np
import pytest

from harness import Lockstep, allclose_report
from oracle import quant
from oracle.rope import RopeTable
from synth import draw_codec_cases, get_workload
from synth.workloads import Rope

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch  # noqa: F401

    import tiered_mixed_precision_gb300 as T

    T.lib()
    return T


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dim", [64, 128])
@pytest.mark.parametrize("n", [1, 7, 1029])
def test_quantize_pack_and_dequantize_bit_exact(T, bits, dim, n):
    import torch

    x = draw_codec_cases(n, dim, seed=bits * 1000 + dim + n)
    xd = torch.from_numpy(x).cuda()
    codes = torch.zeros((n, dim * bits // 8), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n, dim // 32), dtype=torch.float16, device="cuda")
    T.fade_quantize_pack(xd, n, dim, bits, codes, scales)
    rc, rs = quant.quantize_pack(x, bits)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs.view(np.uint16))
    out = torch.empty((n, dim), dtype=torch.float32, device="cuda")
    T.fade_dequantize(codes, scales, n, dim, bits, out)
    q, s = quant.quantize(x, bits)
    assert np.array_equal(out.cpu().numpy(), quant.dequantize(q, s).astype(np.float32))


def test_codec_empty_input_is_a_no_op(T):
    import torch

    x = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    c = torch.full((1, 32), 7, dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 2), dtype=torch.float16, device="cuda")
    T.fade_quantize_pack(x, 0, 64, 4, c, s)
    torch.cuda.synchronize()
    assert int(c.sum()) == 7 * 32


_SCALED_ROPES = {
    "linear": Rope("linear", 1e4, factor=4.0),
    "ntk": Rope("ntk", 1e4, factor=8.0),
    "yarn": Rope("yarn", 1e4, factor=8.0, low_freq_factor=1.0, high_freq_factor=32.0,
                 original_max_position=4096),
    # the table length (40 000 here; about 900 in the lockstep case) exceeds the original
    # context, so the base is scaled by the length-derived factor
    "dynamic": Rope("dynamic", 1e4, factor=2.0, original_max_position=4096),
    "dynamic_short": Rope("dynamic", 1e4, factor=2.0, original_max_position=512),
    # proportional RoPE (partial_rotary_factor): 64 of 128 channels rotate (whole groups),
    # 80 of 128 (the third group half rotated), with llama3 frequencies over 48 of 64
    "prop64": Rope("default", 1e4, rotary_dim=64),
    "prop80": Rope("default", 5e5, rotary_dim=80),
    "prop48_llama3": Rope("llama3", 5e5, factor=32.0, low_freq_factor=1.0, high_freq_factor=4.0,
                          original_max_position=8192, rotary_dim=48),
}


@pytest.mark.parametrize("key", [1, 3, 4, "linear", "ntk", "yarn", "dynamic", "prop64", "prop80",
                                 "prop48_llama3"])
def test_rope_table_and_apply(T, key):
    import torch

    if isinstance(key, int):
        wl = get_workload(key)
    elif key == "prop48_llama3":
        wl = get_workload(3).scaled(rope=_SCALED_ROPES[key])
    else:
        wl = get_workload(4).scaled(rope=_SCALED_ROPES[key])
    rh = (wl.rope.rotary_dim or wl.head_dim) // 2   # rotation pairs in the table
    cfg = T.Config.from_workload(wl)
    max_pos = 40000
    table = torch.empty(max_pos * wl.head_dim, dtype=torch.float32, device="cuda")
    T.fade_rope_table_init(cfg, table, max_pos)
    ref = RopeTable.from_workload(wl, max_pos)
    # layout: per position, blocks of two pairs (cos_2b, cos_2b+1, sin_2b, sin_2b+1)
    tab = table.view(max_pos, wl.head_dim // 4, 4).cpu().numpy()
    cos = tab[..., 0:2].reshape(max_pos, wl.head_dim // 2)[:, :rh]
    sin = tab[..., 2:4].reshape(max_pos, wl.head_dim // 2)[:, :rh]
    for got, want in ((cos, ref.cos), (sin, ref.sin)):
        ulps = np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
        assert ulps.max() <= 1, "table entry more than 1 fp32 ulp from the oracle"
        assert (ulps != 0).mean() < 1e-4
    rng = np.random.default_rng(key if isinstance(key, int) else 10 + list(_SCALED_ROPES).index(key))
    x = rng.standard_normal((300, wl.head_dim)).astype(np.float16)
    pos = rng.integers(0, max_pos, 300).astype(np.int32)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    T.fade_rope_apply(cfg, table, max_pos, xd, yd, 300, 1, torch.from_numpy(pos).cuda(), 0)
    want = ref.apply(x, pos)
    got16 = yd.cpu().numpy().view(np.uint16)
    want16 = want.view(np.uint16)
    # where the two tables' rows agree the rotation must give identical bytes; a row with a
    # 1-ulp table entry may move an fp16 rounding by at most one ulp
    rows_agree = (np.all(cos[pos] == ref.cos[pos], axis=1)
                  & np.all(sin[pos] == ref.sin[pos], axis=1))
    assert rows_agree.mean() > 0.9
    assert np.array_equal(got16[rows_agree], want16[rows_agree])

    def ordered(u):  # fp16 bits -> integers in float order
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)

    assert np.abs(ordered(got16) - ordered(want16)).max() <= 1


@pytest.mark.parametrize("d,hq,hkv,rope,prompt", [
    (128, 8, 2, "default", 30),       # ring slots
    (128, 4, 4, "default", 2),        # sink slots (fewer than n_sink held)
    (64, 16, 2, "prop48", 30),        # proportional RoPE, G = 8
    (64, 8, 2, "none", 30),           # no positional encoding: copies
])
def test_rope_append_fused_matches_separate_calls(T, d, hq, hkv, rope, prompt):
    """fade_rope_append gives q_rot and the appended key, value, score and counts bit for bit
    as fade_rope_apply (q and k) followed by fade_cache_append, over several steps."""
    import torch

    from synth import draw_prompt, draw_vectors
    from tiered_mixed_precision_gb300.model import FadeCache

    r = {"default": Rope("default", 1e4), "none": Rope("none"),
         "prop48": _SCALED_ROPES["prop48_llama3"]}[rope]
    wl = get_workload(4).scaled(layers=1, batch=3, num_q_heads=hq, num_kv_heads=hkv,
                                head_dim=d, prompt_len=prompt, int4_budget=200, rope=r, steps=3)

    def make():
        fc = FadeCache(T.Config.from_workload(wl), 1, prompt, prompt + 16, "cuda")
        pr = draw_prompt(wl, 0)
        fc.prefill(0, torch.from_numpy(pr["k"]).cuda(), torch.from_numpy(pr["v"]).cuda())
        return fc

    sep, fus = make(), make()
    B = wl.batch
    for step in range(3):
        q = torch.from_numpy(draw_vectors(wl, "q", (B, hq, d), "fuse", step)).cuda()
        k = torch.from_numpy(draw_vectors(wl, "k", (B, hkv, d), "fuse", step)).cuda()
        v = torch.from_numpy(draw_vectors(wl, "v", (B, hkv, d), "fuse", step)).cuda()
        for fc in (sep, fus):
            fc.set_positions(fc.next_positions())
        c, L = sep.cfg, sep.layers[0]
        k_rot = torch.empty_like(k)
        T.fade.fade_rope_apply(c, sep.table, sep.max_pos, q, sep.q_rot, B, hq, sep.pos, 0)
        T.fade.fade_rope_apply(c, sep.table, sep.max_pos, k, k_rot, B, hkv, sep.pos, 0)
        T.fade.fade_cache_append(L, k_rot, v)
        T.fade.fade_rope_append(fus.layers[0], fus.table, fus.max_pos, q, k, v, fus.pos,
                                fus.q_rot)
        torch.cuda.synchronize()
        assert torch.equal(sep.q_rot.view(torch.int16), fus.q_rot.view(torch.int16)), step
        for b in range(B):
            for h in range(hkv):
                x, y = sep.unit_state(0, b, h), fus.unit_state(0, b, h)
                for key in x:
                    if isinstance(x[key], np.ndarray):
                        assert np.array_equal(x[key], y[key]), (step, b, h, key)
                    else:
                        assert x[key] == y[key], (step, b, h, key)
        assert (sep.layers[0].h_n_recent == fus.layers[0].h_n_recent).all()
        assert (sep.layers[0].h_n_sink == fus.layers[0].h_n_sink).all()


@pytest.mark.parametrize("d,kb,vb,codec,ragged", [(128, 4, 4, "int", None),
                                                   (64, 4, 2, "int", None),
                                                   (64, 2, 2, "int", None),
                                                   (128, 4, 2, "pq", None),
                                                   (128, 4, 4, "int", (30, 140))])
def test_rope_append_with_demotion_matches_separate_calls(T, d, kb, vb, codec, ragged):
    """fade_rope_append with demote: the demotion (K and V quantise-packed, or V PQ-encoded,
    into the next middle slot, the score moved), the RoPE of q and k and the append, in one
    launch, bit for bit as fade_cache_demote, fade_rope_apply twice and fade_cache_append."""
    import torch

    from synth import draw_prompt, draw_vectors
    from synth.draws import pq_calibration, ragged_context_lengths
    from tiered_mixed_precision_gb300.model import FadeCache

    # ragged: rows of 35 to 80 prompt tokens, so some rings are full (those rows demote) and
    # others are not, in the same launch
    wl = get_workload(2).scaled(layers=1, batch=4 if ragged else 2, num_q_heads=8,
                                num_kv_heads=2, head_dim=d, middle_k_bits=kb, middle_v_bits=vb,
                                prompt_len=140 if ragged else 100, steps=3, ragged=ragged)
    lens = ragged_context_lengths(wl)
    P = int(lens.max())

    def make():
        cfg = T.Config.from_workload(wl, mid_capacity=200)
        cfg.v_codec = codec
        fc = FadeCache(cfg, 1, P, P + 20, "cuda")
        if codec == "pq":
            rows = pq_calibration(wl, 256)
            cb = rows.reshape(256, d // 4, 4).transpose(1, 0, 2).copy()
            fc.set_pq_codebook(torch.from_numpy(cb).cuda())
        pr = draw_prompt(wl, 0, P)
        fc.prefill(0, torch.from_numpy(pr["k"]).cuda(), torch.from_numpy(pr["v"]).cuda(), lens)
        return fc

    sep, fus = make(), make()
    full = sep.layers[0].h_n_recent == wl.recent_window
    if ragged:
        assert full.any() and not full.all()   # both kinds of row in the launch
    else:
        assert full.all()                      # every step demotes
    B, hq, hkv = wl.batch, wl.num_q_heads, wl.num_kv_heads
    for step in range(3):
        q = torch.from_numpy(draw_vectors(wl, "q", (B, hq, d), "fuse_dem", step)).cuda()
        k = torch.from_numpy(draw_vectors(wl, "k", (B, hkv, d), "fuse_dem", step)).cuda()
        v = torch.from_numpy(draw_vectors(wl, "v", (B, hkv, d), "fuse_dem", step)).cuda()
        for fc in (sep, fus):
            fc.set_positions(fc.next_positions())
        c, L = sep.cfg, sep.layers[0]
        k_rot = torch.empty_like(k)
        T.fade.fade_cache_demote(L)
        T.fade.fade_rope_apply(c, sep.table, sep.max_pos, q, sep.q_rot, B, hq, sep.pos, 0)
        T.fade.fade_rope_apply(c, sep.table, sep.max_pos, k, k_rot, B, hkv, sep.pos, 0)
        T.fade.fade_cache_append(L, k_rot, v)
        T.fade.fade_rope_append(fus.layers[0], fus.table, fus.max_pos, q, k, v, fus.pos,
                                fus.q_rot, demote=True)
        torch.cuda.synchronize()
        assert torch.equal(sep.q_rot.view(torch.int16), fus.q_rot.view(torch.int16)), step
        for b in range(B):
            for h in range(hkv):
                x, y = sep.unit_state(0, b, h), fus.unit_state(0, b, h)
                for key in x:
                    if isinstance(x[key], np.ndarray):
                        assert np.array_equal(x[key], y[key]), (step, b, h, key)
                    else:
                        assert x[key] == y[key], (step, b, h, key)
        for name in ("h_n_sink", "h_n_mid", "h_n_recent"):
            assert (getattr(sep.layers[0], name) == getattr(fus.layers[0], name)).all(), name
        assert fus.layers[0].meta.cpu().numpy()[:, :, 3].tolist() == \
            sep.layers[0].meta.cpu().numpy()[:, :, 3].tolist()   # ring heads


def _small(key):
    if key == "1":
        return get_workload(1).scaled(steps=6), None
    if key == "2s":
        return get_workload(2).scaled(layers=2, prompt_len=300, steps=6), None
    if key == "3s":
        return get_workload(3).scaled(layers=1, batch=2, prompt_len=700, int4_budget=200,
                                      steps=12), None
    if key == "4s":
        return get_workload(4).scaled(layers=1, batch=3, num_q_heads=8, num_kv_heads=2,
                                      prompt_len=1500, int4_budget=600, steps=6), None
    if key == "5s":
        return get_workload(5).scaled(layers=1, batch=3, num_q_heads=8, num_kv_heads=2,
                                      ragged=(900, 1600), prompt_len=1600, int4_budget=700,
                                      steps=6), None
    if key == "5bs":
        return get_workload("5b").scaled(layers=1, batch=3, num_q_heads=8, num_kv_heads=2,
                                         ragged=(900, 1600), prompt_len=1600, steps=4), None
    if key == "g2_k2v4":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=4, num_kv_heads=2,
                                      middle_k_bits=2, middle_v_bits=4, prompt_len=1000,
                                      int4_budget=300, steps=5), None
    if key == "g1_h2o_d128":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=4, num_kv_heads=4,
                                      head_dim=128, prompt_len=600, int4_budget=150,
                                      steps=8), None
    if key == "d64_g8":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=16, num_kv_heads=2,
                                      prompt_len=900, int4_budget=500, steps=6), None
    if key == "d128_g8":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=16, num_kv_heads=2,
                                      prompt_len=1300, int4_budget=700, steps=5), None
    # the remaining (head_dim, K bits, V bits) combinations of the eviction kernels
    if key == "d64_k2v4_h2o":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      middle_k_bits=2, middle_v_bits=4, prompt_len=800,
                                      int4_budget=300, steps=6), None
    if key == "d128_k4v4_pos":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      middle_v_bits=4, prompt_len=1100, int4_budget=400,
                                      steps=5), None
    if key == "d64_k2v2_ema":
        return get_workload(5).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      head_dim=64, middle_k_bits=2, middle_v_bits=2,
                                      ragged=(700, 1200), prompt_len=1200, int4_budget=500,
                                      steps=5), None
    if key == "d128_k2v2_pos":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      middle_k_bits=2, middle_v_bits=2, prompt_len=900,
                                      int4_budget=350, steps=5), None
    if key == "d64_k4v4_pos":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      head_dim=64, middle_v_bits=4, prompt_len=900,
                                      int4_budget=350, steps=5), None
    # INT4 V on the tensor-core kernel (INT4 K) at every query-group size and head dimension
    if key == "v4_g1_h2o_d128":   # logits written for H2O, three tiles per unit
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=4, num_kv_heads=4,
                                      head_dim=128, middle_v_bits=4, prompt_len=900,
                                      int4_budget=600, steps=6), None
    if key == "v4_g2_ema_d64":    # ragged rows, EMA
        return get_workload(5).scaled(layers=1, batch=3, num_q_heads=4, num_kv_heads=2,
                                      head_dim=64, middle_v_bits=4, ragged=(700, 1300),
                                      prompt_len=1300, int4_budget=800, steps=5), None
    if key == "v4_g8_d64_h2o":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=16, num_kv_heads=2,
                                      middle_v_bits=4, prompt_len=900, int4_budget=500,
                                      steps=6), None
    # INT2 K on the tensor-core kernel at the query-group sizes the other INT2-K cases miss
    if key == "k2v2_g8_d128":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=16, num_kv_heads=2,
                                      middle_k_bits=2, prompt_len=1300, int4_budget=700,
                                      steps=5), None
    if key == "k2v4_g1_d64_h2o":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=4, num_kv_heads=4,
                                      middle_k_bits=2, middle_v_bits=4, prompt_len=900,
                                      int4_budget=500, steps=6), None
    if key == "v4_g8_d128_grow":  # the safe preset's shape, six tiles per unit, no eviction
        return get_workload(2).scaled(layers=1, batch=2, prompt_len=1400, steps=4), None
    # degenerate cases of the method
    if key == "deg_nosink":  # no sinks: the recent ring and the middle tier only
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      head_dim=64, n_sink=0, recent_window=16, prompt_len=300,
                                      int4_budget=120, steps=6), None
    if key == "deg_w1_h2o":  # a one-token recent window: every step demotes the previous token
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      n_sink=2, recent_window=1, prompt_len=200,
                                      int4_budget=60, steps=8), None
    if key == "deg_budget0":  # budget 0: every demoted token is evicted in the same step
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      prompt_len=200, int4_budget=0, steps=5), None
    if key == "deg_short_ragged":  # rows whose prompts do not reach the middle tier at first
        return get_workload(5).scaled(layers=1, batch=4, num_q_heads=8, num_kv_heads=2,
                                      recent_window=16, ragged=(2, 60), prompt_len=60,
                                      int4_budget=30, steps=10), None
    if key == "deg_norope_ema":  # no positional encoding: re-positioning is the identity
        return get_workload(5).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=Rope("none"), ragged=None, prompt_len=400,
                                      int4_budget=150, steps=6), None
    # the scaled RoPE schemes under each eviction policy (re-positioning uses their tables)
    if key == "rope_linear_pos":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["linear"], prompt_len=900,
                                      int4_budget=300, steps=5), None
    if key == "rope_ntk_h2o":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["ntk"], prompt_len=700,
                                      int4_budget=250, steps=6), None
    if key == "rope_dynamic_pos":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["dynamic_short"], prompt_len=900,
                                      int4_budget=300, steps=5), None
    # proportional RoPE under each eviction policy: whole groups rotated, a group split
    if key == "prop_pos_r64":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["prop64"], prompt_len=900,
                                      int4_budget=300, steps=5), None
    if key == "prop_h2o_r48":
        return get_workload(3).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["prop48_llama3"], prompt_len=700,
                                      int4_budget=250, steps=6), None
    if key == "prop_pos_r80":
        return get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["prop80"], prompt_len=900,
                                      int4_budget=300, steps=5), None
    if key == "prop_ema_r80":
        return get_workload(5).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["prop80"], ragged=(900, 1300),
                                      prompt_len=1300, int4_budget=500, steps=5), None
    if key == "rope_yarn_ema":
        return get_workload(5).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                      rope=_SCALED_ROPES["yarn"], ragged=(900, 1300),
                                      prompt_len=1300, int4_budget=500, steps=5), None
    raise KeyError(key)


@pytest.mark.parametrize("key", ["1", "2s", "3s", "4s", "5s", "5bs", "g2_k2v4", "g1_h2o_d128",
                                 "d64_g8", "d128_g8", "d64_k2v4_h2o", "d128_k4v4_pos",
                                 "d64_k2v2_ema", "d128_k2v2_pos", "d64_k4v4_pos",
                                 "v4_g1_h2o_d128", "v4_g2_ema_d64", "v4_g8_d64_h2o",
                                 "v4_g8_d128_grow", "k2v2_g8_d128", "k2v4_g1_d64_h2o",
                                 "deg_nosink", "deg_w1_h2o", "deg_budget0", "deg_short_ragged",
                                 "deg_norope_ema", "rope_linear_pos", "rope_ntk_h2o",
                                 "rope_yarn_ema", "rope_dynamic_pos", "prop_pos_r64",
                                 "prop_h2o_r48", "prop_pos_r80", "prop_ema_r80"])
def test_lockstep_small_workloads(T, key):
    wl, cap = _small(key)
    ls = Lockstep(wl, mid_capacity=cap)
    for layer in range(ls.L):
        ls.prefill(layer)
        ls.check_layer_state(layer)
    for _ in range(ls.steps):
        ls.step()
    ls.check_near_ties()


@pytest.mark.parametrize("policy,skip", [("position", 40), ("h2o", 40), ("position", 3)])
def test_deferred_eviction_many_victims(T, policy, skip):
    """Eviction left out for `skip` steps, then steps that evict every pending token at once:
    with 40 pending victims a compaction block needs more RoPE rows than it stages in shared
    memory, so its re-positioning reads the table from global memory."""
    if policy == "position":
        wl = get_workload(4).scaled(layers=1, batch=2, num_q_heads=4, num_kv_heads=2,
                                    prompt_len=1000, int4_budget=300, steps=skip + 2)
    else:
        wl = get_workload(3).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                    prompt_len=900, int4_budget=500, steps=skip + 2)
    ls = Lockstep(wl, mid_capacity=wl.int4_budget + skip + 8)
    ls.prefill(0)
    ls.check_layer_state(0)
    for _ in range(skip):
        ls.step(evict=False)
    for _ in range(2):
        ls.step()
    ls.check_near_ties()


@pytest.mark.parametrize("policy", ["h2o", "ema", "position"])
def test_shared_row_decisions_lockstep(T, policy):
    """Rows sharing their tier decisions (FADE-zh §批处理支持): the victims of every row of a
    KV head come from the row-summed scores (H2O: the row-summed prefill mass at prefill)."""
    base = {"h2o": 3, "ema": 5, "position": 4}[policy]
    wl = get_workload(base).scaled(layers=1, batch=3, num_q_heads=8, num_kv_heads=2,
                                   ragged=None, prompt_len=700, int4_budget=250, steps=8)
    ls = Lockstep(wl, shared_rows=True)
    ls.prefill(0)
    ls.check_layer_state(0)
    for _ in range(ls.steps):
        ls.step()
    ls.check_near_ties()


@pytest.mark.parametrize("key,P", [(3, 700), (3, 130), (4, 300)])
def test_prefill_mass_matches_oracle(T, key, P):
    """GPU prefill attention mass vs the oracle's fp64 causal column sums (d = 64 and 128),
    and the same bits on a second run."""
    import torch

    from oracle import attention
    from synth import draw_prompt

    wl = get_workload(key).scaled(batch=2, prompt_len=P)
    cfg = T.Config.from_workload(wl)
    lens = np.array([P, P - 37], np.int32)
    pr = draw_prompt(wl, 0, P, with_q=True)
    rope = RopeTable.from_workload(wl, P)
    pos = np.arange(P)
    qd = torch.from_numpy(pr["q"]).cuda()
    kd = torch.from_numpy(pr["k"]).cuda()
    table = torch.empty(P * wl.head_dim, dtype=torch.float32, device="cuda")
    T.fade_rope_table_init(cfg, table, P)
    B, Hq, Hkv = wl.batch, wl.num_q_heads, wl.num_kv_heads
    T.fade_rope_apply(cfg, table, P, qd, qd, B * Hq, P, None, 1)
    T.fade_rope_apply(cfg, table, P, kd, kd, B * Hkv, P, None, 1)
    mass = torch.full((B, Hkv, P), 7.0, dtype=torch.float32, device="cuda")
    T.fade_prefill_mass(cfg, qd, kd, P, lens, mass)
    got = mass.cpu().numpy()
    again = torch.full((B, Hkv, P), -1.0, dtype=torch.float32, device="cuda")
    T.fade_prefill_mass(cfg, qd, kd, P, lens, again)
    assert np.array_equal(again.cpu().numpy().view(np.uint32), got.view(np.uint32))
    G = wl.group
    for b in range(B):
        n = int(lens[b])
        for h in range(Hkv):
            q = np.stack([rope.apply(pr["q"][b, h * G + g, :n], pos[:n]) for g in range(G)])
            k = rope.apply(pr["k"][b, h, :n], pos[:n])
            ref = attention.prefill_mass(q.astype(np.float64), k.astype(np.float64))
            ok, err, nbad = allclose_report(got[b, h, :n], ref, atol=1e-5, rtol=1e-4)
            assert ok, f"row {b} head {h}: max err {err}, {nbad} bad"
            assert np.all(got[b, h, n:] == 0.0)


@pytest.mark.parametrize("key", ["3s", "g1_h2o_d128", "d64_g8"])
def test_gpu_prefill_mass_lockstep(T, key):
    """The product path of an H2O cache: the GPU computes the prefill mass and its prefill
    evicts by it. The mass must be deterministic and within tolerance of the oracle's, the
    selection rule replayed on the GPU's mass must give the GPU's victims (the prefilled state
    is compared bit for bit), and the decode steps that follow stay in lockstep."""
    wl, cap = _small(key)
    ls = Lockstep(wl, mid_capacity=cap)
    for layer in range(ls.L):
        ls.prefill(layer, gpu_mass=True)
        ls.check_layer_state(layer)
    for _ in range(ls.steps):
        ls.step()
    print(f"prefill near-ties (fp64 mass vs the GPU's fp32 mass): {ls.prefill_near_ties}")
    assert ls.prefill_near_ties <= max(1, wl.batch * wl.num_kv_heads * ls.L // 100)
    ls.check_near_ties()


@pytest.mark.parametrize("key,kv", [(3, (4, 2)), (4, (4, 2)), (2, (4, 4))])
def test_max_batch_ragged_lockstep(T, key, kv):
    """The largest batch the ABI admits (256 rows), ragged prompt lengths: every per-row
    schedule (stream-K row starts, selection grids, split partials) at its bound."""
    from tiered_mixed_precision_gb300.fade import MAX_BATCH

    kb, vb = kv
    over = dict(layers=1, batch=MAX_BATCH, num_q_heads=4, num_kv_heads=1, ragged=(90, 160),
                prompt_len=160, steps=3, middle_k_bits=kb, middle_v_bits=vb)
    if key != 2:
        over["int4_budget"] = 40
    wl = get_workload(key).scaled(**over)
    ls = Lockstep(wl)
    ls.prefill(0)
    ls.check_layer_state(0)
    for _ in range(ls.steps):
        ls.step()
    ls.check_near_ties()


@pytest.mark.parametrize("d,window,policy", [(64, 100, "h2o"), (128, 96, "position"),
                                             (128, 140, "ema")])
def test_wide_fp16_tiers_lockstep(T, d, window, policy):
    """Sink + recent windows around and past what one ring stage of the tensor-core kernel
    holds (about 100 rows): the FP16 tiers then go through the stage (tensor cores) or are
    read from global memory (CUDA cores); both against the oracle."""
    base = {"h2o": 3, "position": 4, "ema": 5}[policy]
    wl = get_workload(base).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                   head_dim=d, n_sink=8, recent_window=window, ragged=None,
                                   prompt_len=window + 400, int4_budget=200, steps=4)
    ls = Lockstep(wl)
    ls.prefill(0)
    ls.check_layer_state(0)
    for _ in range(ls.steps):
        ls.step()
    ls.check_near_ties()
