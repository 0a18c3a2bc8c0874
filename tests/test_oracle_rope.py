"""Pins of the oracle's RoPE against facts that do not come from it."""

import math

import numpy as np
import pytest

from oracle import rope

F32 = np.float32


def _complex_rotate(x, angle):
    """Independent formulation: pairs (x_i, x_{i+d/2}) as complex numbers times e^{i angle}."""
    half = x.shape[-1] // 2
    z = (x[..., :half].astype(np.complex128) + 1j * x[..., half:]) * np.exp(1j * angle)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rotation_is_complex_multiplication():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 128))
    ang = rng.uniform(-50, 50, (64, 64))
    assert np.allclose(rope.rotate64(x, ang), _complex_rotate(x, ang), atol=1e-12, rtol=0)
    # the fp32 table variant agrees to fp32 rounding
    rt = rope.RopeTable("default", 128, 4096, base=10000.0)
    pos = rng.integers(0, 4096, 64)
    x32 = x.astype(F32)
    got = rope.rotate(x32, rt.cos[pos], rt.sin[pos]).astype(np.float64)
    ang32 = (pos.astype(F32)[:, None] * rt.inv_freq[None, :]).astype(F32).astype(np.float64)
    want = _complex_rotate(x32.astype(np.float64), ang32)
    assert np.allclose(got, want, atol=4e-6, rtol=4e-6)


def test_position_zero_is_identity():
    rt = rope.RopeTable("llama3", 64, 8, base=5e5, factor=32, low_freq_factor=1,
                        high_freq_factor=4, original_max_position=8192)
    x = np.random.default_rng(1).standard_normal((5, 64)).astype(np.float16)
    assert np.array_equal(rt.apply(x, 0).view(np.uint16), x.view(np.uint16))
    assert np.all(rt.cos[0] == 1) and np.all(rt.sin[0] == 0)


def test_inverse_of_forward_is_identity():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((32, 128))
    ang = rng.uniform(-1e4, 1e4, (32, 64))
    back = rope.rotate64(rope.rotate64(x, ang), ang, inverse=True)
    assert np.allclose(back, x, atol=1e-13, rtol=0)
    rt = rope.RopeTable("default", 128, 40000, base=5e5)
    pos = rng.integers(0, 40000, 32)
    x32 = x.astype(F32)
    c, s = rt.cos[pos], rt.sin[pos]
    back32 = rope.rotate(rope.rotate(x32, c, s), c, s, inverse=True)
    ulp = np.spacing(np.abs(x32).max())
    assert np.max(np.abs(back32 - x32)) <= 8 * ulp


def test_pair_norms_preserved():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 64))
    y = rope.rotate64(x, rng.uniform(0, 100, (16, 32)))
    n0 = x[:, :32] ** 2 + x[:, 32:] ** 2
    n1 = y[:, :32] ** 2 + y[:, 32:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13, atol=0)


def test_llama3_bands_closed_form():
    d, base, L, factor, lf, hf = 64, 5e5, 8192, 32.0, 1.0, 4.0
    default = rope.inv_freq("default", base, d)
    l3 = rope.inv_freq("llama3", base, d, factor, lf, hf, L)
    wl = 2 * math.pi / default.astype(np.float64)
    high = wl < L / hf              # short wavelengths: unchanged
    low = wl > L / lf               # long wavelengths: divided by the factor
    assert high.any() and low.any() and (~high & ~low).any()
    assert np.array_equal(l3[high], default[high])
    ratio = default[low].astype(np.float64) / l3[low].astype(np.float64)
    assert np.allclose(ratio, factor, rtol=2 ** -22)
    # the mixed band lies strictly between the two unmixed values and is monotone in i
    mid = ~high & ~low
    assert np.all(l3[mid] < default[mid]) and np.all(l3[mid] > default[mid] / factor)
    assert np.all(np.diff(l3.astype(np.float64)) < 0)


def test_linear_scaling_is_position_interpolation():
    """Linear scaling rotates position p by the unscaled angle of position p / factor."""
    d, base, factor = 128, 1e4, 4.0
    lin = rope.inv_freq("linear", base, d, factor).astype(np.float64)
    ref = rope.inv_freq("default", base, d).astype(np.float64)
    for p in (4, 400, 40000):
        assert np.allclose(p * lin, (p / factor) * ref, rtol=2 ** -22, atol=0)


def test_ntk_keeps_the_highest_and_divides_the_lowest_frequency():
    """NTK-aware scaling: pair 0 keeps frequency 1; the last pair's frequency is divided by
    exactly the factor (closed form of base * factor^(d/(d-2)) at exponent -(d-2)/d)."""
    for d, base, factor in [(64, 1e4, 8.0), (128, 5e5, 2.0)]:
        ntk = rope.inv_freq("ntk", base, d, factor).astype(np.float64)
        ref = rope.inv_freq("default", base, d).astype(np.float64)
        assert ntk[0] == 1.0 == ref[0]
        assert math.isclose(ref[-1] / ntk[-1], factor, rel_tol=2 ** -21)
        assert np.all(ntk[1:-1] < ref[1:-1]) and np.all(ntk[1:-1] > ref[1:-1] / factor)


def test_dynamic_ntk_follows_the_sequence_length():
    """Dynamic NTK: up to the original context the default frequencies; beyond it pair 0
    keeps frequency 1 and the last pair's frequency is divided by exactly
    factor * L / L0 - (factor - 1) (e.g. 2 * 16384 / 4096 - 1 = 7); longer sequences scale
    more (monotone), and the table of length L is the one RopeTable builds."""
    d, base, L0, factor = 128, 1e4, 4096, 2.0
    ref = rope.inv_freq("default", base, d).astype(np.float64)
    for L in (100, 4096):
        dyn = rope.inv_freq("dynamic", base, d, factor, original_max_position=L0, seq_len=L)
        assert np.array_equal(dyn, rope.inv_freq("default", base, d))
    prev = ref
    for L, want in ((8192, 3.0), (16384, 7.0), (40000, 2 * 40000 / 4096 - 1)):
        dyn = rope.inv_freq("dynamic", base, d, factor, original_max_position=L0,
                            seq_len=L).astype(np.float64)
        assert dyn[0] == 1.0
        assert math.isclose(ref[-1] / dyn[-1], want, rel_tol=2 ** -21)
        assert np.all(dyn[1:] < prev[1:])   # a longer sequence lowers every frequency further
        prev = dyn
    t = rope.RopeTable("dynamic", d, 16384, base=base, factor=factor, original_max_position=L0)
    assert math.isclose(ref[-1] / float(t.inv_freq[-1]), 7.0, rel_tol=2 ** -21)
    with pytest.raises(ValueError):
        rope.inv_freq("dynamic", base, d, factor, original_max_position=L0)


def test_yarn_bands_over_rotations_per_context():
    """YaRN (alpha = 1, beta = 32): pairs making more than beta rotations over the original
    context keep their frequency, pairs making fewer than alpha are interpolated by the factor,
    the ones between are blended (between the two values, monotone)."""
    d, base, L, factor, alpha, beta = 128, 1e4, 4096, 8.0, 1.0, 32.0
    yarn = rope.inv_freq("yarn", base, d, factor, alpha, beta, L)
    ref = rope.inv_freq("default", base, d)
    rot = L * ref.astype(np.float64) / (2 * math.pi)   # rotations over the original context
    keep, interp = rot > beta, rot < alpha
    assert keep.any() and interp.any() and (~keep & ~interp).any()
    assert np.array_equal(yarn[keep], ref[keep])
    assert np.allclose(ref[interp].astype(np.float64) / yarn[interp], factor, rtol=2 ** -22)
    mid = ~keep & ~interp
    assert np.all(yarn[mid] < ref[mid]) and np.all(yarn[mid] > ref[mid] / factor)
    assert np.all(np.diff(yarn.astype(np.float64)) < 0)


def test_scores_depend_only_on_relative_distance():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    inv = rope.inv_freq("default", 1e4, 128).astype(np.float64)
    dot = lambda P, j: rope.rotate64(q, P * inv) @ rope.rotate64(k, j * inv)
    for P, j, shift in [(100, 7, 13), (5000, 4000, -3000), (64, 64, 1000)]:
        assert math.isclose(dot(P, j), dot(P + shift, j + shift), rel_tol=1e-9, abs_tol=1e-9)


def test_reposition_matches_direct_rotation_to_fp16_rounding():
    rng = np.random.default_rng(5)
    rt = rope.RopeTable("default", 128, 40000, base=5e5)
    x = rng.standard_normal((200, 128)).astype(np.float16)
    old = rng.integers(1000, 40000, 200)
    new = rng.integers(0, 1000, 200)
    k_old = rt.apply(x, old)
    k_new = rt.reposition(k_old.astype(F32), old, new)
    direct = rt.apply(x, new)
    diff = np.abs(k_new.astype(np.float64) - direct.astype(np.float64))
    # two fp16 roundings on the way; a rotation mixes a pair, so the bound is a few fp16
    # ulps of the pair's norm
    dd = direct.astype(np.float64)
    r = np.sqrt(dd[:, :64] ** 2 + dd[:, 64:] ** 2)
    tol = 3 * np.spacing(r.astype(np.float16)).astype(np.float64) + 2.0 ** -24
    tol = np.concatenate([tol, tol], axis=1)
    assert np.all(diff <= tol)


# ---------------------------------------------------------------- proportional (partial) RoPE
# FADE-zh §RoPE方案兼容性 lists proportional RoPE (Gemma 4, partial_rotary_factor): only the
# first rotary_dim channels rotate, paired (i, i + rotary_dim/2), frequencies over rotary_dim.


def test_proportional_full_width_equals_standard_rope():
    full = rope.RopeTable("default", 128, 2048, base=1e4)
    same = rope.RopeTable("default", 128, 2048, base=1e4, rotary_dim=128)
    assert np.array_equal(full.cos, same.cos) and np.array_equal(full.sin, same.sin)
    x = np.random.default_rng(20).standard_normal((40, 128)).astype(np.float16)
    pos = np.arange(40) * 37
    assert np.array_equal(full.apply(x, pos).view(np.uint16), same.apply(x, pos).view(np.uint16))


@pytest.mark.parametrize("d,r", [(128, 64), (128, 96), (64, 32), (64, 48), (64, 16)])
def test_proportional_pass_through_and_closed_form(d, r):
    rt = rope.RopeTable("default", d, 5000, base=1e4, rotary_dim=r)
    assert rt.cos.shape == (5000, r // 2)
    # the frequencies are the standard ones of an r-dimensional RoPE (closed form, fp64)
    i = np.arange(r // 2, dtype=np.float64)
    assert np.array_equal(rt.inv_freq, (1e4 ** (-2.0 * i / r)).astype(F32))
    rng = np.random.default_rng(d + r)
    x = rng.standard_normal((64, d)).astype(np.float16)
    pos = rng.integers(0, 5000, 64)
    y = rt.apply(x, pos)
    # channels past the rotary width are untouched, bit for bit
    assert np.array_equal(y[:, r:].view(np.uint16), x[:, r:].view(np.uint16))
    # the rotated ones are the complex rotation of pairs (i, i + r/2) by pos * inv_freq
    ang = (pos.astype(F32)[:, None] * rt.inv_freq[None, :]).astype(F32).astype(np.float64)
    z = (x[:, :r // 2].astype(np.complex128) + 1j * x[:, r // 2:r]) * np.exp(1j * ang)
    want = np.concatenate([z.real, z.imag], axis=-1)
    assert np.allclose(y[:, :r].astype(np.float64), want, atol=2e-3, rtol=2e-3)
    # re-positioning back to the same position is the fp16 cast of the input
    same = rt.reposition(x.astype(F32), pos, pos)
    assert np.array_equal(same[:, r:].view(np.uint16), x[:, r:].view(np.uint16))


@pytest.mark.parametrize("d,r", [(128, 64), (64, 48)])
def test_proportional_scores_depend_only_on_relative_distance(d, r):
    rt = rope.RopeTable("default", d, 6000, base=1e4, rotary_dim=r)
    rng = np.random.default_rng(7)
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    inv = rt.inv_freq.astype(np.float64)
    s = []
    for shift in (0, 100, 4000):
        P, j = 1000 + shift, 900 + shift
        qr = rope.rotate64(q, P * inv)
        kr = rope.rotate64(k, j * inv)
        s.append(float(qr @ kr))
    assert np.allclose(s, s[0], atol=1e-9)
    # and the pass-through channels contribute their plain dot product at any position
    qr, kr = rope.rotate64(q, 5 * inv), rope.rotate64(k, 3 * inv)
    assert math.isclose(float(qr[r:] @ kr[r:]), float(q[r:] @ k[r:]), abs_tol=1e-12)


def test_proportional_inverse_of_forward():
    rt = rope.RopeTable("llama3", 128, 9000, base=5e5, factor=8, low_freq_factor=1,
                        high_freq_factor=4, original_max_position=8192, rotary_dim=64)
    rng = np.random.default_rng(9)
    x32 = rng.standard_normal((32, 128)).astype(F32)
    pos = rng.integers(0, 9000, 32)
    c, s = rt.cos[pos], rt.sin[pos]
    back = rope.rotate(rope.rotate(x32, c, s), c, s, inverse=True)
    assert np.array_equal(back[:, 64:], x32[:, 64:])
    assert np.max(np.abs(back - x32)) <= 8 * np.spacing(np.abs(x32).max())


def test_proportional_rejects_bad_widths():
    for r in (3, 130, -2):
        with pytest.raises(ValueError):
            rope.RopeTable("default", 128, 16, rotary_dim=r)
