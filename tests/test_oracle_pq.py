"""Pins of the oracle's product quantiser (FADE-zh §产品量化) against facts that do not come
from it: exact nearest search, hand-built ties and clusters, the rate."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import accounting, pq
from oracle.cache import Params, UnitCache
from oracle.rope import RopeTable
from synth import draws

FP16_1_2 = np.arange(0x3C00, 0x4000, dtype=np.uint16).view(np.float16)  # [1, 2)


def _separated_codebook(rng, S):
    """Centroids on a coarse lattice (multiples of 1/4 in [-8, 8)), all distinct."""
    lat = rng.choice(np.arange(-32, 32), size=(S, pq.CENTROIDS, pq.SUB)) / 4.0
    for s in range(S):
        while len({tuple(r) for r in lat[s]}) < pq.CENTROIDS:
            lat[s] = rng.choice(np.arange(-32, 32), size=(pq.CENTROIDS, pq.SUB)) / 4.0
    return lat.astype(np.float16)


def test_encode_matches_exact_nearest_search():
    rng = np.random.default_rng(11)
    S = 8
    cb = _separated_codebook(rng, S)
    x = (rng.standard_normal((400, S * pq.SUB)) * 3).astype(np.float16)
    codes = pq.encode(x, cb)
    xs = x.astype(np.float64).reshape(400, S, pq.SUB)
    d64 = ((xs[:, :, None, :] - cb.astype(np.float64)[None]) ** 2).sum(-1)  # exact in fp64
    order = np.sort(d64, axis=-1)
    clear = order[..., 1] - order[..., 0] > 1e-3 * (1 + order[..., 0])
    assert clear.mean() > 0.9
    assert np.array_equal(codes[clear], np.argmin(d64, axis=-1)[clear])


def test_ties_go_to_the_lowest_index():
    cb = np.zeros((1, pq.CENTROIDS, pq.SUB), np.float16)
    cb[0, :] = 100.0
    cb[0, 3] = [-1, 0, 0, 0]
    cb[0, 7] = [1, 0, 0, 0]       # as far from 0 as index 3
    cb[0, 200] = [-1, 0, 0, 0]    # a duplicate of index 3
    assert pq.encode(np.zeros((1, 4), np.float16), cb).tolist() == [[3]]
    x = np.array([[-1, 0, 0, 0]], np.float16)
    assert pq.encode(x, cb).tolist() == [[3]]
    x = np.array([[1, 0, 0, 0]], np.float16)
    assert pq.encode(x, cb).tolist() == [[7]]


def test_decode_layout_and_identity_on_centroids():
    rng = np.random.default_rng(5)
    S = 4
    cb = _separated_codebook(rng, S)
    # hand-worked layout: code byte s selects centroid of sub-space s for channels 4s..4s+3
    codes = np.array([[2, 0, 255, 17]], np.uint8)
    want = np.concatenate([cb[0, 2], cb[1, 0], cb[2, 255], cb[3, 17]])[None]
    assert np.array_equal(pq.decode(codes, cb), want)
    # every centroid is its own unique nearest point (distance 0, the others are distinct)
    rows = cb.transpose(1, 0, 2).reshape(pq.CENTROIDS, S * pq.SUB)   # row c = centroid c
    assert np.array_equal(pq.encode(rows, cb),
                          np.repeat(np.arange(pq.CENTROIDS, dtype=np.uint8)[:, None], S, 1))
    assert np.array_equal(pq.decode(pq.encode(rows, cb), cb), rows)


def _nearest_fp16_in_1_2(x: Fraction) -> np.float16:
    return min(FP16_1_2, key=lambda v: (abs(Fraction(float(v)) - x),
                                        int(np.array(v).view(np.uint16)) & 1))


def test_lloyd_round_hand_built_clusters():
    # one sub-space (d = 4); calibration rows in three clusters and one far row F; the 256
    # init rows are index 0 (cluster A), 3 (cluster B), 6 (cluster C), then F repeated.
    A = [[1.0, 1.5, -2, 0], [1.5, 1.0, -2, 0], [1.25, 1.25, -2, 0]]          # mean exact
    B = [[10, 10, 10, 10], [10, 10, 10, 11], [10, 10, 10, 10]]              # mean 31/3
    C = [[-9, 1, 1, 1], [-9, 1, 1, 2], [-9, 1, 1, 1], [-9, 1, 1, 1]]        # mean 5/4
    F = [[100, 100, 100, 100]]
    calib = np.array(A + B + C + F, np.float16)
    init = np.array([0, 3, 6, 10] + [10] * 252)
    cb0 = pq.init_codebook(calib, init)
    assert np.array_equal(cb0[0, 0], calib[0]) and np.array_equal(cb0[0, 1], calib[3])
    cb1 = pq.lloyd_round(calib, cb0)
    assert cb1[0, 0].tolist() == [1.25, 1.25, -2, 0]
    # 31/3 = 10.333..: fp16 spacing in [8, 16) is 2^-7; nearest is 1323 * 2^-7
    assert cb1[0, 1].tolist() == [10, 10, 10, float(Fraction(1323, 128))]
    assert cb1[0, 2].tolist() == [-9, 1, 1, 1.25]
    assert cb1[0, 3].tolist() == F[0]
    # the duplicates of F (indices 4..255) lose every tie to index 3: no members, so they
    # keep their value (neither zero nor undefined)
    assert np.array_equal(cb1[0, 4:], cb0[0, 4:]) and (cb1[0, 4:] == 100).all()
    # a second round is a fixed point (the means are their clusters' nearest centroids)
    assert np.array_equal(pq.lloyd_round(calib, cb1), cb1)
    assert np.array_equal(pq.train(calib, init, 3), cb1)


def test_lloyd_mean_rounds_to_nearest_fp16():
    # members 1, 1, 2 in channel 0: mean 4/3, rounded once to fp16 (nearest, ties even)
    calib = np.array([[1, 0, 0, 0], [1, 0, 0, 0], [2, 0, 0, 0], [50, 50, 50, 50]], np.float16)
    init = np.array([0, 3] + [3] * 254)
    cb = pq.lloyd_round(calib, pq.init_codebook(calib, init))
    assert cb[0, 0, 0] == _nearest_fp16_in_1_2(Fraction(4, 3))
    assert cb[0, 1].tolist() == [50, 50, 50, 50]


def test_rate_and_bytes():
    assert pq.bits_per_element() == 2.0
    # head_dim 128: 32 sub-spaces, 32 code bytes per token = the INT2 row; no V scales
    assert 128 // pq.SUB == 32
    assert accounting.middle_token_bytes(128, 4, 2, v_codec="pq") == 64 + 8 + 32
    assert accounting.middle_token_bytes(128, 4, 2) == 64 + 8 + 32 + 8
    assert accounting.pq_codebook_bytes(128) == 65536


def test_train_rejects_bad_init_and_sizes():
    calib = np.zeros((10, 8), np.float16)
    with pytest.raises(ValueError):
        pq.train(calib, np.arange(256), 1)             # indices beyond the rows
    with pytest.raises(ValueError):
        pq.train(calib, np.zeros(255, np.int64), 1)    # not 256 indices
    with pytest.raises(ValueError):
        pq.encode(np.zeros((1, 6), np.float16), np.zeros((1, 256, 4), np.float16))


def test_unit_cache_demotes_v_through_the_codebook():
    # wiring: with PQ V, the middle tier's values are decode(encode(v)) of the demoted tokens
    rng = np.random.default_rng(3)
    d = 64
    p = Params(d, 2, 2, 4, -1, "none", 4, 2, v_codec="pq")
    cb = _separated_codebook(rng, d // pq.SUB)
    u = UnitCache(p, RopeTable("default", d, 64, base=10000.0), codebook=cb)
    vs = []
    for t in range(12):
        q = rng.standard_normal((2, d)).astype(np.float16)
        k = rng.standard_normal(d).astype(np.float16)
        v = (rng.standard_normal(d) * 4).astype(np.float16)
        vs.append(v)
        u.step(q, k, v)
    assert u.n_sink == 2 and u.n_recent == 4 and u.n_mid == 6
    mid_v = np.array(vs[2:8])
    assert u.mid_vq.dtype == np.uint8 and u.mid_vq.shape == (6, d // 4)
    assert np.array_equal(u.values()[2:8], pq.decode(pq.encode(mid_v, cb), cb).astype(np.float64))
    assert not u.mid_vs.any()


def test_synth_codebook_draw_shape():
    cb = draws.pq_codebook(np.random.default_rng(0), 128)
    assert cb.shape == (32, 256, 4) and cb.dtype == np.float16
