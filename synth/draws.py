"""Seeded raw draws: q, k, v as fp16 (pre-RoPE), score arrays, ragged context lengths.

Recipe (the same on both backends):
  * every value is an fp32 draw from N(0, 1), rounded to fp16 (round to nearest even);
  * outlier channels are a seeded, fixed set of channels (the same for every token, layer,
    head and row; K and V share the set when both have outliers); their fp32 draws are
    multiplied by the workload's ``outlier_scale`` before the fp16 rounding, and for the
    heavy-tailed workload they come from Student-t with 3 degrees of freedom instead;
  * q never has outliers.
RoPE is not applied here: the caller rotates q and k at their cache positions.

Two backends give the same recipe at different sizes:
  * ``"numpy"``: host arrays from ``numpy.random.Generator(PCG64)``, used where the oracle
    sees the whole input;
  * ``"torch"``: device tensors from a seeded ``torch.Generator`` on the given device, used
    for the full-size workloads; a test that checks sampled units copies the drawn slice
    of the raw input to the host for the oracle.
"""

from __future__ import annotations

import hashlib

import numpy as np

from .workloads import Workload

_KINDS = {"q": 1, "k": 2, "v": 3, "scores": 4, "ctx": 5, "mass": 6, "x": 7, "pq": 8}


def _seed(wl_seed: int, *parts) -> int:
    h = hashlib.sha256(repr((int(wl_seed),) + tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def outlier_channels(wl: Workload) -> np.ndarray:
    """Seeded fixed outlier channel indices (sorted); K uses the first ``k_outlier_channels``
    of the permutation and V the first ``v_outlier_channels``."""
    n = max(wl.k_outlier_channels, wl.v_outlier_channels)
    rng = np.random.Generator(np.random.PCG64(_seed(wl.seed, "outlier_channels")))
    return rng.permutation(wl.head_dim)[:n]


def _channel_scale(wl: Workload, kind: str):
    """Per-channel multiplier (fp32) and mask of heavy-tailed channels for ``kind``."""
    d = wl.head_dim
    scale = np.ones(d, np.float32)
    heavy = np.zeros(d, bool)
    perm = outlier_channels(wl)
    n = {"k": wl.k_outlier_channels, "v": wl.v_outlier_channels}.get(kind, 0)
    ch = perm[:n]
    scale[ch] = np.float32(wl.outlier_scale)
    if wl.outlier_dist == "student_t3":
        heavy[ch] = True
    return scale, heavy


def _numpy_draw(seed: int, shape, scale, heavy) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    z = rng.standard_normal(shape, dtype=np.float32)
    if heavy.any():
        chi = rng.standard_normal((3,) + tuple(shape), dtype=np.float32)
        chi2 = (chi * chi).sum(0, dtype=np.float32) / np.float32(3.0)
        t = z / np.sqrt(chi2, dtype=np.float32)
        z = np.where(heavy, t, z).astype(np.float32)
    return (z * scale).astype(np.float16)


def _torch_draw(seed: int, shape, scale, heavy, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if heavy.any():
        chi = torch.randn((3,) + tuple(shape), generator=g, device=device, dtype=torch.float32)
        chi2 = (chi * chi).sum(0) / 3.0
        t = z / torch.sqrt(chi2)
        hv = torch.as_tensor(heavy, device=device)
        z = torch.where(hv, t, z)
        del chi, chi2, t
    sc = torch.as_tensor(scale, device=device)
    return (z * sc).to(torch.float16)


def draw_vectors(wl: Workload, kind: str, shape, *key, backend="numpy", device=None):
    """fp16 raw draws of ``shape`` (last dim = head_dim) for q/k/v under the workload's
    outlier recipe. ``key`` selects an independent stream (layer, step, ...)."""
    scale, heavy = _channel_scale(wl, kind)
    seed = _seed(wl.seed, _KINDS[kind], *key)
    if backend == "numpy":
        return _numpy_draw(seed, tuple(shape), scale, heavy)
    if backend == "torch":
        return _torch_draw(seed, tuple(shape), scale, heavy, device)
    raise ValueError(f"unknown backend {backend!r}")


def draw_prompt(wl: Workload, layer: int, prompt_len=None, *, with_q=False,
                backend="numpy", device=None):
    """Raw prompt for one layer: k, v [B][Hkv][P][d] (and q [B][Hq][P][d] when asked)."""
    P = wl.prompt_len if prompt_len is None else prompt_len
    B, hq, hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    out = {
        "k": draw_vectors(wl, "k", (B, hkv, P, d), "prompt", layer, backend=backend, device=device),
        "v": draw_vectors(wl, "v", (B, hkv, P, d), "prompt", layer, backend=backend, device=device),
    }
    if with_q:
        out["q"] = draw_vectors(wl, "q", (B, hq, P, d), "prompt", layer, backend=backend,
                                device=device)
    return out


def draw_decode_tokens(wl: Workload, layer: int, step: int, *, backend="numpy", device=None):
    """Raw decode inputs for one layer and step: q [B][Hq][d], k, v [B][Hkv][d]."""
    B, hq, hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    return {
        "q": draw_vectors(wl, "q", (B, hq, d), "step", layer, step, backend=backend, device=device),
        "k": draw_vectors(wl, "k", (B, hkv, d), "step", layer, step, backend=backend, device=device),
        "v": draw_vectors(wl, "v", (B, hkv, d), "step", layer, step, backend=backend, device=device),
    }


def ragged_context_lengths(wl: Workload) -> np.ndarray:
    """Per-row context lengths, uniform on the workload's inclusive range (int32)."""
    if wl.ragged is None:
        return np.full(wl.batch, wl.prompt_len, np.int32)
    lo, hi = wl.ragged
    rng = np.random.Generator(np.random.PCG64(_seed(wl.seed, _KINDS["ctx"])))
    return rng.integers(lo, hi + 1, size=wl.batch).astype(np.int32)


def draw_scores(shape, seed: int, *, tie_fraction=0.25, levels=None) -> np.ndarray:
    """Non-negative fp32 score arrays with deliberate exact ties, for selection tests.

    A ``tie_fraction`` of the entries is replaced by values from a small set of levels, so
    equal keys occur and the tie rule is exercised."""
    rng = np.random.Generator(np.random.PCG64(_seed(seed, _KINDS["scores"])))
    s = rng.exponential(1.0, size=shape).astype(np.float32)
    if levels is None:
        levels = np.array([0.0, 0.25, 0.5, 1.0], np.float32)
    mask = rng.random(size=shape) < tie_fraction
    pick = rng.integers(0, len(levels), size=shape)
    return np.where(mask, levels[pick], s).astype(np.float32)


def draw_mass_like(shape, seed: int) -> np.ndarray:
    """Positive fp32 values shaped like accumulated attention mass (for prefill tests)."""
    rng = np.random.Generator(np.random.PCG64(_seed(seed, _KINDS["mass"])))
    return rng.gamma(0.5, 2.0, size=shape).astype(np.float32)


def draw_codec_cases(n_vec: int, dim: int, seed: int) -> np.ndarray:
    """fp16 [n_vec][dim] vectors for codec tests: seeded N(0,1) rows with outlier channels,
    plus rows that exercise the edge cases of an absmax grid: an all-zero group, a group
    holding only the smallest subnormal, a group whose largest magnitude is 7 (so that with
    INT4 the step is exactly 1 and the other entries sit on half-integers), negative zeros,
    and values near the fp16 maximum."""
    rng = np.random.Generator(np.random.PCG64(_seed(seed, _KINDS["x"], n_vec, dim)))
    x = rng.standard_normal((n_vec, dim), dtype=np.float32)
    x[:, rng.integers(0, dim)] *= 10.0
    x = x.astype(np.float16)
    specials = []
    z = np.zeros(dim, np.float16)
    specials.append(z.copy())                                   # all zero
    r = z.copy(); r[min(3, dim - 1)] = np.float16(2.0 ** -24); specials.append(r)
    r = np.array([7.0] + [(k % 13) - 6.0 + 0.5 for k in range(31)], np.float16)
    specials.append(np.tile(r, dim // 32)[:dim])                # half-integer steps
    r = -np.zeros(dim, np.float16); r[0] = np.float16(1.0); specials.append(r)
    r = rng.uniform(-65504, 65504, dim).astype(np.float16); specials.append(r)
    r = (rng.standard_normal(dim) * 1e-6).astype(np.float16); specials.append(r)
    for i, s in enumerate(specials):
        if i < n_vec:
            x[(i * 7919) % n_vec] = s
    return x


def pq_calibration(wl: Workload, n: int, *, backend="numpy", device=None):
    """Calibration V rows for a PQ codebook: ``n`` fp16 [n][d] draws of the workload's V
    recipe, from a stream of their own."""
    return draw_vectors(wl, "v", (n, wl.head_dim), "pq_calibration", backend=backend,
                        device=device)


def pq_init_indices(n: int, seed: int) -> np.ndarray:
    """The random draw that seeds k-means: 256 distinct row indices in [0, n) (n >= 256),
    or 256 indices with repeats when n < 256."""
    rng = np.random.Generator(np.random.PCG64(_seed(seed, _KINDS["pq"], n)))
    return rng.choice(n, size=256, replace=n < 256).astype(np.int32)


def pq_codebook(rng: np.random.Generator, head_dim: int, scale: float = 1.0) -> np.ndarray:
    """A codebook-shaped draw, fp16 [head_dim/4][256][4] from N(0, scale^2): a stand-in for a
    trained codebook where only its shape and value range matter."""
    x = rng.standard_normal((head_dim // 4, 256, 4), dtype=np.float32) * np.float32(scale)
    return x.astype(np.float16)
