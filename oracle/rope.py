"""RoPE tables, rotation, and re-positioning of keys (oracle).

FADE-zh §驱逐策略: evicting tokens triggers an un-RoPE of K at the old position and a re-RoPE
at the contiguous StreamingLLM position, so attention distances stay right.
FADE-zh §RoPE重计算: all RoPE math is done in float32, then cast through the model dtype.
FADE-zh §RoPE方案兼容性: standard RoPE (Qwen2/Qwen3, Mistral, ...), Llama-3.1 frequency
scaling ("llama3"); ALiBi models make re-RoPE a no-op.
KVLong §1.2.2 StreamingLLM: positions are assigned by index within the cache, so the key held
at cache index j carries rotation j.

Readings:
  * rotate-half pairing: channel i pairs with channel i + d/2, i < d/2 (the pairing of the
    model families the pages list);
  * proportional RoPE (FADE-zh §RoPE方案兼容性: Gemma 4, ``partial_rotary_factor``): only the
    first ``rotary_dim`` = factor * d channels rotate, paired as (i, i + rotary_dim/2), with
    the frequencies taken over rotary_dim (base ** (-2i/rotary_dim)); the other channels pass
    through unchanged (the published partial-rotary convention). rotary_dim = d is full RoPE;
  * inv_freq_i = base ** (-2i/d) computed in fp64 and rounded once to fp32; the llama3 rule
    adjusts it in fp64 first: wavelength lam = 2*pi/inv_freq; lam < L/hf keeps inv_freq,
    lam > L/lf divides it by ``factor``, otherwise it is mixed with
    t = (L/lam - lf)/(hf - lf) as (1-t)*inv/factor + t*inv (L = original max position);
  * angle = fp32(pos) * inv_freq in one fp32 multiply; cos and sin of that fp32 angle are
    evaluated in fp64 and rounded to fp32 (the table);
  * forward rotation: y_i = x_i*c - x_{i+d/2}*s, y_{i+d/2} = x_{i+d/2}*c + x_i*s with every
    product and sum rounded to fp32 separately (no fused multiply-add); inverse: s -> -s;
  * re-positioning: K' = fp16(forward(inverse(K, old), new)), no fp16 rounding in between.
Pinned by: rotation equals complex multiplication by exp(i*angle) to fp32 rounding,
pass-through channels bit-identical under proportional RoPE (and the full-width case equal to
standard RoPE bit for bit),
inverse-of-forward is the identity (exactly in the fp64 variant, within a few fp32 ulps in
the table variant), position 0 is the identity, pair norms are preserved, the llama3 bands
match their closed forms, and scores depend only on the relative distance.
"""

from __future__ import annotations

import math

import numpy as np

F32 = np.float32


def inv_freq(kind: str, base: float, head_dim: int, factor=1.0, low_freq_factor=1.0,
             high_freq_factor=4.0, original_max_position=8192, seq_len=None) -> np.ndarray:
    """fp32 inverse frequencies [head_dim/2] for the rotation pairs. ``head_dim`` is the
    rotated width: the rotary dimension under proportional (partial) RoPE.

    FADE-zh §RoPE方案兼容性 names the scaling types; each follows its published definition:
      * "linear" (position interpolation): every frequency divided by ``factor``, i.e. the
        positions divided by it;
      * "ntk" (NTK-aware scaling): the base raised to base * factor^(d/(d-2)), which keeps
        the highest frequency and divides the lowest by ``factor``;
      * "yarn": YaRN's ramp gamma(r) = clamp((r - alpha)/(beta - alpha), 0, 1) over the
        number of rotations r = L/lambda a pair makes over the original context L, blending
        theta/factor (gamma = 0) with theta (gamma = 1); alpha and beta come in
        ``low_freq_factor`` and ``high_freq_factor``. It is the llama3 rule with those
        boundaries. YaRN's attention temperature is left out: the table holds pure rotations;
      * "dynamic" (dynamic NTK): the ntk rule with the factor taken from the sequence length
        ``seq_len``, factor * seq_len / original_max_position - (factor - 1), once the
        sequence is longer than the original context (default frequencies before). Reading:
        ``seq_len`` is the length the table is built for, so one table serves every rotation
        and re-positioning; the rule's re-basing at every decode step is not modelled.
    """
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    b = np.float64(base)
    if kind == "ntk":
        b = b * np.power(np.float64(factor), head_dim / (head_dim - 2.0))
    if kind == "dynamic":
        if seq_len is None:
            raise ValueError("dynamic NTK needs the sequence length")
        if seq_len > original_max_position:
            f_dyn = factor * float(seq_len) / float(original_max_position) - (factor - 1.0)
            b = b * np.power(np.float64(f_dyn), head_dim / (head_dim - 2.0))
    f = np.power(b, -(2.0 * i) / head_dim)
    if kind == "linear":
        f = f / factor
    elif kind in ("llama3", "yarn"):
        lam = 2.0 * math.pi / f
        L = float(original_max_position)
        low_wl = L / low_freq_factor      # wavelengths above this: fully scaled
        high_wl = L / high_freq_factor    # wavelengths below this: unchanged
        t = (L / lam - low_freq_factor) / (high_freq_factor - low_freq_factor)
        mixed = (1.0 - t) * f / factor + t * f
        f = np.where(lam < high_wl, f, np.where(lam > low_wl, f / factor, mixed))
    elif kind not in ("default", "ntk", "dynamic"):
        raise ValueError(f"unsupported rope kind {kind!r}")
    return f.astype(F32)


def table(inv_freq32: np.ndarray, max_pos: int):
    """(cos, sin) fp32 [max_pos][d/2] for positions 0..max_pos-1."""
    pos = np.arange(max_pos, dtype=F32)[:, None]
    ang = (pos * inv_freq32[None, :]).astype(F32)             # one fp32 multiply
    a64 = ang.astype(np.float64)
    return np.cos(a64).astype(F32), np.sin(a64).astype(F32)


def rotate(x32: np.ndarray, c: np.ndarray, s: np.ndarray, inverse=False) -> np.ndarray:
    """Rotate fp32 vectors [..., d] by per-pair fp32 (cos, sin) [..., r/2]: channel i pairs
    with i + r/2 for i < r/2; channels r..d-1 pass through unchanged (r = d: full RoPE)."""
    x32 = np.asarray(x32, F32)
    half = np.shape(c)[-1]
    x1, x2, rest = x32[..., :half], x32[..., half:2 * half], x32[..., 2 * half:]
    if inverse:
        s = -s
    y1 = (x1 * c).astype(F32) - (x2 * s).astype(F32)
    y2 = (x2 * c).astype(F32) + (x1 * s).astype(F32)
    return np.concatenate([y1.astype(F32), y2.astype(F32), rest], axis=-1)


class RopeTable:
    """A model's RoPE: kind "none" makes every operation the identity (ALiBi models)."""

    def __init__(self, kind: str, head_dim: int, max_pos: int, base=10000.0, factor=1.0,
                 low_freq_factor=1.0, high_freq_factor=4.0, original_max_position=8192,
                 rotary_dim=0):
        self.kind = kind
        self.head_dim = head_dim
        self.max_pos = max_pos
        # proportional (partial) RoPE: the rotated width; 0 = every channel
        self.rotary_dim = head_dim if not rotary_dim else int(rotary_dim)
        if not (0 < self.rotary_dim <= head_dim and self.rotary_dim % 2 == 0):
            raise ValueError("rotary_dim must be even and within (0, head_dim]")
        if kind != "none":
            self.inv_freq = inv_freq(kind, base, self.rotary_dim, factor, low_freq_factor,
                                     high_freq_factor, original_max_position, seq_len=max_pos)
            self.cos, self.sin = table(self.inv_freq, max_pos)

    @classmethod
    def from_workload(cls, wl, max_pos: int) -> "RopeTable":
        r = wl.rope
        return cls(r.kind, wl.head_dim, max_pos, r.base, r.factor, r.low_freq_factor,
                   r.high_freq_factor, r.original_max_position,
                   getattr(r, "rotary_dim", 0))

    def _cs(self, pos):
        pos = np.asarray(pos, np.int64)
        if pos.size and (pos.min() < 0 or pos.max() >= self.max_pos):
            raise ValueError("position outside the RoPE table")
        return self.cos[pos], self.sin[pos]

    def apply(self, x16: np.ndarray, pos) -> np.ndarray:
        """fp16 [..., d] rotated to ``pos`` (a scalar, or one position per row of a 2-D x) -> fp16."""
        if self.kind == "none":
            return np.asarray(x16, np.float16).copy()
        c, s = self._cs(pos)
        return rotate(np.asarray(x16, np.float16).astype(F32), c, s).astype(np.float16)

    def reposition(self, x, old_pos, new_pos) -> np.ndarray:
        """Un-rotate at ``old_pos``, rotate at ``new_pos``, all in fp32, then cast to fp16.
        ``x`` is fp16 or an exactly representable fp32 (a dequantised key)."""
        if self.kind == "none":
            return np.asarray(x, F32).astype(np.float16)
        co, so = self._cs(old_pos)
        cn, sn = self._cs(new_pos)
        y = rotate(np.asarray(x, F32), co, so, inverse=True)
        return rotate(y, cn, sn).astype(np.float16)


def rotate64(x: np.ndarray, angle: np.ndarray, inverse=False) -> np.ndarray:
    """fp64 rotate-half rotation by explicit angles [..., r/2] (used by the pins only);
    channels past r pass through."""
    x = np.asarray(x, np.float64)
    half = np.shape(angle)[-1]
    c, s = np.cos(angle), np.sin(angle)
    if inverse:
        s = -s
    x1, x2, rest = x[..., :half], x[..., half:2 * half], x[..., 2 * half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s, np.broadcast_to(
        rest, np.broadcast_shapes(rest.shape, x1.shape[:-1] + (rest.shape[-1],)))], axis=-1)
