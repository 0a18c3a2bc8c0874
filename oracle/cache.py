"""The tiered KV cache of one (layer, row, KV head), step by step (oracle).

FADE-zh §核心机制 (three tiers): tier 1 keeps the first N_SINK tokens (sinks) and the last
RECENT_WINDOW tokens (recent) in FP16 (§第一层); mid-aged tokens, the bulk of the cache, are
stored 4-bit and bit-packed (§第二层); V of the middle tier may be 2-bit (§第三层,
§量化与Bit-Packing: ``middle_v_bits=2``).
FADE-zh §驱逐策略 and §RoPE重计算: when INT4_BUDGET is exceeded tokens are evicted; surviving
keys are moved to contiguous StreamingLLM positions by un-RoPE at the old position and
re-RoPE at the new one, in float32, then cast to fp16.
FADE-zh §配置预设 / §自定义配置: presets and the config fields used here.
KVLong §1.2.2 StreamingLLM: sinks plus a rolling window, positions assigned inside the cache.

Step order per decode step (reading; the pages do not order the steps):
  1. demote: if the recent window is full, its oldest token is quantised (K at
     ``middle_k_bits``, V at ``middle_v_bits``) and becomes the newest middle token; its
     index does not change;
  2. evict: if the middle tier holds more than ``int4_budget`` tokens, the excess is chosen
     by the policy among middle tokens only and dropped; every survivor whose index drops
     (middle and recent) is re-positioned: a middle key is dequantised, re-positioned in
     fp32, cast to fp16 and re-quantised; V and the scores move unchanged;
  3. append: the new token (key RoPE'd by the caller at the current held count) becomes a
     sink while fewer than ``n_sink`` sinks are held, else the newest recent token;
  4. attend: the G query heads (RoPE'd at the same position) attend to every held token,
     the new one included;
  5. accumulate: H2O or EMA scores take the step's probabilities.
``int4_budget`` counts middle tokens only; evicted tokens are dropped, not demoted further.
With ``v_codec="pq"`` (FADE-zh §产品量化, the alternative to INT2) the middle tier's V is
product-quantised with a per-layer codebook (pq.py) instead of INT{v_bits}.
Prefill (reading): the prompt's keys are RoPE'd at 0..P-1; sinks are the first n_sink, the
recent window the last recent_window, the rest are middle candidates; the excess over the
budget is evicted by the policy key (H2O: prefill attention mass, EMA: all zero, so the
oldest go first; position: the index); survivors are re-positioned in fp16 and the middle
tier is quantised once. H2O starts from the survivors' mass, EMA from zero.
Pinned through the pins of the pieces (quant, rope, attention, policy) plus: safe mode with
every token in FP16 equals textbook attention, the position-policy kept set equals the
StreamingLLM closed form, the H2O mass sum, relative-position invariance after eviction, and
the re-positioning of keys against exact fp64 rotations: every middle key moved by an
eviction equals the rotation of its previous value by its index change within s/2 plus the
fp16 and fp32 roundings, logits at unchanged distance agree within the bound that follows,
and every key held after a prefill with evictions is its raw key rotated to its cache index
(mutations of the index, the rotation or the re-quantisation fail these pins).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import attention, policy as pol, pq, quant
from .rope import RopeTable


@dataclass(frozen=True)
class Params:
    head_dim: int
    group: int              # query heads per KV head
    n_sink: int
    recent_window: int
    int4_budget: int        # < 0: unbounded
    policy: str             # "none" | "h2o" | "ema" | "position"
    k_bits: int
    v_bits: int
    ema_decay: float = 0.9
    v_codec: str = "int"    # "int": INT{v_bits} V; "pq": product-quantised V (pq.py)

    @classmethod
    def from_workload(cls, wl) -> "Params":
        return cls(wl.head_dim, wl.group, wl.n_sink, wl.recent_window, wl.int4_budget,
                   wl.policy, wl.middle_k_bits, wl.middle_v_bits, wl.ema_decay,
                   getattr(wl, "v_codec", "int"))

    @property
    def evicts(self) -> bool:
        return self.policy != "none" and self.int4_budget >= 0


class UnitCache:
    """State of one (layer, row, KV head): FP16 sinks, packed middle, FP16 recent, scores.

    Arrays are kept in cache-index (logical) order: sinks, then middle, then recent, oldest
    first. ``orig_pos`` records each held token's position in the original sequence."""

    def __init__(self, params: Params, rope: RopeTable, codebook=None):
        p = self.p = params
        d = p.head_dim
        self.rope = rope
        if p.v_codec not in ("int", "pq"):
            raise ValueError("v_codec must be 'int' or 'pq'")
        if p.v_codec == "pq" and codebook is None:
            raise ValueError("PQ-coded V needs a codebook")
        self.codebook = None if codebook is None else np.asarray(codebook, np.float16)
        self.sink_k = np.zeros((0, d), np.float16)
        self.sink_v = np.zeros((0, d), np.float16)
        self.mid_kq = np.zeros((0, d), np.int8)
        self.mid_ks = np.zeros((0, d // quant.GROUP), np.float16)
        self.mid_vq = (np.zeros((0, d // pq.SUB), np.uint8) if p.v_codec == "pq"
                       else np.zeros((0, d), np.int8))
        self.mid_vs = np.zeros((0, d // quant.GROUP), np.float16)
        self.rec_k = np.zeros((0, d), np.float16)
        self.rec_v = np.zeros((0, d), np.float16)
        self.sigma = np.zeros(0, np.float64)
        self.orig_pos = np.zeros(0, np.int64)
        self.seen = 0                      # tokens ever appended (original positions)
        self.last_victims = np.zeros(0, np.int64)

    # -- sizes -------------------------------------------------------------------------
    @property
    def n_sink(self):
        return self.sink_k.shape[0]

    @property
    def n_mid(self):
        return self.mid_kq.shape[0]

    @property
    def n_recent(self):
        return self.rec_k.shape[0]

    @property
    def n_held(self):
        return self.n_sink + self.n_mid + self.n_recent

    def pending_evictions(self) -> int:
        """Evictions the next decode step will make (after its demotion)."""
        n_mid = self.n_mid + (1 if self._ring_full() else 0)
        if self.p.evicts and n_mid > self.p.int4_budget:
            return n_mid - self.p.int4_budget
        return 0

    def next_position(self) -> int:
        """Cache position of the next decode step's token (held count before its append)."""
        return self.n_held - self.pending_evictions()

    def _ring_full(self) -> bool:
        return self.p.recent_window > 0 and self.n_recent == self.p.recent_window

    # -- dequantised views -------------------------------------------------------------
    def keys(self) -> np.ndarray:
        """All held keys as float64 [N, d] in cache order (middle dequantised)."""
        return np.concatenate([self.sink_k.astype(np.float64),
                               quant.dequantize(self.mid_kq, self.mid_ks),
                               self.rec_k.astype(np.float64)])

    def values(self) -> np.ndarray:
        if self.p.v_codec == "pq":
            mid = pq.decode(self.mid_vq, self.codebook).astype(np.float64)
        else:
            mid = quant.dequantize(self.mid_vq, self.mid_vs)
        return np.concatenate([self.sink_v.astype(np.float64), mid,
                               self.rec_v.astype(np.float64)])

    def _code_v(self, v16: np.ndarray):
        """Middle-tier V: INT codes and scales, or PQ codes and all-zero scales (a PQ row
        carries no scale; the scale slots are kept so both codecs share one layout)."""
        if self.p.v_codec == "pq":
            v16 = np.asarray(v16, np.float16)
            return (pq.encode(v16, self.codebook),
                    np.zeros((v16.shape[0], self.p.head_dim // quant.GROUP), np.float16))
        return quant.quantize(v16, self.p.v_bits)

    # -- step pieces -------------------------------------------------------------------
    def demote(self) -> bool:
        """Step 1: the oldest recent token joins the middle tier when the window is full."""
        if not self._ring_full():
            return False
        kq, ks = quant.quantize(self.rec_k[:1], self.p.k_bits)
        vq, vs = self._code_v(self.rec_v[:1])
        self.mid_kq = np.concatenate([self.mid_kq, kq])
        self.mid_ks = np.concatenate([self.mid_ks, ks])
        self.mid_vq = np.concatenate([self.mid_vq, vq])
        self.mid_vs = np.concatenate([self.mid_vs, vs])
        self.rec_k, self.rec_v = self.rec_k[1:], self.rec_v[1:]
        return True

    def choose_victims(self) -> np.ndarray:
        """Middle-tier indices (0-based within the middle tier) to evict now."""
        if not self.p.evicts or self.n_mid <= self.p.int4_budget:
            return np.zeros(0, np.int64)
        k = self.n_mid - self.p.int4_budget
        if self.p.policy == "position":
            return pol.select_victims_position(self.n_mid, k)
        s0 = self.n_sink
        return pol.select_victims(self.sigma[s0:s0 + self.n_mid], k)

    def evict(self, victims=None) -> np.ndarray:
        """Step 2: drop ``victims`` (middle indices; default: the policy's choice) and
        re-position every survivor whose cache index changes."""
        if victims is None:
            victims = self.choose_victims()
        victims = np.asarray(victims, np.int64)
        self.last_victims = victims
        if victims.size == 0:
            return victims
        s0, n_mid = self.n_sink, self.n_mid
        keep = np.ones(n_mid, bool)
        keep[victims] = False
        old_mid = s0 + np.nonzero(keep)[0]
        new_mid = s0 + np.arange(old_mid.size)
        moved = old_mid != new_mid
        kq = self.mid_kq[keep].copy()
        ks = self.mid_ks[keep].copy()
        if moved.any():
            khat = quant.dequantize(kq[moved], ks[moved]).astype(np.float32)  # exact
            k16 = self.rope.reposition(khat, old_mid[moved], new_mid[moved])
            kq[moved], ks[moved] = quant.quantize(k16, self.p.k_bits)
        shift = victims.size
        if self.n_recent:
            old_rec = s0 + n_mid + np.arange(self.n_recent)
            self.rec_k = self.rope.reposition(self.rec_k.astype(np.float32), old_rec,
                                              old_rec - shift)
        self.mid_kq, self.mid_ks = kq, ks
        self.mid_vq, self.mid_vs = self.mid_vq[keep], self.mid_vs[keep]
        drop = s0 + victims
        self.sigma = np.delete(self.sigma, drop)
        self.orig_pos = np.delete(self.orig_pos, drop)
        return victims

    def append(self, k_rot16: np.ndarray, v16: np.ndarray):
        """Step 3: the new token, its key already RoPE'd at ``n_held``."""
        k_rot16 = np.asarray(k_rot16, np.float16).reshape(1, -1)
        v16 = np.asarray(v16, np.float16).reshape(1, -1)
        if self.n_sink < self.p.n_sink:
            if self.n_mid or self.n_recent:
                raise RuntimeError("sinks must fill before any other tier")
            self.sink_k = np.concatenate([self.sink_k, k_rot16])
            self.sink_v = np.concatenate([self.sink_v, v16])
        else:
            if self.n_recent >= max(self.p.recent_window, 0) and self.p.recent_window > 0:
                raise RuntimeError("recent window overflow: demote before append")
            if self.p.recent_window == 0:
                raise RuntimeError("recent_window = 0 is not supported")
            self.rec_k = np.concatenate([self.rec_k, k_rot16])
            self.rec_v = np.concatenate([self.rec_v, v16])
        self.sigma = np.concatenate([self.sigma, [0.0]])
        self.orig_pos = np.concatenate([self.orig_pos, [self.seen]])
        self.seen += 1

    def attend(self, q_rot16: np.ndarray):
        """Step 4: q [G, d] fp16 (RoPE'd) -> (out [G, d], p [G, N], logits [G, N]) float64."""
        return attention.attend(np.asarray(q_rot16, np.float16).astype(np.float64),
                                self.keys(), self.values())

    def accumulate(self, p: np.ndarray):
        """Step 5: H2O sum or EMA update of every held token's score."""
        if self.p.policy == "h2o":
            self.sigma = pol.h2o_update(self.sigma, p)
        elif self.p.policy == "ema":
            self.sigma = pol.ema_update(self.sigma, p, self.p.ema_decay)

    def step(self, q_raw16, k_raw16, v16):
        """One decode step from raw (pre-RoPE) q [G, d], k [d], v [d].

        Returns (out [G, d] float64, p [G, N], logits [G, N], position)."""
        self.demote()
        self.evict()
        pos = self.n_held
        k_rot = self.rope.apply(np.asarray(k_raw16, np.float16).reshape(1, -1), pos)
        q_rot = self.rope.apply(np.asarray(q_raw16, np.float16), pos)
        self.append(k_rot, v16)
        out, p, logits = self.attend(q_rot)
        self.accumulate(p)
        return out, p, logits, pos

    # -- prefill -----------------------------------------------------------------------
    def prefill(self, k_raw16, v16, mass=None, select_mass=None):
        """Build the tiers from a raw prompt: k, v [P, d] fp16 (k pre-RoPE).

        ``mass`` [P] is the prefill attention mass (H2O key and initial score); it is
        required for H2O and ignored otherwise. ``select_mass`` [P], if given, is the key H2O
        selects by instead (rows sharing their decisions: the mass summed over the rows); the
        scores still start at ``mass``. Returns the evicted prompt positions."""
        if self.n_held:
            raise RuntimeError("prefill needs an empty cache")
        k_raw16 = np.asarray(k_raw16, np.float16)
        v16 = np.asarray(v16, np.float16)
        P, d = k_raw16.shape
        pos = np.arange(P)
        k_rot = self.rope.apply(k_raw16, pos)
        n_s = min(self.p.n_sink, P)
        n_r = min(self.p.recent_window, P - n_s)
        n_m = P - n_s - n_r
        cand = np.arange(n_s, n_s + n_m)
        victims = np.zeros(0, np.int64)
        if self.p.evicts and n_m > self.p.int4_budget:
            k = n_m - self.p.int4_budget
            if self.p.policy == "position":
                victims = cand[pol.select_victims_position(n_m, k)]
            elif self.p.policy == "h2o":
                if mass is None:
                    raise ValueError("H2O prefill needs the prefill attention mass")
                key = mass if select_mass is None else select_mass
                victims = cand[pol.select_victims(np.asarray(key)[cand], k)]
            else:  # EMA: every score starts at zero
                victims = cand[pol.select_victims(np.zeros(n_m), k)]
        keep = np.ones(P, bool)
        keep[victims] = False
        old = np.nonzero(keep)[0]
        new = np.arange(old.size)
        k_new = k_rot[old].copy()
        moved = old != new
        if moved.any():
            k_new[moved] = self.rope.reposition(k_rot[old[moved]].astype(np.float32),
                                                old[moved], new[moved])
        v_new = v16[old]
        m_keep = n_m - victims.size
        self.sink_k, self.sink_v = k_new[:n_s].copy(), v_new[:n_s].copy()
        mk, mv = k_new[n_s:n_s + m_keep], v_new[n_s:n_s + m_keep]
        self.mid_kq, self.mid_ks = quant.quantize(mk, self.p.k_bits)
        self.mid_vq, self.mid_vs = self._code_v(mv)
        self.rec_k = k_new[n_s + m_keep:].copy()
        self.rec_v = v_new[n_s + m_keep:].copy()
        if self.p.policy == "h2o":
            self.sigma = np.asarray(mass, np.float64)[old].copy()
        else:
            self.sigma = np.zeros(old.size, np.float64)
        self.orig_pos = old.astype(np.int64)
        self.seen = P
        return victims


def choose_shared_victims(units) -> np.ndarray:
    """Batch-shared tier decisions (FADE-zh §批处理支持: all rows share their positions and tier
    decisions): the victims of every row of one (layer, KV head), chosen once among the middle
    candidates by the sum over the rows of each candidate's score (position policy: the oldest).
    The rows must hold equal tier counts."""
    u0 = units[0]
    counts = (u0.n_sink, u0.n_mid, u0.n_recent)
    if any((u.n_sink, u.n_mid, u.n_recent) != counts for u in units):
        raise ValueError("rows sharing their decisions must hold equal tier counts")
    if not u0.p.evicts or u0.n_mid <= u0.p.int4_budget:
        return np.zeros(0, np.int64)
    k = u0.n_mid - u0.p.int4_budget
    if u0.p.policy == "position":
        return pol.select_victims_position(u0.n_mid, k)
    s0 = u0.n_sink
    keys = np.sum([u.sigma[s0:s0 + u0.n_mid] for u in units], axis=0)
    return pol.select_victims(keys, k)


def packed_state(u: UnitCache) -> dict:
    """The unit's tiers in the library's byte format (for byte-exact comparison)."""
    return {
        "sink_k": u.sink_k, "sink_v": u.sink_v,
        "mid_k_codes": quant.pack(u.mid_kq, u.p.k_bits), "mid_k_scales": u.mid_ks,
        "mid_v_codes": (u.mid_vq if u.p.v_codec == "pq" else quant.pack(u.mid_vq, u.p.v_bits)),
        "mid_v_scales": u.mid_vs,
        "recent_k": u.rec_k, "recent_v": u.rec_v, "sigma": u.sigma,
    }
