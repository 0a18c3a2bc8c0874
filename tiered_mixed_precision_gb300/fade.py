"""ctypes binding of libfade (argument marshalling only; every step runs in the CUDA library).

The functions keep the C names (``fade_quantize_pack``, ``fade_decode_attention``, ...).
Tensors are torch tensors on a CUDA device; their data pointers and the current CUDA stream
are passed to the C entry points. A missing library raises ``ImportError``: there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# FADE_LIBRARY=debug loads the FADE_DEBUG=1 build (build.build(debug=True)) instead
LIB_PATH = os.path.join(_PKG, "_build_debug" if os.environ.get("FADE_LIBRARY") == "debug"
                        else "_build", "libfade.so")

FADE_OK, FADE_ERR_INVALID_ARGUMENT, FADE_ERR_UNSUPPORTED, FADE_ERR_CAPACITY, FADE_ERR_CUDA = range(5)
ROPE_KINDS = {"none": 0, "default": 1, "llama3": 2, "linear": 3, "ntk": 4, "yarn": 5,
              "dynamic": 6}
POLICIES = {"none": 0, "h2o": 1, "ema": 2, "position": 3}
V_CODECS = {"int": 0, "pq": 1}
PQ_SUB, PQ_CENTROIDS, PQ_MAX_CALIB = 4, 256, 8192


def pq_train_ws_bytes(dim: int) -> int:
    """FADE_PQ_TRAIN_WS_BYTES(dim)."""
    return dim * 2304 + 1024
META_FIELDS = 8
META = {"n_sink": 0, "n_mid": 1, "n_recent": 2, "head": 3, "cur": 4, "n_ev": 5, "sync": 6}
MAX_BATCH = 256
STATUS_WORDS = 4
ATTN_TILE_TOKENS = 256   # FADE_ATTN_TILE_TOKENS


class FadeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libfade status {status}: {message}")
        self.status = status


c_i32, c_i64, c_f32, c_f64, c_sz, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                          ctypes.c_double, ctypes.c_size_t, ctypes.c_void_p)


class RopeT(ctypes.Structure):
    _fields_ = [("kind", c_i32), ("original_max_position", c_i32), ("base", c_f64),
                ("factor", c_f64), ("low_freq_factor", c_f64), ("high_freq_factor", c_f64),
                ("rotary_dim", c_i32)]


class ConfigT(ctypes.Structure):
    _fields_ = [("batch", c_i32), ("num_q_heads", c_i32), ("num_kv_heads", c_i32),
                ("head_dim", c_i32), ("n_sink", c_i32), ("recent_window", c_i32),
                ("int4_budget", c_i32), ("middle_k_bits", c_i32), ("middle_v_bits", c_i32),
                ("mid_capacity", c_i32), ("policy", c_i32), ("ema_decay", c_f32),
                ("shared_rows", c_i32), ("v_codec", c_i32), ("rope", RopeT)]


class LayerT(ctypes.Structure):
    _fields_ = [("sink_k", c_vp), ("sink_v", c_vp), ("recent_k", c_vp), ("recent_v", c_vp),
                ("mid_k_codes", c_vp * 2), ("mid_k_scales", c_vp * 2),
                ("mid_v_codes", c_vp * 2), ("mid_v_scales", c_vp * 2),
                ("sink_scores", c_vp), ("mid_scores", c_vp * 2), ("recent_scores", c_vp),
                ("meta", c_vp), ("victims", c_vp), ("chunk_base", c_vp),
                ("victim_words", c_i32), ("chunk_slots", c_i32), ("status", c_vp),
                ("h_n_sink", c_vp), ("h_n_mid", c_vp), ("h_n_recent", c_vp),
                ("pq_codebook", c_vp)]


class LayoutT(ctypes.Structure):
    _fields_ = [(n, c_sz) for n in (
        "sink_k", "sink_v", "recent_k", "recent_v", "mid_k_codes", "mid_k_scales",
        "mid_v_codes", "mid_v_scales", "sink_scores", "mid_scores", "recent_scores", "meta",
        "victims", "chunk_base", "status", "logits_ws")] + [("mid_stride", c_i32)] + [
        (n, c_sz) for n in ("ml_ws", "attn_ws")] + [
        ("victim_words", c_i32), ("chunk_slots", c_i32), ("max_prompt", c_i32),
        ("max_splits", c_i32), ("prefill_mass_ws", c_sz)]


_lib = None


def lib():
    """The loaded libfade (ImportError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libfade is not built ({LIB_PATH} missing): run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        S = ctypes.POINTER
        sig = {
            "fade_layout": (c_i32, [S(ConfigT), c_i32, S(LayoutT)]),
            "fade_rope_table_init": (c_i32, [S(ConfigT), c_vp, c_i32, c_vp]),
            "fade_rope_apply": (c_i32, [S(ConfigT), c_vp, c_i32, c_vp, c_vp, c_i64, c_i32,
                                        c_vp, c_i32, c_vp]),
            "fade_quantize_pack": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_vp, c_vp, c_vp]),
            "fade_dequantize": (c_i32, [c_vp, c_vp, c_i64, c_i32, c_i32, c_vp, c_vp]),
            "fade_cache_reset": (c_i32, [S(ConfigT), S(LayerT), c_vp]),
            "fade_cache_prefill": (c_i32, [S(ConfigT), S(LayerT), c_vp, c_vp, c_i32, c_vp,
                                           c_vp, c_vp, c_i32, c_vp]),
            "fade_prefill_mass": (c_i32, [S(ConfigT), c_vp, c_vp, c_i32, c_vp, c_vp, c_vp,
                                          c_sz, c_vp]),
            "fade_cache_demote": (c_i32, [S(ConfigT), S(LayerT), c_vp]),
            "fade_evict_rerope": (c_i32, [S(ConfigT), S(LayerT), c_vp, c_i32, c_vp]),
            "fade_cache_append": (c_i32, [S(ConfigT), S(LayerT), c_vp, c_vp, c_vp]),
            "fade_rope_append": (c_i32, [S(ConfigT), S(LayerT), c_vp, c_i32, c_vp, c_vp, c_vp,
                                         c_vp, c_vp, c_i32, c_vp]),
            "fade_decode_attention": (c_i32, [S(ConfigT), S(LayerT), c_vp, c_vp, c_vp, c_vp,
                                              c_vp, c_sz, c_vp]),
            "fade_h2o_accumulate": (c_i32, [S(ConfigT), S(LayerT), c_vp, c_vp, c_vp]),
            "fade_next_position": (c_i32, [S(ConfigT), S(LayerT), c_i32]),
            "fade_compressed_bytes": (ctypes.c_uint64, [S(ConfigT), S(LayerT)]),
            "fade_cache_advance_host": (c_i32, [S(ConfigT), S(LayerT)]),
            "fade_cache_advance_host_layers": (c_i32, [S(ConfigT), c_vp, c_i32]),
            "fade_pq_encode": (c_i32, [c_vp, c_vp, c_i64, c_i32, c_vp, c_vp]),
            "fade_pq_decode": (c_i32, [c_vp, c_vp, c_i64, c_i32, c_vp, c_vp]),
            "fade_pq_train": (c_i32, [c_vp, c_i64, c_i32, c_vp, c_i32, c_vp, c_vp, c_sz, c_vp]),
            "fade_check_status": (c_i32, [S(LayerT), c_vp]),
            "fade_tier_counts": (c_i32, [S(ConfigT), S(LayerT), c_vp]),
            "fade_attention_tiled": (c_i32, [S(ConfigT)]),
            "fade_measure_fp32_rate": (c_i32, [c_i32, c_i32, c_vp, ctypes.POINTER(c_f64), c_vp]),
            "fade_selftest_bounded_wait": (c_i32, [c_vp, c_i32, c_i64, c_vp]),
            "fade_last_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def fade_last_error() -> str:
    return lib().fade_last_error().decode()


def _check(status: int):
    if status != FADE_OK:
        raise FadeError(status, fade_last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_raw_stream = None


def _stream(stream):
    """The handle of ``stream``, or of the current CUDA stream (the raw-handle query when
    torch has it: it skips building a Stream object on every call)."""
    global _raw_stream
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    import torch

    if _raw_stream is None:
        fn = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream = ((lambda: fn(torch.cuda.current_device())) if fn is not None
                       else (lambda: torch.cuda.current_stream().cuda_stream))
    return ctypes.c_void_p(_raw_stream())


# --------------------------------------------------------------------------- config
@dataclass
class Config:
    """One layer's cache configuration (the FadeConfig fields plus shapes)."""
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_sink: int = 4
    recent_window: int = 64
    int4_budget: int = -1
    middle_k_bits: int = 4
    middle_v_bits: int = 2
    mid_capacity: int = 0
    policy: str = "none"
    ema_decay: float = 0.9
    rope_kind: str = "default"
    rope_base: float = 10000.0
    rope_factor: float = 1.0
    rope_low_freq_factor: float = 1.0
    rope_high_freq_factor: float = 4.0
    rope_original_max_position: int = 8192
    rope_rotary_dim: int = 0   # proportional RoPE: rotated channels (0 = every channel)
    shared_rows: bool = False  # the rows share their tier decisions (row-summed scores)
    v_codec: str = "int"       # "pq": product-quantised middle V (needs middle_v_bits = 2)
    _c: ConfigT = field(default=None, init=False, repr=False, compare=False)

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_c":   # any change of a field invalidates the cached C struct
            object.__setattr__(self, "_c", None)

    def c(self) -> ConfigT:
        """The C struct (built once per set of field values: every entry point takes it)."""
        if self._c is None:
            r = RopeT(ROPE_KINDS[self.rope_kind], self.rope_original_max_position,
                      self.rope_base, self.rope_factor, self.rope_low_freq_factor,
                      self.rope_high_freq_factor, self.rope_rotary_dim)
            object.__setattr__(self, "_c", ConfigT(
                self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim, self.n_sink,
                self.recent_window, self.int4_budget, self.middle_k_bits, self.middle_v_bits,
                self.mid_capacity, POLICIES[self.policy], self.ema_decay,
                int(self.shared_rows), V_CODECS[self.v_codec], r))
        return self._c

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def evicts(self):
        return self.policy != "none" and self.int4_budget >= 0

    @classmethod
    def from_workload(cls, wl, mid_capacity=None, batch=None) -> "Config":
        evicts = wl.policy != "none" and wl.int4_budget >= 0
        if mid_capacity is None:
            if evicts:
                mid_capacity = wl.int4_budget + 1
            else:
                longest = wl.ragged[1] if wl.ragged else wl.prompt_len
                mid_capacity = max(1, longest + wl.steps - wl.n_sink - wl.recent_window)
        r = wl.rope
        return cls(batch or wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.n_sink,
                   wl.recent_window, wl.int4_budget, wl.middle_k_bits, wl.middle_v_bits,
                   mid_capacity, wl.policy, wl.ema_decay, r.kind, r.base, r.factor,
                   r.low_freq_factor, r.high_freq_factor, r.original_max_position,
                   getattr(r, "rotary_dim", 0))


def preset(name: str, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
           **kw) -> Config:
    """The pages' presets as configurations: "safe" (no eviction, INT4 K and V), "balanced"
    (H2O, budget 400, INT4 K / INT2 V), "aggressive" (position eviction, INT4 K / INT2 V,
    budget 4096 unless given)."""
    base = dict(batch=batch, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, n_sink=4, recent_window=64)
    if name == "safe":
        base.update(policy="none", int4_budget=-1, middle_k_bits=4, middle_v_bits=4)
    elif name == "balanced":
        base.update(policy="h2o", int4_budget=400, middle_k_bits=4, middle_v_bits=2)
    elif name == "aggressive":
        base.update(policy="position", int4_budget=4096, middle_k_bits=4, middle_v_bits=2)
    else:
        raise ValueError(f"unknown preset {name!r}")
    base.update(kw)
    if "mid_capacity" not in kw:
        base["mid_capacity"] = base["int4_budget"] + 1 if base["int4_budget"] >= 0 else 8192
    return Config(**base)


def fade_layout(cfg: Config, max_prompt: int) -> LayoutT:
    out = LayoutT()
    _check(lib().fade_layout(ctypes.byref(cfg.c()), max_prompt, ctypes.byref(out)))
    return out


# --------------------------------------------------------------------------- layer buffers
class TieredLayer:
    """Device buffers of one layer (torch-allocated) plus the host mirror of tier counts."""

    def __init__(self, cfg: Config, max_prompt: int, device="cuda"):
        import torch

        self.cfg = cfg
        self.layout = lay = fade_layout(cfg, max_prompt)
        B, H, d = cfg.batch, cfg.num_kv_heads, cfg.head_dim
        S, W, C = cfg.n_sink, cfg.recent_window, lay.mid_stride
        dev = torch.device(device)
        u8, f16, f32, i32 = torch.uint8, torch.float16, torch.float32, torch.int32
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=dev)
        self.sink_k = z((B, H, S, d), f16)
        self.sink_v = z((B, H, S, d), f16)
        self.recent_k = z((B, H, W, d), f16)
        self.recent_v = z((B, H, W, d), f16)
        self.mid_k_codes = [z((B, H, C, d * cfg.middle_k_bits // 8), u8) for _ in range(2)]
        self.mid_k_scales = [z((B, H, C, d // 32), f16) for _ in range(2)]
        self.mid_v_codes = [z((B, H, C, d * cfg.middle_v_bits // 8), u8) for _ in range(2)]
        self.mid_v_scales = [z((B, H, C, d // 32), f16) for _ in range(2)]
        self.sink_scores = z((B, H, max(S, 0)), f32)
        self.mid_scores = [z((B, H, C), f32) for _ in range(2)]
        self.recent_scores = z((B, H, W), f32)
        self.meta = z((B, H, META_FIELDS), i32)
        self.victims = z((B, H, lay.victim_words), torch.int32)
        self.chunk_base = z((B, H, lay.chunk_slots), i32)
        self.status = z((STATUS_WORDS,), i32)
        self.h_n_sink = np.zeros(B, np.int32)
        self.h_n_mid = np.zeros(B, np.int32)
        self.h_n_recent = np.zeros(B, np.int32)
        # the layer's PQ codebook (product-quantised V only): fp16 [d/4][256][4]
        self.pq_codebook = z((d // PQ_SUB, PQ_CENTROIDS, PQ_SUB), f16) if cfg.v_codec == "pq" else None
        self.pq_codebook_set = False   # PQ: encoding needs a codebook installed first
        p = lambda t: t.data_ptr()
        self.c = LayerT(
            p(self.sink_k), p(self.sink_v), p(self.recent_k), p(self.recent_v),
            (c_vp * 2)(*map(p, self.mid_k_codes)), (c_vp * 2)(*map(p, self.mid_k_scales)),
            (c_vp * 2)(*map(p, self.mid_v_codes)), (c_vp * 2)(*map(p, self.mid_v_scales)),
            p(self.sink_scores), (c_vp * 2)(*map(p, self.mid_scores)), p(self.recent_scores),
            p(self.meta), p(self.victims), p(self.chunk_base), lay.victim_words,
            lay.chunk_slots, p(self.status), self.h_n_sink.ctypes.data, self.h_n_mid.ctypes.data,
            self.h_n_recent.ctypes.data,
            None if self.pq_codebook is None else p(self.pq_codebook))

    def set_pq_codebook(self, codebook):
        """Copy a codebook (fp16 [d/4][256][4], e.g. from fade_pq_train) into the layer."""
        if self.pq_codebook is None:
            raise ValueError("the layer does not use product-quantised V")
        self.pq_codebook.copy_(codebook)
        self.pq_codebook_set = True

    def workspaces(self):
        """(logits_ws, ml_ws, attn_ws) tensors sized by the layout."""
        import torch

        dev = self.meta.device
        lay = self.layout
        return (torch.empty(lay.logits_ws // 4, dtype=torch.float32, device=dev),
                torch.empty(lay.ml_ws // 4, dtype=torch.float32, device=dev),
                torch.empty(lay.attn_ws, dtype=torch.uint8, device=dev))


# --------------------------------------------------------------------------- entry points
def fade_rope_table_init(cfg: Config, table, max_pos: int, stream=None):
    _check(lib().fade_rope_table_init(ctypes.byref(cfg.c()), _ptr(table), max_pos, _stream(stream)))


def fade_rope_apply(cfg: Config, table, max_pos, x, y, n_groups, group_len, pos_start=None,
                    pos_step=1, stream=None):
    _check(lib().fade_rope_apply(ctypes.byref(cfg.c()), _ptr(table), max_pos, _ptr(x), _ptr(y),
                                 n_groups, group_len, _ptr(pos_start), pos_step, _stream(stream)))


def fade_quantize_pack(x, n_vec, dim, bits, codes, scales, stream=None):
    _check(lib().fade_quantize_pack(_ptr(x), n_vec, dim, bits, _ptr(codes), _ptr(scales),
                                    _stream(stream)))


def fade_dequantize(codes, scales, n_vec, dim, bits, out, stream=None):
    _check(lib().fade_dequantize(_ptr(codes), _ptr(scales), n_vec, dim, bits, _ptr(out),
                                 _stream(stream)))


def fade_cache_reset(layer: TieredLayer, stream=None):
    _check(lib().fade_cache_reset(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                  _stream(stream)))


def _require_codebook(layer: TieredLayer):
    if layer.pq_codebook is not None and not layer.pq_codebook_set:
        raise ValueError("product-quantised V: install the layer's codebook first "
                         "(set_pq_codebook, or FadeCache.train_pq_codebook)")


def fade_cache_prefill(layer: TieredLayer, k_rot, v, max_prompt, prompt_len, mass, table,
                       max_pos, stream=None):
    _require_codebook(layer)
    lens = np.ascontiguousarray(prompt_len, np.int32)
    _check(lib().fade_cache_prefill(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                    _ptr(k_rot), _ptr(v), max_prompt, lens.ctypes.data,
                                    _ptr(mass), _ptr(table), max_pos, _stream(stream)))


def fade_prefill_mass(cfg: Config, q_rot, k_rot, max_prompt, prompt_len, mass, ws=None,
                      stream=None):
    """ws: device workspace of at least layout(cfg, max_prompt).prefill_mass_ws bytes (made
    here when not given)."""
    lens = np.ascontiguousarray(prompt_len, np.int32)
    if ws is None:
        import torch

        ws = torch.empty(fade_layout(cfg, max_prompt).prefill_mass_ws, dtype=torch.uint8,
                         device=q_rot.device)
    nbytes = ws.numel() * ws.element_size()
    _check(lib().fade_prefill_mass(ctypes.byref(cfg.c()), _ptr(q_rot), _ptr(k_rot), max_prompt,
                                   lens.ctypes.data, _ptr(mass), _ptr(ws), nbytes,
                                   _stream(stream)))


def fade_cache_demote(layer: TieredLayer, stream=None):
    _require_codebook(layer)
    _check(lib().fade_cache_demote(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                   _stream(stream)))


def fade_evict_rerope(layer: TieredLayer, table, max_pos, stream=None):
    _check(lib().fade_evict_rerope(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                   _ptr(table), max_pos, _stream(stream)))


def fade_cache_append(layer: TieredLayer, k_rot, v, stream=None):
    _check(lib().fade_cache_append(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                   _ptr(k_rot), _ptr(v), _stream(stream)))


def fade_rope_append(layer: TieredLayer, table, max_pos, q_raw, k_raw, v, pos, q_rot,
                     demote=False, stream=None):
    """RoPE of q_raw into q_rot and of k_raw at pos[b] (device i32 [B]), and the append of the
    rotated key and v, in one launch (the same bits as fade_rope_apply twice and
    fade_cache_append); demote: fade_cache_demote first, in the same launch."""
    _check(lib().fade_rope_append(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                  _ptr(table), max_pos, _ptr(q_raw), _ptr(k_raw), _ptr(v),
                                  _ptr(pos), _ptr(q_rot), int(bool(demote)), _stream(stream)))


def fade_decode_attention(layer: TieredLayer, q_rot, out, logits_ws, ml_ws, ws, stream=None):
    _check(lib().fade_decode_attention(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                       _ptr(q_rot), _ptr(out), _ptr(logits_ws), _ptr(ml_ws),
                                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def fade_h2o_accumulate(layer: TieredLayer, logits_ws, ml_ws, stream=None):
    _check(lib().fade_h2o_accumulate(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                     _ptr(logits_ws), _ptr(ml_ws), _stream(stream)))


def fade_next_position(layer: TieredLayer, row: int) -> int:
    r = lib().fade_next_position(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c), row)
    if r < 0:
        raise FadeError(FADE_ERR_INVALID_ARGUMENT, fade_last_error())
    return r


def fade_cache_advance_host(layer: TieredLayer):
    _check(lib().fade_cache_advance_host(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c)))


def layer_pointer_array(layers):
    """A host array of the layers' C structs (for fade_cache_advance_host_layers); it stays
    valid while the layers live."""
    arr = (ctypes.POINTER(LayerT) * len(layers))(*[ctypes.pointer(L.c) for L in layers])
    return arr


def fade_cache_advance_host_layers(cfg: "Config", layer_array, n_layers: int):
    """fade_cache_advance_host for every layer of ``layer_array`` (``layer_pointer_array``)."""
    _check(lib().fade_cache_advance_host_layers(ctypes.byref(cfg.c()), layer_array, n_layers))


def fade_compressed_bytes(layer: TieredLayer) -> int:
    return int(lib().fade_compressed_bytes(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c)))


def fade_decode_attention_noalloc(layer: TieredLayer, q_rot, out, logits_ws, ml_ws, stream=None):
    """Decode attention with the split scratch inside the library (no workspace argument), for
    callers that cannot allocate device memory; see include/fade.h for its limits."""
    fn = lib().fade_decode_attention_noalloc
    fn.restype = c_i32
    fn.argtypes = [ctypes.POINTER(ConfigT), ctypes.POINTER(LayerT), c_vp, c_vp, c_vp, c_vp, c_vp]
    _check(fn(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c), _ptr(q_rot), _ptr(out),
              _ptr(logits_ws), _ptr(ml_ws), _stream(stream)))


def fade_pq_encode(codebook, x, n_vec, dim, codes, stream=None):
    _check(lib().fade_pq_encode(_ptr(codebook), _ptr(x), n_vec, dim, _ptr(codes),
                                _stream(stream)))


def fade_pq_decode(codebook, codes, n_vec, dim, out, stream=None):
    _check(lib().fade_pq_decode(_ptr(codebook), _ptr(codes), n_vec, dim, _ptr(out),
                                _stream(stream)))


def fade_pq_train(calib, n_vec, dim, init_idx, iters, codebook, ws, stream=None):
    """``init_idx``: 256 host row indices (any int sequence); ``ws``: a device tensor of at
    least pq_train_ws_bytes(dim) bytes."""
    idx = np.ascontiguousarray(init_idx, np.int32)
    if idx.shape != (PQ_CENTROIDS,):
        raise ValueError("init_idx must hold 256 indices")
    _check(lib().fade_pq_train(_ptr(calib), n_vec, dim, idx.ctypes.data, iters, _ptr(codebook),
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def fade_check_status(layer: TieredLayer, stream=None):
    """Synchronise the stream and raise FadeError (status 5, FADE_ERR_TIMEOUT) if a kernel of
    the layer gave up a bounded wait since the last reset."""
    _check(lib().fade_check_status(ctypes.byref(layer.c), _stream(stream)))


def fade_selftest_bounded_wait(status, producer_arrives: bool, limit_cycles: int, stream=None):
    """Launch the bounded-wait self-test kernel (status: a device int32 tensor)."""
    _check(lib().fade_selftest_bounded_wait(_ptr(status), int(bool(producer_arrives)),
                                            int(limit_cycles), _stream(stream)))


def fade_measure_fp32_rate(blocks: int, iters: int, sink, stream=None) -> float:
    """Launch the fp32-rate measurement kernel; returns the fp32 operations it performs."""
    ops = c_f64(0.0)
    _check(lib().fade_measure_fp32_rate(int(blocks), int(iters), _ptr(sink), ctypes.byref(ops),
                                        _stream(stream)))
    return ops.value


def fade_attention_tiled(cfg: Config) -> bool:
    """Whether decode attention for ``cfg`` runs the tensor-core kernel, whose launch is
    scheduled from every row's count of ATTN_TILE_TOKENS-token middle tiles (the host mirror
    at the call), so that a captured call stays valid only while those counts are unchanged."""
    r = lib().fade_attention_tiled(ctypes.byref(cfg.c()))
    if r < 0:
        raise FadeError(FADE_ERR_INVALID_ARGUMENT, fade_last_error())
    return bool(r)


def fade_tier_counts(layer: TieredLayer) -> np.ndarray:
    """Per-row (sinks, middle, recent) token counts from the host mirror: i32 [B][3]."""
    out = np.zeros((layer.cfg.batch, 3), np.int32)
    _check(lib().fade_tier_counts(ctypes.byref(layer.cfg.c()), ctypes.byref(layer.c),
                                  out.ctypes.data))
    return out
