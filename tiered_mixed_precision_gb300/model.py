"""Multi-layer tiered KV cache driven through the libfade C ABI.

A decode step of one layer enqueues, in the method's order: RoPE of the new q and k at the
next cache position, demote (quantise-pack the token leaving the recent window), evict +
re-position, append, decode attention, and H2O / EMA accumulation. Everything runs in the
CUDA library on the caller's stream; this module only allocates buffers and passes pointers.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import fade as F

_cudart = None


def _record_event(ev):
    """Record a timing event on the current stream; inside a CUDA-graph capture it becomes an
    external event node (cudaEventRecordExternal), whose timestamps the host can read after
    each replay."""
    if not torch.cuda.is_current_stream_capturing():
        ev.record()
        return
    global _cudart
    if _cudart is None:
        _cudart = ctypes.CDLL("libcudart.so.13", mode=ctypes.RTLD_GLOBAL)
        _cudart.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                      ctypes.c_uint]
        _cudart.cudaEventRecordWithFlags.restype = ctypes.c_int
    rc = _cudart.cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                          1)  # cudaEventRecordExternal
    if rc != 0:
        raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")


class FadeCache:
    """All layers of one model's cache (layers share a config, a RoPE table and workspaces)."""

    def __init__(self, cfg: F.Config, num_layers: int, max_prompt: int, max_pos: int,
                 device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.layers = [F.TieredLayer(cfg, max_prompt, self.device) for _ in range(num_layers)]
        self.max_pos = max_pos
        self.max_prompt = max_prompt
        self.table = None
        if cfg.rope_kind != "none":
            self.table = torch.empty(max_pos * cfg.head_dim, dtype=torch.float32, device=self.device)
            F.fade_rope_table_init(cfg, self.table, max_pos)
        self.logits, self.ml, self.ws = self.layers[0].workspaces()
        self.pos = torch.zeros(cfg.batch, dtype=torch.int32, device=self.device)
        self._pos_host = torch.zeros(cfg.batch, dtype=torch.int32).pin_memory() \
            if self.device.type == "cuda" else torch.zeros(cfg.batch, dtype=torch.int32)
        self.needs_logits = cfg.policy in ("h2o", "ema")
        # rotated copies of the step's q and k (the caller's raw inputs stay intact)
        self.q_rot = torch.empty((cfg.batch, cfg.num_q_heads, cfg.head_dim), dtype=torch.float16,
                                 device=self.device)
        self.k_rot = torch.empty((cfg.batch, cfg.num_kv_heads, cfg.head_dim),
                                 dtype=torch.float16, device=self.device)
        # RoPE and the append (and, without eviction, the demotion) in one launch for layers of
        # at most FUSED_PROLOGUE_UNITS units, where launch latency dominates (measured faster at
        # 2, 32 and 64 units); larger layers keep the separate launches (faster at 512 units,
        # where they spread the same work over more threads)
        self.fused_prologue = cfg.batch * cfg.num_kv_heads <= self.FUSED_PROLOGUE_UNITS
        self.timers = None      # optional {"attention": [...], "evict": [...]} of event pairs
        self._graph_events = []  # timing events referenced by captured graphs
        self.launches = 0       # kernels enqueued by step_layer calls
        self._pos_ring, self._pos_ring_ev, self._pos_ring_i = None, None, 0
        self._growing = None        # (key, graph) of growing_step
        self.growing_captures = 0   # captures made by growing_step

    # ------------------------------------------------------------------ session persistence
    # Page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §会话持久化: the compressed cache is
    # saved and restored (cache_state_dict / load_cache_state_dict, then torch.save / torch.load).
    FUSED_PROLOGUE_UNITS = 128

    _STATE_BUFFERS = ("sink_k", "sink_v", "recent_k", "recent_v", "mid_k_codes", "mid_k_scales",
                      "mid_v_codes", "mid_v_scales", "sink_scores", "mid_scores", "recent_scores",
                      "meta")
    _CONFIG_FIELDS = ("batch", "num_q_heads", "num_kv_heads", "head_dim", "n_sink",
                      "recent_window", "int4_budget", "middle_k_bits", "middle_v_bits",
                      "mid_capacity", "policy", "ema_decay", "rope_kind", "rope_base",
                      "rope_factor", "rope_low_freq_factor", "rope_high_freq_factor",
                      "rope_original_max_position", "rope_rotary_dim", "shared_rows", "v_codec")

    def cache_state_dict(self) -> dict:
        """Every layer's tier buffers (both middle buffers and the device metadata, which says
        which one is live) and host tier counts, copied to host memory, with the configuration
        and sizes; only tensors, numbers and strings, so torch.load(weights_only=True) reads
        it. Pending work on the current stream is finished first."""
        layers = []
        for L in self.layers:
            d = {}
            for name in self._STATE_BUFFERS:
                v = getattr(L, name)
                d[name] = [t.cpu() for t in v] if isinstance(v, list) else v.cpu()
            for name in ("h_n_sink", "h_n_mid", "h_n_recent"):
                d[name] = torch.from_numpy(getattr(L, name).copy())
            if L.pq_codebook is not None:
                d["pq_codebook"] = L.pq_codebook.cpu()
            layers.append(d)
        return {"config": {f: getattr(self.cfg, f) for f in self._CONFIG_FIELDS},
                "num_layers": len(self.layers), "max_prompt": self.max_prompt,
                "max_pos": self.max_pos, "layers": layers}

    def load_cache_state_dict(self, sd: dict):
        """Restore a state saved by cache_state_dict into this cache, which must have been made
        with the same configuration, layer count and sizes (ValueError otherwise)."""
        mine = {f: getattr(self.cfg, f) for f in self._CONFIG_FIELDS}
        if sd["config"] != mine:
            raise ValueError(f"configuration differs: saved {sd['config']}, this cache {mine}")
        if (sd["num_layers"], sd["max_prompt"], sd["max_pos"]) != (
                len(self.layers), self.max_prompt, self.max_pos):
            raise ValueError("layer count, max_prompt or max_pos differs from the saved cache")
        for L, d in zip(self.layers, sd["layers"]):
            for name in self._STATE_BUFFERS:
                dst, src = getattr(L, name), d[name]
                for t, u in (zip(dst, src) if isinstance(dst, list) else [(dst, src)]):
                    if t.shape != u.shape or t.dtype != u.dtype:
                        raise ValueError(f"buffer {name}: saved {tuple(u.shape)} {u.dtype}, "
                                         f"this cache {tuple(t.shape)} {t.dtype}")
                    t.copy_(u)
            for name in ("h_n_sink", "h_n_mid", "h_n_recent"):
                getattr(L, name)[:] = d[name].numpy()  # in place: the C struct points at them
            if L.pq_codebook is not None:
                L.set_pq_codebook(d["pq_codebook"])
        torch.cuda.synchronize(self.device)

    # ------------------------------------------------------------------ PQ codebooks
    # Page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §产品量化: V can be product-quantised
    # with a codebook trained from calibration vectors (256 centroids, uint8 codes).
    def set_pq_codebook(self, codebook: torch.Tensor, layer=None):
        """Install a codebook (fp16 [d/4][256][4]) in one layer, or in every layer."""
        for L in (self.layers if layer is None else [self.layers[layer]]):
            L.set_pq_codebook(codebook)

    def train_pq_codebook(self, calib: torch.Tensor, init_idx, iters: int, layer=None):
        """Train a codebook on the GPU from calibration V rows (fp16 [n][d], n <= 8192; the
        256 start rows ``init_idx`` are the caller's random draw) and install it in one layer
        or every layer. Returns the codebook."""
        d = self.cfg.head_dim
        cb = torch.empty((d // F.PQ_SUB, F.PQ_CENTROIDS, F.PQ_SUB), dtype=torch.float16,
                         device=self.device)
        ws = torch.empty(F.pq_train_ws_bytes(d), dtype=torch.uint8, device=self.device)
        F.fade_pq_train(calib, calib.shape[0], d, init_idx, iters, cb, ws)
        self.set_pq_codebook(cb, layer)
        return cb

    # ------------------------------------------------------------------ pieces
    def rope_(self, x: torch.Tensor, n_groups: int, group_len: int, pos_start=None, pos_step=1):
        """Rotate x in place (fp16 [n_groups][group_len][d])."""
        F.fade_rope_apply(self.cfg, self.table, self.max_pos, x, x, n_groups, group_len,
                          pos_start, pos_step)
        return x

    def prefill(self, layer: int, k_raw: torch.Tensor, v: torch.Tensor, prompt_len=None,
                mass: torch.Tensor | None = None, q_raw: torch.Tensor | None = None):
        """k_raw, v: fp16 [B][Hkv][P][d] device tensors (k pre-RoPE; rotated in place).

        For H2O either ``mass`` (f32 [B][Hkv][P]) is given, or ``q_raw`` (fp16 [B][Hq][P][d],
        pre-RoPE, rotated in place) and the prefill attention mass is computed on the GPU.
        Returns the mass the prefill used (None when it used none)."""
        c = self.cfg
        B, H, P, d = k_raw.shape
        if prompt_len is None:
            prompt_len = np.full(B, P, np.int32)
        self.rope_(k_raw, B * H, P, None, 1)
        if mass is None and q_raw is not None and c.policy == "h2o":
            self.rope_(q_raw, B * c.num_q_heads, P, None, 1)
            mass = torch.empty((B, H, P), dtype=torch.float32, device=k_raw.device)
            F.fade_prefill_mass(c, q_raw, k_raw, P, prompt_len, mass)
        L = self.layers[layer]
        F.fade_cache_reset(L)
        F.fade_cache_prefill(L, k_raw, v, P, prompt_len, mass, self.table, self.max_pos)
        return mass

    def next_positions(self) -> np.ndarray:
        L = self.layers[0]
        return np.array([F.fade_next_position(L, b) for b in range(self.cfg.batch)], np.int32)

    def set_positions(self, pos: np.ndarray):
        self._pos_host.copy_(torch.from_numpy(np.ascontiguousarray(pos, np.int32)))
        self.pos.copy_(self._pos_host, non_blocking=True)

    def maintain_layer(self, layer: int):
        """The part of a layer's decode step that precedes the append: demote (quantise-pack the
        token leaving the recent window) and evict + re-position."""
        c = self.cfg
        L = self.layers[layer]
        ring_full = bool((L.h_n_recent == c.recent_window).any())
        F.fade_cache_demote(L)
        n = 1 if ring_full else 0
        evicting = c.evicts and bool((L.h_n_mid > c.int4_budget).any())
        t = self._tick("evict") if evicting else None
        F.fade_evict_rerope(L, self.table, self.max_pos)
        self._tock(t)
        n += (2 if c.policy == "position" else 3) if evicting else 0
        self.launches += n

    def attend_layer(self, layer: int, q_raw: torch.Tensor, k_raw: torch.Tensor,
                     v: torch.Tensor, out: torch.Tensor, demote: bool = False):
        """The rest of a layer's decode step: RoPE of the new q and k (into work buffers) at the
        positions last set by ``set_positions`` and the append of the new token (with
        ``demote`` the demotion first), in one launch (``fade_rope_append``) when the layer is
        small (``fused_prologue``), else as separate launches; attention; H2O / EMA
        accumulation."""
        c = self.cfg
        L = self.layers[layer]
        if self.fused_prologue:
            F.fade_rope_append(L, self.table, self.max_pos, q_raw, k_raw, v, self.pos,
                               self.q_rot, demote=demote)
            n = 1
        else:
            if demote:
                F.fade_cache_demote(L)
            F.fade_rope_apply(c, self.table, self.max_pos, q_raw, self.q_rot, c.batch,
                              c.num_q_heads, self.pos, 0)
            F.fade_rope_apply(c, self.table, self.max_pos, k_raw, self.k_rot, c.batch,
                              c.num_kv_heads, self.pos, 0)
            F.fade_cache_append(L, self.k_rot, v)
            n = (1 if demote else 0) + (3 if c.rope_kind != "none" else 1)
        t = self._tick("attention")
        F.fade_decode_attention(L, self.q_rot, out, self.logits if self.needs_logits else None,
                                self.ml, self.ws)
        self._tock(t)
        n += 3
        if self.needs_logits:
            t = self._tick("accumulate")
            F.fade_h2o_accumulate(L, self.logits, self.ml)
            self._tock(t)
            n += 1
        self.launches += n

    def step_layer(self, layer: int, q_raw: torch.Tensor, k_raw: torch.Tensor, v: torch.Tensor,
                   out: torch.Tensor):
        """One decode step of one layer in the method's order: demote, evict + re-position,
        append, attention, accumulation. q_raw [B][Hq][d], k_raw/v [B][Hkv][d] fp16, pre-RoPE;
        out [B][Hq][d] fp16. A cache that never evicts has nothing between its demotion and
        its append, so both go into the RoPE + append launch."""
        if not self.cfg.evicts:
            self.attend_layer(layer, q_raw, k_raw, v, out, demote=True)
            return
        self.maintain_layer(layer)
        self.attend_layer(layer, q_raw, k_raw, v, out)

    def mirror(self):
        """Host mirror of the tier counts of every layer (for steady-state checks)."""
        return [(L.h_n_sink.copy(), L.h_n_mid.copy(), L.h_n_recent.copy()) for L in self.layers]

    def step_all(self, q, k, v, out):
        """One decode step of every layer: q [L][B][Hq][d], k/v [L][B][Hkv][d], out like q."""
        self.set_positions(self.next_positions())
        for layer in range(len(self.layers)):
            self.step_layer(layer, q[layer], k[layer], v[layer], out[layer])

    def maintain_all(self):
        """Every layer's maintenance for the coming step (the prologue of pipelined steps)."""
        for layer in range(len(self.layers)):
            self.maintain_layer(layer)

    def step_all_pipelined(self, q, k, v, out, side):
        """One decode step of every layer whose maintenance was already done (by
        ``maintain_all`` or the previous pipelined step): each layer attends on the current
        stream, then its maintenance for the NEXT step is issued on a side stream and overlaps
        the following layers. ``side``: one stream, or several taken in turn by layer (so that
        one layer's short maintenance launches overlap the next layer's), or None (issued
        inline, no overlap). Per layer the operations run in the same order as ``step_all``;
        the step ends when every side stream has finished."""
        self.set_positions(self.next_positions())
        main = torch.cuda.current_stream()
        sides = [] if side is None else (list(side) if isinstance(side, (list, tuple)) else [side])
        for layer in range(len(self.layers)):
            self.attend_layer(layer, q[layer], k[layer], v[layer], out[layer])
            if not sides:
                self.maintain_layer(layer)
                continue
            st = sides[layer % len(sides)]
            ev = torch.cuda.Event()
            ev.record(main)
            st.wait_event(ev)
            with torch.cuda.stream(st):
                self.maintain_layer(layer)
        for st in sides[:len(self.layers)]:  # the streams some layer used (joined back)
            done = torch.cuda.Event()
            done.record(st)
            main.wait_event(done)

    def capture_step(self, q, k, v, out, side=None, pipelined: bool = False):
        """Capture step_all (or step_all_pipelined, with ``pipelined`` or a side stream) on fixed
        input/output buffers as a CUDA graph.

        Valid only in steady state, where a step leaves every tier count unchanged (the cache
        holds its budget; each step demotes one token, evicts one and appends one): the
        launch shapes are then the same every step and the kernels follow the device-side
        metadata (ring head, live buffer). Raises if a step would change the counts."""
        before = self.mirror()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if side is None and not pipelined:
                self.step_all(q, k, v, out)
            else:
                self.step_all_pipelined(q, k, v, out, side)
        # the graph records into the timing events captured above: they must outlive it
        if self.timers:
            self._graph_events.append({n: list(p) for n, p in self.timers.items()})
        after = self.mirror()
        for a, b in zip(before, after):
            if any((x != y).any() for x, y in zip(a, b)):
                raise RuntimeError("capture_step needs a steady-state cache (tier counts changed)")
        return g

    # ------------------------------------------------------------------ host-fed steps
    def prepare_host_pipeline(self, side=None):
        """Capture the two step graphs ``run_from_host`` alternates between (steady state
        only, see ``capture_step``): each reads its own q/k/v buffers and writes its own output
        buffer, so one step's inputs can be copied in while the other graph runs."""
        if getattr(self, "_host_pipe", None) is not None:
            return
        c, L, dev = self.cfg, len(self.layers), self.device
        shp_q = (L, c.batch, c.num_q_heads, c.head_dim)
        shp_kv = (L, c.batch, c.num_kv_heads, c.head_dim)
        bufs = []
        for _ in range(2):
            qb = torch.zeros(shp_q, dtype=torch.float16, device=dev)
            kb = torch.zeros(shp_kv, dtype=torch.float16, device=dev)
            vb = torch.zeros(shp_kv, dtype=torch.float16, device=dev)
            ob = torch.empty(shp_q, dtype=torch.float16, device=dev)
            bufs.append((qb, kb, vb, ob))
        graphs = [self.capture_step(qb, kb, vb, ob, side) for qb, kb, vb, ob in bufs]
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
        self._host_pipe = {"graphs": graphs, "bufs": bufs, "copy": torch.cuda.Stream(device=dev),
                           "in_ready": ev(), "done": ev(), "out_copied": ev(),
                           "out_used": [False, False]}

    def run_from_host(self, qh, kh, vh, oh, side=None):
        """K decode steps fed from host memory: qh [K][L][B][Hq][d], kh/vh [K][L][B][Hkv][d]
        (pinned, fp16) in, oh like qh (pinned) out. Step s+1's inputs are copied to the device
        on a copy stream while step s runs (the two captured graphs of
        ``prepare_host_pipeline`` take the steps in turn), and step s's outputs are copied back
        while step s+1 runs. Enqueued on the current stream, which waits for the last output
        copy: synchronise it (or record an event on it) to know the outputs have arrived."""
        self.prepare_host_pipeline(side)
        P = self._host_pipe
        main, cs = torch.cuda.current_stream(), P["copy"]
        K = qh.shape[0]
        if K == 0:
            return

        def copy_in(s, j):
            qb, kb, vb, _ = P["bufs"][j]
            qb.copy_(qh[s], non_blocking=True)
            kb.copy_(kh[s], non_blocking=True)
            vb.copy_(vh[s], non_blocking=True)
            P["in_ready"][j].record(cs)

        start = torch.cuda.Event()
        start.record(main)
        cs.wait_event(start)                   # nothing of this call starts before the caller's work
        with torch.cuda.stream(cs):
            copy_in(0, 0)
        for s in range(K):
            j, jn = s % 2, (s + 1) % 2
            if s + 1 < K:
                with torch.cuda.stream(cs):
                    if s >= 1:                 # the other graph (step s-1) has read its inputs
                        cs.wait_event(P["done"][jn])
                    copy_in(s + 1, jn)
            main.wait_event(P["in_ready"][j])
            if P["out_used"][j]:               # step s-2's outputs have left the buffer
                main.wait_event(P["out_copied"][j])
            P["graphs"][j].replay()
            P["done"][j].record(main)
            with torch.cuda.stream(cs):
                cs.wait_event(P["done"][j])
                oh[s].copy_(P["bufs"][j][3], non_blocking=True)
                P["out_copied"][j].record(cs)
            P["out_used"][j] = True
        main.wait_event(P["out_copied"][(K - 1) % 2])

    # ------------------------------------------------------------------ growing caches
    def growing_graph_ok(self) -> bool:
        """A step of this cache can be captured and replayed while the cache grows: no
        eviction, and every row with full sinks and a full recent window, so that each step
        demotes one token and appends one in every row (see ``growing_graph_key`` for when a
        captured step has to be captured again)."""
        c = self.cfg
        if c.evicts:
            return False
        return all(bool((L.h_n_sink == c.n_sink).all() and (L.h_n_recent == c.recent_window).all())
                   for L in self.layers)

    def growing_graph_key(self) -> tuple:
        """What a captured growing step depends on beyond the device-side counts: every
        layer's and row's number of middle tiles at the coming step's attention call (after its
        demotion: one more middle token), from which the attention launch's stream-K schedule
        is built (empty if a configuration's launch were not scheduled by tiles)."""
        tiled = getattr(self, "_attn_tiled", None)
        if tiled is None:   # a property of the configuration: asked once
            tiled = self._attn_tiled = bool(F.fade_attention_tiled(self.cfg))
        if not tiled or not self.layers:
            return ()
        # one array operation for all layers (this runs on the host before every replay)
        t = F.ATTN_TILE_TOKENS
        tiles = ((np.concatenate([L.h_n_mid for L in self.layers]).astype(np.int64) + t) //
                 t).tolist()
        B = len(tiles) // len(self.layers)
        return tuple(tuple(tiles[i * B:(i + 1) * B]) for i in range(len(self.layers)))

    def capture_growing_step(self, q, k, v, out):
        """Capture every layer's step (positions excluded: ``replay_growing`` sets them) as a
        CUDA graph for a cache that grows by one token a step (see ``growing_graph_ok``).
        The host mirror is left as it was before the capture."""
        if not self.growing_graph_ok():
            raise RuntimeError("capture_growing_step needs a growing cache without eviction "
                               "and with full sinks and recent windows")
        before = self.mirror()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for layer in range(len(self.layers)):
                self.step_layer(layer, q[layer], k[layer], v[layer], out[layer])
        for L, (s, m, r) in zip(self.layers, before):
            L.h_n_sink[:], L.h_n_mid[:], L.h_n_recent[:] = s, m, r
        return g

    def growing_step(self, q, k, v, out):
        """One step of a growing cache (``growing_graph_ok``) on fixed buffers through a
        captured graph: captured on the first call and again whenever the buffers or
        ``growing_graph_key`` change (a row's middle tier reaching a new tile, with the
        tensor-core kernel), replayed otherwise."""
        key = (tuple(x.data_ptr() for x in (q, k, v, out)), self.growing_graph_key())
        if self._growing is None or self._growing[0] != key:
            self._growing = None  # the previous graph is released before the next capture
            self._growing = (key, self.capture_growing_step(q, k, v, out))
            self.growing_captures += 1
        self.replay_growing(self._growing[1])

    def replay_growing(self, graph):
        """One step from a graph of ``capture_growing_step``: the positions (from the host
        mirror) are copied in through a ring of pinned buffers, the graph is replayed, and the
        host mirror advances by the step's count changes."""
        if self._pos_ring is None:
            self._pos_ring = [torch.zeros(self.cfg.batch, dtype=torch.int32).pin_memory()
                              for _ in range(4)]
            self._pos_ring_ev = [None] * 4
        i = self._pos_ring_i
        self._pos_ring_i = (i + 1) % len(self._pos_ring)
        if self._pos_ring_ev[i] is not None:
            self._pos_ring_ev[i].synchronize()   # the copy that last read this buffer is done
        buf = self._pos_ring[i]
        buf.copy_(torch.from_numpy(self.next_positions()))
        self.pos.copy_(buf, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record()
        self._pos_ring_ev[i] = ev
        graph.replay()
        if getattr(self, "_layer_array", None) is None:
            self._layer_array = F.layer_pointer_array(self.layers)
        F.fade_cache_advance_host_layers(self.cfg, self._layer_array, len(self.layers))

    def _tick(self, name):
        if self.timers is None:
            return None
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if torch.cuda.is_current_stream_capturing():
            # create the events outside the capture (they are created on first record)
            side = torch.cuda.Stream()
            e0.record(side)
            e1.record(side)
        _record_event(e0)
        self.timers.setdefault(name, []).append((e0, e1))
        return e1

    @staticmethod
    def _tock(e1):
        if e1 is not None:
            _record_event(e1)

    def attention_only(self, layer: int, q_rot: torch.Tensor, out: torch.Tensor):
        F.fade_decode_attention(self.layers[layer], q_rot, out,
                                self.logits if self.needs_logits else None, self.ml, self.ws)

    # ------------------------------------------------------------------ inspection
    def unit_state(self, layer: int, row: int, head: int) -> dict:
        """One unit's tiers copied to the host, in cache order (for tests and debugging)."""
        L = self.layers[layer]
        m = L.meta[row, head].cpu().numpy()
        n_sink, n_mid, n_rec, head_slot, cur = (int(m[i]) for i in range(5))
        W = self.cfg.recent_window
        ring = [(head_slot + i) % W for i in range(n_rec)]
        g = lambda t: t[row, head].cpu()
        rk, rv, rs = g(L.recent_k), g(L.recent_v), g(L.recent_scores)
        return {
            "n_sink": n_sink, "n_mid": n_mid, "n_recent": n_rec, "cur": cur,
            "sink_k": g(L.sink_k)[:n_sink].numpy(), "sink_v": g(L.sink_v)[:n_sink].numpy(),
            "mid_k_codes": g(L.mid_k_codes[cur])[:n_mid].numpy(),
            "mid_k_scales": g(L.mid_k_scales[cur])[:n_mid].numpy(),
            "mid_v_codes": g(L.mid_v_codes[cur])[:n_mid].numpy(),
            "mid_v_scales": g(L.mid_v_scales[cur])[:n_mid].numpy(),
            "recent_k": rk[ring].numpy(), "recent_v": rv[ring].numpy(),
            "scores": np.concatenate([g(L.sink_scores)[:n_sink].numpy(),
                                      g(L.mid_scores[cur])[:n_mid].numpy(),
                                      rs[ring].numpy()]),
        }
