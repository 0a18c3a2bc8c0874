"""The five synthetic workloads, stated as plain shapes and tier parameters.

They stand in for the pages' model runs (Qwen2.5-3B-Instruct, Llama-3.2-1B and a
Llama-3-8B-shaped sweep). No weights or datasets are used: every tensor is a seeded draw.

Fields follow the FADE config vocabulary: ``n_sink``, ``recent_window``, ``int4_budget``,
``eviction_policy``, ``middle_k_bits``, ``middle_v_bits`` (page "FADE：面向LLM推理的注意力感知
分层KV缓存压缩技术", §自定义配置).
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional


@dataclass(frozen=True)
class Rope:
    kind: str = "default"          # "none" | "default" | "llama3" | "linear" | "ntk" | "yarn"
                                   # | "dynamic"
    base: float = 10000.0
    factor: float = 1.0            # llama3, linear, ntk, yarn, dynamic
    low_freq_factor: float = 1.0   # llama3; yarn: alpha
    high_freq_factor: float = 4.0  # llama3; yarn: beta
    original_max_position: int = 8192   # llama3, yarn, dynamic
    rotary_dim: int = 0            # proportional (partial) RoPE: rotated channels; 0 = all


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_sink: int
    recent_window: int
    int4_budget: int               # < 0: unbounded (no eviction)
    policy: str                    # "none" | "h2o" | "ema" | "position"
    middle_k_bits: int
    middle_v_bits: int
    prompt_len: int                # tokens in the cache before the first decode step
    steps: int                     # decode steps
    rope: Rope = field(default_factory=Rope)
    ema_decay: float = 0.9
    # value distribution of K/V: outlier channels and their treatment
    k_outlier_channels: int = 0    # number of outlier channels in K (fixed across tokens)
    v_outlier_channels: int = 0    # same set as K's when both are non-zero
    outlier_scale: float = 1.0     # multiplier of outlier channels (pre-RoPE)
    outlier_dist: str = "normal"   # "normal" | "student_t3"
    ragged: Optional[tuple] = None  # (lo, hi) context lengths per row, uniform, inclusive
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "Workload":
        """Copy with some fields replaced (smaller variants for fast tests)."""
        return replace(self, **kw)


# Config 1: single layer, batch 1, GQA 8/2, d=64; 512 cached tokens seen by one decode
# query. The query's own token is the 512th: a 511-token prompt, then one decode step.
W1 = Workload(
    name="single_layer_d64_ctx512", layers=1, batch=1, num_q_heads=8, num_kv_heads=2,
    head_dim=64, n_sink=4, recent_window=64, int4_budget=-1, policy="none",
    middle_k_bits=4, middle_v_bits=2, prompt_len=511, steps=1,
    rope=Rope("default", 10000.0), k_outlier_channels=4, outlier_scale=10.0, seed=101)

# Config 2: Qwen2.5-3B-shaped cache in safe mode.
W2 = Workload(
    name="qwen2.5-3b_safe_ctx4096", layers=36, batch=1, num_q_heads=16, num_kv_heads=2,
    head_dim=128, n_sink=4, recent_window=64, int4_budget=-1, policy="none",
    middle_k_bits=4, middle_v_bits=4, prompt_len=4096, steps=256,
    rope=Rope("default", 1.0e6), k_outlier_channels=1, v_outlier_channels=1,
    outlier_scale=8.0, seed=102)

# Config 3: Llama-3.2-1B-shaped cache in balanced mode (H2O, budget 400).
W3 = Workload(
    name="llama3.2-1b_balanced_h2o", layers=16, batch=8, num_q_heads=32, num_kv_heads=8,
    head_dim=64, n_sink=4, recent_window=64, int4_budget=400, policy="h2o",
    middle_k_bits=4, middle_v_bits=2, prompt_len=2048, steps=512,
    rope=Rope("llama3", 500000.0, factor=32.0, low_freq_factor=1.0, high_freq_factor=4.0,
              original_max_position=8192), seed=103)

# Config 4: Llama-3-8B-shaped throughput sweep, aggressive mode (position eviction).
W4 = Workload(
    name="llama3-8b_b64_ctx32k_position", layers=32, batch=64, num_q_heads=32,
    num_kv_heads=8, head_dim=128, n_sink=4, recent_window=64, int4_budget=4096,
    policy="position", middle_k_bits=4, middle_v_bits=2, prompt_len=32768, steps=128,
    rope=Rope("default", 500000.0), k_outlier_channels=1, v_outlier_channels=1,
    outlier_scale=1.0, outlier_dist="student_t3", seed=104)

# Config 5a: ragged long-context batch with EMA eviction capped at 16384 middle tokens.
W5 = Workload(
    name="llama3-8b_b4_ragged64k-128k_ema", layers=32, batch=4, num_q_heads=32,
    num_kv_heads=8, head_dim=128, n_sink=4, recent_window=64, int4_budget=16384,
    policy="ema", middle_k_bits=4, middle_v_bits=2, prompt_len=131072, steps=64,
    rope=Rope("default", 500000.0), k_outlier_channels=1, v_outlier_channels=1,
    outlier_scale=10.0, ragged=(65536, 131072), seed=105)

# Config 5b: the same rows with no cap (safe mode), so split-KV sees uneven lengths.
W5B = W5.scaled(name="llama3-8b_b4_ragged64k-128k_safe", int4_budget=-1, policy="none",
                seed=106)

WORKLOADS = {1: W1, 2: W2, 3: W3, 4: W4, 5: W5, "5b": W5B}


def get_workload(key) -> Workload:
    return WORKLOADS[key]
