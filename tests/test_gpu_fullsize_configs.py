"""Lockstep at the workloads' stated sizes (every unit of every layer, every decode step) for
the Qwen2.5-3B-shaped safe cache and the Llama-3.2-1B-shaped H2O cache, and the ragged
64k-128k safe batch at its full lengths on sampled units; the oracle's units run in worker
processes (parallel_lockstep). Near-tie selections (fp32 vs fp64 keys) are adopted from the
GPU and counted; they must stay within 1 % of the unit-steps."""

import numpy as np
import pytest

from parallel_lockstep import ParallelLockstep
from synth import get_workload

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_driver_on_a_reduced_h2o_cache():
    """The parallel driver itself on a small H2O case (GPU prefill mass, every unit)."""
    wl = get_workload(3).scaled(layers=2, batch=2, prompt_len=700, int4_budget=200, steps=24)
    ParallelLockstep(wl, workers=3).run(check_every=8)


def test_qwen25_3b_safe_cache_every_unit():
    """Config 2 in full: 36 layers, 16/2 heads, d 128, batch 1, prompt 4096, 256 decode steps
    (each demotes one token: INT4 K and V), every (layer, KV head) unit."""
    ParallelLockstep(get_workload(2)).run(check_every=64)


def test_llama32_1b_h2o_cache_every_unit():
    """Config 3 in full: 16 layers, batch 8, 32/8 heads, d 64, prompt 2048, budget 400, H2O
    seeded from the GPU's own prefill mass, llama3 RoPE, 512 decode steps, every unit."""
    ParallelLockstep(get_workload(3)).run(check_every=128)


def test_ragged_long_context_safe_batch_sampled_units():
    """Config 5b at its full ragged lengths (64k-128k per row, batch 4, 32/8 heads, d 128, no
    cap), 64 decode steps; four layers of the full shape, two sampled units in each."""
    wl = get_workload("5b").scaled(layers=4)
    rng = np.random.default_rng(55)
    units = sorted({(l, int(rng.integers(wl.batch)), int(rng.integers(wl.num_kv_heads)))
                    for l in range(wl.layers) for _ in range(2)})
    ParallelLockstep(wl, units=units).run(check_every=16)
