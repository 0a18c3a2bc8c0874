"""Host-side logic of bench.py without a GPU: the max-over-ranks timing across two gloo
ranks, and the reference arm's JSON line (the oracle timed on host cores)."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        q.put((rank, bench.max_over_ranks(10.0 + rank * 5.0, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "1", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_byte_accounting_follows_the_oracle():
    """The bench's algorithmic bytes per middle token (INT and PQ V) and per accumulate call
    agree with the oracle's accounting and the definition of the score update."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    from oracle import accounting
    import tiered_mixed_precision_gb300 as T

    for d, kb, vb, codec in [(128, 4, 2, "int"), (64, 4, 4, "int"), (128, 2, 2, "int"),
                             (128, 4, 2, "pq")]:
        cfg = T.Config(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=d, middle_k_bits=kb,
                       middle_v_bits=vb, mid_capacity=64, v_codec=codec)
        assert bench.mid_token_bytes(cfg) == accounting.middle_token_bytes(d, kb, vb,
                                                                           v_codec=codec)

    class _L:  # host mirrors only
        h_n_sink = np.array([4, 4], np.int32)
        h_n_mid = np.array([100, 50], np.int32)
        h_n_recent = np.array([64, 10], np.int32)

    cfg = T.Config(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, mid_capacity=128)
    held = (4 + 100 + 64 + 4 + 50 + 10) * 2          # token-heads held
    # G = 4 logits read, a score read and written, per held token; (M, L) per query head
    assert bench.accumulate_bytes(cfg, _L) == held * (4 * 4 + 8) + 2 * 8 * 8
