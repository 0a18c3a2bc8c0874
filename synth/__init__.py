"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the benchmark.

This package holds workload shapes and random draws only. It contains none of the tiered
cache's arithmetic (no quantisation, no RoPE, no attention): everything it returns is a raw
fp16 draw or a plain shape description, so both sides of a parity test start from identical
bytes without sharing any method code.
"""

from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401
from .draws import (  # noqa: F401
    draw_codec_cases,
    draw_mass_like,
    draw_decode_tokens,
    draw_prompt,
    draw_scores,
    draw_vectors,
    outlier_channels,
    ragged_context_lengths,
)
