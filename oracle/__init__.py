"""Oracle for the FADE tiered KV cache: a plain, slow CPU restatement of what the pages define.

THIS IS TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline
leg may import it. It shares no code, header, table or constant generator with the CUDA
library under ``tiered_mixed_precision_gb300``, and neither imports the other; the only
code both sides use is the seeded input module ``synth``, which holds no cache arithmetic.

Sources (cited by page title and section in every module):
  * FADE-zh: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术" (primary).
  * FADE-en: page "FADE: Attention-Aware Hierarchical KV Cache Compression for LLM Inference".
  * KVLong: page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列"
    (§1.2 attention as a weighted average, §1.2.2 StreamingLLM, §1.3.1 H2O).

Precision: fp64 wherever the pages leave it open, except
  * RoPE, which FADE-zh §RoPE重计算 fixes at float32 math followed by a cast to the model
    dtype (fp16), and
  * the quantiser's scale and code decisions, which are taken in fp32 (IEEE division, round
    to nearest even) because those decisions produce integers and must be taken in the same
    precision as the kernel; a pinned test shows fp64 gives identical results for every
    fp16 input.

Parity status of each function is stated in its module header. Functions whose result the
pages pin only by model-quality figures (greedy match, coherence) have no parity pin and say
"parity unpinned".
"""

from . import accounting, attention, cache, policy, pq, quant, rope  # noqa: F401
