"""fade_decode_attention_noalloc, the attention call for callers that cannot allocate device
memory (an allocator-free region of a serving loop, a plugin handed only its inputs and
outputs): its split scratch is a fixed array inside the library instead of a caller-provided
workspace. Checked through the C ABI against fade_decode_attention, bit for bit, on two calls
in a row and on a smaller call after them, and for its rejection of shapes larger than the
array. Collected last on purpose."""

import numpy as np
import pytest

from harness import allclose_report
from synth import draw_prompt, draw_vectors, get_workload

pytestmark = pytest.mark.gpu


def _cache(wl):
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300.model import FadeCache

    cfg = T.Config.from_workload(wl)
    P = wl.prompt_len
    fc = FadeCache(cfg, 1, P, P + 16, "cuda")
    pr = draw_prompt(wl, 0, P)
    fc.prefill(0, torch.from_numpy(pr["k"]).cuda(), torch.from_numpy(pr["v"]).cuda())
    return T, fc


def _both(T, fc, wl, call):
    """One call of each entry point on the same query; returns both outputs and (M, L)."""
    import torch

    L = fc.layers[0]
    B, Hq, d = wl.batch, wl.num_q_heads, wl.head_dim
    q = torch.from_numpy(draw_vectors(wl, "q", (B, Hq, d), "noalloc", call)).cuda()
    out_ref = torch.empty_like(q)
    out_na = torch.full_like(q, float("nan"))
    ml_ref = torch.empty(B * Hq * 2, dtype=torch.float32, device="cuda")
    ml_na = torch.full_like(ml_ref, float("nan"))
    T.fade_decode_attention(L, q, out_ref, None, ml_ref, fc.ws)
    T.fade.fade_decode_attention_noalloc(L, q, out_na, None, ml_na)
    torch.cuda.synchronize()
    return out_ref, out_na, ml_ref, ml_na


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    """Both entry points run the same kernels with the same split count on the same inputs,
    so their results must agree bit for bit; a third call with a smaller batch and context
    follows the larger ones, so partials a larger call left in the shared array would show."""
    import torch

    wl = get_workload(4).scaled(layers=1, batch=4, num_q_heads=8, num_kv_heads=2,
                                prompt_len=2000, int4_budget=900)
    T, fc = _cache(wl)
    for call in range(2):
        out_ref, out_na, ml_ref, ml_na = _both(T, fc, wl, call)
        ok, err, nbad = allclose_report(out_na.float().cpu().numpy(),
                                        out_ref.float().cpu().numpy())
        assert ok, f"call {call}: outputs differ (max err {err}, {nbad} bad)"
        assert torch.equal(out_na.view(torch.int16), out_ref.view(torch.int16)), \
            f"call {call}: outputs are not bit-identical"
        assert torch.equal(ml_na.view(torch.int32), ml_ref.view(torch.int32)), \
            f"call {call}: softmax statistics are not bit-identical"
    small = get_workload(4).scaled(layers=1, batch=2, num_q_heads=4, num_kv_heads=1,
                                   prompt_len=700, int4_budget=300)
    T, fc_small = _cache(small)
    out_ref, out_na, ml_ref, ml_na = _both(T, fc_small, small, 2)
    assert torch.equal(out_na.view(torch.int16), out_ref.view(torch.int16)), \
        "smaller call after larger ones: outputs are not bit-identical"
    assert torch.equal(ml_na.view(torch.int32), ml_ref.view(torch.int32)), \
        "smaller call after larger ones: softmax statistics are not bit-identical"


def test_noalloc_rejects_shapes_larger_than_its_scratch():
    import torch

    # 256 rows x 64 query heads: even two splits need 256*64*2*130*4 bytes > 8 MiB
    wl = get_workload(4).scaled(layers=1, batch=256, num_q_heads=64, num_kv_heads=8,
                                prompt_len=70, int4_budget=-1, policy="none")
    T, fc = _cache(wl)
    q = torch.zeros((256, 64, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    ml = torch.empty(256 * 64 * 2, dtype=torch.float32, device="cuda")
    with pytest.raises(T.FadeError) as e:
        T.fade.fade_decode_attention_noalloc(fc.layers[0], q, out, None, ml)
    assert e.value.status == 3
    assert "fixed" in str(e.value)
