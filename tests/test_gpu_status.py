"""Device-side status words: a bounded wait that runs out is reported, not hung on.

The self-test kernel has a consumer wait on an mbarrier with the bounded wait of the attention
kernel while a producer warp, told by a host flag never to arrive, leaves it incomplete: the
wait gives up after its (short) limit, records code 1 and the kernel returns. fade_check_status
then reports FADE_ERR_TIMEOUT, and the context stays usable (an attention call afterwards
still matches the oracle)."""

import numpy as np
import pytest

from harness import Lockstep
from synth import get_workload

pytestmark = pytest.mark.gpu

FADE_ERR_TIMEOUT = 5


def test_bounded_wait_that_runs_out_is_reported_and_the_context_survives():
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300 import fade as F

    wl = get_workload(1).scaled(steps=2)
    ls = Lockstep(wl)
    ls.prefill(0)
    L = ls.fc.layers[0]
    F.fade_check_status(L)                      # clean after the prefill
    # the producer arrives: the wait completes, nothing recorded
    F.fade_selftest_bounded_wait(L.status, True, 2_000_000)
    F.fade_check_status(L)
    # the producer never arrives: a ~1 ms wait runs out and the kernel returns
    F.fade_selftest_bounded_wait(L.status, False, 2_000_000)
    with pytest.raises(T.FadeError) as e:
        F.fade_check_status(L)
    assert e.value.status == FADE_ERR_TIMEOUT
    assert "bounded wait" in str(e.value)
    assert int(L.status[0]) == 1
    # the context is still usable: clear the word and keep stepping in lockstep
    L.status.zero_()
    torch.cuda.synchronize()
    for _ in range(ls.steps):
        ls.step()
    F.fade_check_status(L)
    assert np.all(L.status.cpu().numpy() == 0)


def test_selftest_rejects_bad_arguments():
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300 import fade as F

    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    for limit in (0, -5, 10 ** 12):
        with pytest.raises(T.FadeError) as e:
            F.fade_selftest_bounded_wait(st, False, limit)
        assert e.value.status == 1


def test_debug_build_runs_a_lockstep_without_device_check_failures():
    """The FADE_DEBUG=1 library (index checks on every compacted row and attention tile) steps
    a small position-eviction cache in lockstep with the oracle in a fresh process; no check
    fires and the status words stay clear."""
    import os
    import subprocess
    import sys

    from tiered_mixed_precision_gb300 import build

    build.build(debug=True)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "from harness import Lockstep\n"
        "from synth import get_workload\n"
        "from tiered_mixed_precision_gb300 import fade as F\n"
        "assert F.LIB_PATH.endswith('_build_debug/libfade.so')\n"
        "wl = get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,\n"
        "                            prompt_len=900, int4_budget=300, steps=4)\n"
        "ls = Lockstep(wl)\n"
        "ls.prefill(0)\n"
        "for _ in range(ls.steps):\n"
        "    ls.step()\n"
        "F.fade_check_status(ls.fc.layers[0])\n"
        "print('debug lockstep ok')\n" % (root, os.path.join(root, "tests")))
    env = dict(os.environ, FADE_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "debug lockstep ok" in r.stdout


def test_device_index_guard_records_its_code_instead_of_writing_out_of_bounds():
    """A unit whose device metadata claims a full middle tier (a state the host-side checks
    exclude; planted here in the metadata) makes the demote kernel's guard skip the unit and
    record its code; fade_check_status reports FADE_ERR_DEVICE_CHECK."""
    import torch

    import tiered_mixed_precision_gb300 as T
    from tiered_mixed_precision_gb300 import fade as F

    wl = get_workload(4).scaled(layers=1, batch=2, num_q_heads=8, num_kv_heads=2,
                                prompt_len=900, int4_budget=300, steps=1)
    ls = Lockstep(wl)
    ls.prefill(0)
    L = ls.fc.layers[0]
    assert int(L.h_n_recent[0]) == wl.recent_window          # the next demote would run
    C = int(L.layout.mid_stride)
    before = L.meta.clone()
    L.meta[0, 0, 1] = C                                       # N_MID at the slot stride
    F.fade_cache_demote(L)
    with pytest.raises(T.FadeError) as e:
        F.fade_check_status(L)
    assert e.value.status == 6 and int(L.status[0]) == 16
    assert torch.equal(L.meta[0, 0], torch.tensor([int(before[0, 0, 0]), C] +
                                                  before[0, 0, 2:].tolist(), dtype=L.meta.dtype,
                                                  device=L.meta.device))
