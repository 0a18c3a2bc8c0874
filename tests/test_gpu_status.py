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
