"""Failure detection on the GPU without faulting it: the onesweep sort's
look-back wait is bounded; made to run out (it waits on a partition that
never publishes), it records SS_ERR_TIMEOUT in the workspace status word,
returns, and leaves the context usable."""
import time

import pytest

import synth

pytestmark = pytest.mark.gpu


def test_lookback_wait_gives_up_and_reports():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_differentiable_gb300 as ss
    import parity
    ws = torch.empty(ss.ss_workspace_bytes(0, 2 * 4096, 16, 16), dtype=torch.uint8, device="cuda")
    t0 = time.time()
    ss.ss_test_sort_wait_timeout(ws)
    st = ss.ss_sort_status(ws)
    dt = time.time() - t0
    assert st == 4, ss.ss_last_error()          # SS_ERR_TIMEOUT
    assert "look-back" in ss.ss_last_error()
    assert dt < 10.0
    # the context still works: a full path run matches the oracle
    parity.full_parity(synth.make_scene(1))
