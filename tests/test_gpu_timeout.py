"""A bounded device-side wait that runs out ends as a status, not a hung GPU: a barrier that nothing
arrives at gives CVR_E_TIMEOUT after about a second, and the same handle then scores correctly."""
import time

import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_the_handle_recovers():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    t0 = time.perf_counter()
    st = g.sc.selftest_wait_timeout()
    dt = time.perf_counter() - t0
    assert st == 7, g.sc.last_error()            # CVR_E_TIMEOUT
    assert "wait" in g.sc.last_error()
    assert 0.5 < dt < 30.0
    assert g.run() == 0                           # the error word was cleared; the context is usable
    assert_pcvr_close(g.out(), oracle.score(wl, w).out, "after a timeout")
