"""The allocation-free prediction entry point (cvr_predict_noalloc) against the full scoring entry point.

cvr_score runs the whole forward pass; its last Token Mixer output (CVR_STAGE_Y) is handed to
cvr_predict_noalloc, whose PLE + heads must give the same pCVR within the scoring path's tolerance, on
two calls in a row (the fixed scratch array is reused: its error word must come back clean). The file is named to be collected last, so it also runs after every other GPU test.
"""
import numpy as np
import pytest

import synth
from gpu_util import ATOL, RTOL, GpuRun

pytestmark = pytest.mark.gpu


def _y_of_last_call(g):
    import torch
    import cvr_ranking_model_gb300 as cvr
    y = torch.empty((g.wl.n_cand, 16, 128), dtype=torch.bfloat16, device="cuda:0")
    g.sc.debug_stage(cvr.STAGE_Y, y.data_ptr(), y.numel() * y.element_size())
    return y


def _close(a, b, what):
    err = np.abs(a - b)
    bound = ATOL + RTOL * np.abs(b)
    assert np.all(np.isfinite(a)), f"{what}: non-finite output"
    assert np.all(err <= bound), f"{what}: max |d| = {err.max():.3e}"


@pytest.mark.parametrize("name,kw", [
    ("tiny", dict()),
    ("tiny", dict(n_req=5, cand_per_req=[1, 70, 3, 64, 9], seq_len=(3, 70, 129), user_rows=5000, item_rows=3000)),
    ("deep", dict(n_req=3, n_cand=40, seq_len=(17, 33, 65), user_rows=1000, item_rows=1000, seq_rows=10_000)),
    ("prod", dict(n_req=2)),  # 1024 candidates: the largest batch the fixed scratch holds
])
def test_noalloc_prediction_matches_scoring_entry_point(name, kw):
    import torch
    wl = synth.make_workload(name, **kw)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    g = GpuRun(wl, w, debug=False)
    g.run()
    ref = g.out()
    y = _y_of_last_call(g)
    for call in range(2):
        out = torch.full((wl.n_cand, 2), float("nan"), dtype=torch.float32, device="cuda:0")
        g.sc.predict_noalloc(wl.n_cand, y.data_ptr(), out.data_ptr())
        _close(out.cpu().numpy().astype(np.float64), ref, f"{name} call {call}")


@pytest.mark.parametrize("name,kw", [
    ("tiny", dict(n_req=3, cand_per_req=[150, 2, 33])),
    ("prod", dict(n_req=2)),
])
def test_noalloc_prediction_on_8bit_weights(name, kw):
    """With CVR_OPT_PLE_INT8 both entry points run the PLE on the 8-bit rows: the same pCVR within tolerance."""
    import torch
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload(name, **kw)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    g = GpuRun(wl, w, debug=False)
    g.sc.set_option(cvr.OPT_PLE_INT8, 1)
    g.run()
    ref = g.out()
    y = _y_of_last_call(g)
    out = torch.full((wl.n_cand, 2), float("nan"), dtype=torch.float32, device="cuda:0")
    g.sc.predict_noalloc(wl.n_cand, y.data_ptr(), out.data_ptr())
    _close(out.cpu().numpy().astype(np.float64), ref, f"{name} int8")


def test_noalloc_rejects_oversize_and_misaligned_and_accepts_empty():
    import torch
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    g.run()
    n = cvr.NOALLOC_MAX_CAND + 1
    y = torch.zeros((n, 16, 128), dtype=torch.bfloat16, device="cuda:0")
    out = torch.zeros((n, 2), dtype=torch.float32, device="cuda:0")
    st = g.sc.predict_noalloc(n, y.data_ptr(), out.data_ptr(), check=False)
    assert st == 2  # CVR_E_SHAPE
    assert str(cvr.NOALLOC_MAX_CAND) in g.sc.last_error()
    assert g.sc.predict_noalloc(4, y.data_ptr() + 2, out.data_ptr(), check=False) == 1  # CVR_E_ARG
    assert g.sc.predict_noalloc(0, y.data_ptr(), out.data_ptr(), check=False) == 0
    # the handle still scores afterwards
    g.run()
    y4 = _y_of_last_call(g)
    out4 = torch.zeros((wl.n_cand, 2), dtype=torch.float32, device="cuda:0")
    g.sc.predict_noalloc(wl.n_cand, y4.data_ptr(), out4.data_ptr())
    _close(out4.cpu().numpy().astype(np.float64), g.out(), "after rejected calls")
