"""The PLE kernel with 8-bit weights (CVR_OPT_PLE_INT8) against the oracle.

The scheme (mixed-precision inference, iQIYI ad-CVR article, outlook section): every expert and gate row of
the PLE is held as integers q with one scale per row, scale = max|w| / 127 and q = round-half-even(w / scale);
activations stay bf16. The test makes q and the scales from the fp32 weights itself and gives the oracle
q x scale in place of those weights, so the CUDA path is held to the usual pCVR tolerance against the model it
computes (parity). Against the unquantised model the quantisation alone reaches 0.85 of the tolerance on the
full two-layer batch (CPU accuracy gate) and the bf16 activations add their own error, so there the bar is
looser: at most 0.1% of the pCVR values outside the tolerance, none beyond 1.1 times it (measured: none on
the production batch, one of 2048 at 1.03 times on the sampled two-layer requests). Cases: a ragged batch of
several row blocks, the full production batch, the two-layer shape, and switching the option off again
(bit-identical to before).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import ATOL, RTOL, GpuRun, assert_pcvr_close

pytestmark = pytest.mark.gpu


def _quantised_rows(W):
    W = np.asarray(W, np.float32).astype(np.float64)
    s = np.abs(W).max(axis=1, keepdims=True) / 127.0
    q = np.clip(np.rint(W / np.where(s > 0, s, 1.0)), -127, 127)
    return (q * s.astype(np.float32)).astype(np.float32)


def _int8_weights(w):
    wq = dict(w)
    for k in range(synth.DIMS["n_experts"]):
        wq[f"ple{k}_w"] = _quantised_rows(w[f"ple{k}_w"])
    for t in range(synth.DIMS["n_tasks"]):
        wq[f"gate{t}_w"] = _quantised_rows(w[f"gate{t}_w"])
    return wq


def _int8_run(wl, w, requests=None, graph=True):
    import cvr_ranking_model_gb300 as cvr
    g = GpuRun(wl, w, graph=graph, debug=False)
    g.sc.set_option(cvr.OPT_PLE_INT8, 1)
    g.run()
    got = g.out()
    sel = np.ones(wl.n_cand, bool) if requests is None else np.isin(wl.req_ids, requests)
    ref_q = oracle.score(wl, _int8_weights(w), requests=requests)
    assert ref_q.status == 0
    assert_pcvr_close(got[sel], ref_q.out[sel], f"{wl.name} int8 vs oracle on the quantised weights")
    ref = oracle.score(wl, w, requests=requests)
    err = np.abs(got[sel] - ref.out[sel]) / (ATOL + RTOL * np.abs(ref.out[sel]))
    assert np.mean(err > 1.0) <= 1e-3 and err.max() <= 1.1, (wl.name, float(np.mean(err > 1.0)), float(err.max()))
    return g, got


def test_quantiser_pins():
    W = np.array([[127.0, 0.5, -63.5, 1.5], [0.0, 0.0, 0.0, 0.0], [-2.0, 1.0, 0.0, 0.0]], np.float32)
    q = _quantised_rows(W)
    # scale 1: half-way values go to the even neighbour; a zero row stays zero; scale 2/127: exact endpoints
    assert np.array_equal(q[0], [127.0, 0.0, -64.0, 2.0]) and not q[1].any()
    assert q[2, 0] == -2.0 and abs(q[2, 1] - 64 * np.float32(2 / 127)) < 1e-6


def test_ragged_row_blocks():
    wl = synth.make_workload("tiny", n_req=4, cand_per_req=[129, 1, 200, 57], seq_len=(20, 33, 64),
                             user_rows=5000, item_rows=5000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05, gain_jitter=0.1)
    _int8_run(wl, w, graph=False)


def test_prod_full_batch():
    wl = synth.make_workload("prod")
    _int8_run(wl, synth.make_weights(wl.n_layers, wl.seed))


def test_deep_sampled():
    wl = synth.make_workload("deep")
    _int8_run(wl, synth.make_weights(wl.n_layers, wl.seed), requests=[0, 31])


def test_switching_back_restores_bf16_weights():
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload("tiny", n_req=2, n_cand=150)
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, graph=True, debug=False)
    g.run()
    before = g.out()
    g.sc.set_option(cvr.OPT_PLE_INT8, 1)
    g.run()
    int8 = g.out()
    g.sc.set_option(cvr.OPT_PLE_INT8, 0)
    g.run()
    assert np.array_equal(g.out(), before)
    assert not np.array_equal(int8, before)
    assert_pcvr_close(int8, oracle.score(wl, _int8_weights(w)).out, "tiny int8")
