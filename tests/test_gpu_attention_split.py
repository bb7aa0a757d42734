"""Cross-attention over sequences longer than 512 positions, split over several CTAs whose softmax states
the last one merges: against the oracle, for single-request tiles (split), ragged multi-request tiles (not
split) and variable lengths that leave whole splits empty."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close, rel_close

pytestmark = pytest.mark.gpu


def _wl(**kw):
    return synth.make_workload("tiny", seq_len=(600, 1100, 1500), user_rows=3000, item_rows=3000, seq_rows=20000,
                               **kw)


def _stage_check(g, wl, ref):
    import torch
    import cvr_ranking_model_gb300 as cvr
    Z = g.stage(cvr.STAGE_Z, (wl.n_cand, 16, 128), torch.bfloat16)
    for gi in range(3):
        rel_close(Z[:, 13 + gi], ref.dumps["Z"][0][:, 13 + gi], 0.05, f"decoded token {gi}")


def test_split_sequences_single_request_tiles():
    wl = _wl(n_req=3, n_cand=64)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    g = GpuRun(wl, w, debug=False)
    g.run()
    ref = oracle.score(wl, w, dumps=True)
    _stage_check(g, wl, ref)
    assert_pcvr_close(g.out(), ref.out, "split")
    g.run()   # the merge counters were reset: a second call gives the same result
    assert_pcvr_close(g.out(), ref.out, "split, second call")


def test_ragged_tiles_are_not_split():
    wl = _wl(n_req=4, cand_per_req=[5, 40, 1, 20])
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    g.run()
    ref = oracle.score(wl, w, dumps=True)
    _stage_check(g, wl, ref)
    assert_pcvr_close(g.out(), ref.out, "ragged")


def test_split_with_variable_lengths():
    import torch
    wl = _wl(n_req=4, n_cand=32)
    w = synth.make_weights(wl.n_layers, wl.seed)
    lens = synth.make_seq_lens(wl, min_len=0, seed=9)
    lens[0] = [0, 100, 1500]   # empty group, one split used of three, every split used
    g = GpuRun(wl, w, debug=False)
    d_lens = torch.from_numpy(lens).to("cuda:0")
    r, b, o, s, out = g.dw.ptrs()
    g.sc.score_varlen(wl.n_req, wl.n_cand, r, b, o, s, d_lens.data_ptr(), out)
    ref = oracle.score(wl, w, seq_lens=lens)
    assert_pcvr_close(g.out(), ref.out, "split varlen")
