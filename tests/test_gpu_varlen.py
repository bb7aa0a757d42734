"""Variable-length sequences on the CUDA path (cvr_score_varlen) against the oracle's (pinned in
test_oracle_varlen.py): pCVR within abs 2e-3 / rel 1e-2, decoded tokens against the oracle's, padding
never read, full lengths identical to the fixed-length entry point, bad lengths reported."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close, rel_close

pytestmark = pytest.mark.gpu


def _run_varlen(wl, w, lens, check=True, **cfg):
    import torch
    g = GpuRun(wl, w, debug=False, **cfg)
    d_lens = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to("cuda:0")
    r, b, o, s, out = g.dw.ptrs()
    st = g.sc.score_varlen(wl.n_req, wl.n_cand, r, b, o, s, d_lens.data_ptr(), out, check=check)
    return g, st


def _check(wl, w, lens, requests=None, stages=False, **cfg):
    import torch
    import cvr_ranking_model_gb300 as cvr
    g, st = _run_varlen(wl, w, lens, **cfg)
    ref = oracle.score(wl, w, requests=requests, seq_lens=lens, dumps=stages, **cfg)
    assert st == 0 and ref.status == 0
    if stages:
        Z = g.stage(cvr.STAGE_Z, (wl.n_cand, 16, 128), torch.bfloat16)
        last = wl.n_layers - 1
        for gi in range(3):
            rel_close(Z[:, 13 + gi], ref.dumps["Z"][last][:, 13 + gi], 0.05, f"decoded token {gi}")
    sel = np.isfinite(ref.out).all(axis=1)
    return assert_pcvr_close(g.out()[sel], ref.out[sel], wl.name + " varlen")


def test_ragged_lengths_with_garbage_padding():
    wl = synth.make_workload("tiny", n_req=5, cand_per_req=[1, 70, 3, 64, 9], seq_len=(3, 70, 129),
                             user_rows=5000, item_rows=3000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    lens = synth.make_seq_lens(wl, min_len=0, seed=11)
    lens[1] = [0, 1, 65]       # an empty group, a single event, a length past one 64-position chunk
    wl = dataclasses.replace(wl, seq_ids=synth.pad_seq_ids(wl, lens, -5))   # out-of-range padding ids
    _check(wl, w, lens, stages=True)


def test_two_layers_varlen():
    wl = synth.make_workload("deep", n_req=3, n_cand=40, seq_len=(17, 33, 65), user_rows=1000, item_rows=1000,
                             seq_rows=10_000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    _check(wl, w, synth.make_seq_lens(wl, min_len=1, seed=5), stages=True)


def test_full_lengths_identical_to_fixed_entry_point():
    wl = synth.make_workload("tiny", n_req=3, n_cand=50)
    w = synth.make_weights(wl.n_layers, wl.seed)
    full = np.tile(np.array(wl.seq_len, np.int32), (wl.n_req, 1))
    g, st = _run_varlen(wl, w, full)
    var = g.out()
    g.run()
    assert np.array_equal(var, g.out())


def test_prod_shape_sampled():
    wl = synth.make_workload("prod")
    w = synth.make_weights(wl.n_layers, wl.seed)
    lens = synth.make_seq_lens(wl, min_len=1)
    _check(wl, w, lens, requests=[0, 5])


def test_lengths_out_of_range_are_reported():
    wl = synth.make_workload("tiny", n_req=2, n_cand=4)
    w = synth.make_weights(wl.n_layers, wl.seed)
    lens = np.tile(np.array(wl.seq_len, np.int32), (wl.n_req, 1))
    lens[1, 2] = wl.seq_len[2] + 3
    g, st = _run_varlen(wl, w, lens, check=False)
    assert st == 6   # CVR_E_INPUT
    lens[1, 2] = -1
    g, st = _run_varlen(wl, w, lens, check=False)
    assert st == 6
