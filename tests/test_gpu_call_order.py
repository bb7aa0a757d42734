"""The two call orders of the forward pass.

A small sequence encoder leaves SMs free, and the tokeniser then runs on a second stream next to the
encoder and its column sums (9 launches with the user-side GEMV as a kernel of its own); the attention
adds the first layer's mean-pooled query term. Per-kernel profiling, and an encoder that fills the GPU,
keep the one-stream order (8 launches), where the tokeniser adds that term itself. Both orders must match
the oracle, and their first-layer queries must agree up to one bf16 rounding.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close, rel_close

pytestmark = pytest.mark.gpu


def test_two_stream_and_one_stream_orders_agree():
    import torch
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload("tiny", n_req=5, cand_per_req=[1, 70, 3, 64, 9], seq_len=(3, 70, 129),
                             user_rows=5000, item_rows=3000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    ref = oracle.score(wl, w, dumps=True)
    g = GpuRun(wl, w, debug=False)

    g.run()
    assert g.sc.last_launch_count() == 7, "a small encoder forks: the tokeniser runs on the side stream"
    two = g.out()
    q_two = g.stage(cvr.STAGE_Q, (wl.n_cand, 3, 128), torch.bfloat16)

    g.sc.set_option(cvr.OPT_PROFILE, 1)
    g.run()
    assert g.sc.last_launch_count() == 7, "per-kernel events keep one stream"
    assert "tokenizer" in g.sc.stage_times()
    one = g.out()
    q_one = g.stage(cvr.STAGE_Q, (wl.n_cand, 3, 128), torch.bfloat16)

    assert_pcvr_close(two, ref.out, "two streams")
    assert_pcvr_close(one, ref.out, "one stream")
    rel_close(q_two, q_one, 0.02, "first-layer queries, two orders")
    rel_close(q_two, ref.dumps["Q"][0], 0.05, "first-layer queries vs the oracle")


def test_large_encoder_keeps_one_stream():
    # 4 requests x 6,000 positions: 188 encoder tiles, more than half the SMs -> no fork
    wl = synth.make_workload("tiny", n_req=4, n_cand=8, seq_len=(2000, 2000, 2000), user_rows=3000,
                             item_rows=3000, seq_rows=40_000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    g = GpuRun(wl, w, debug=False)
    g.run()
    assert g.sc.last_launch_count() == 7
    assert_pcvr_close(g.out(), oracle.score(wl, w).out, "one stream, large encoder")
