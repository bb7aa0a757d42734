"""The tcgen05 cross-attention kernel (CVR_OPT_ATTENTION_TC): S = Q K^T and O = P V accumulated in tensor
memory, one CTA per 128 candidates and group. Against the oracle on the cases that stress its protocol:
tiles holding several requests (one pass per request), sequence lengths off the 64-position chunk, a sharp
softmax that moves the running max (O rescaled in TMEM), sequences split over several CTAs (state merge,
counters reset for the next call), variable lengths with empty groups, and two interaction layers; and
against the default kernel at the prod shape."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close, rel_close

pytestmark = pytest.mark.gpu


def _tc(g):
    import cvr_ranking_model_gb300 as cvr
    g.sc.set_option(cvr.OPT_ATTENTION_TC, 1)
    return g


def _tokens_close(g, wl, ref, what):
    import torch
    import cvr_ranking_model_gb300 as cvr
    Z = g.stage(cvr.STAGE_Z, (wl.n_cand, 16, 128), torch.bfloat16)
    for gi in range(3):
        rel_close(Z[:, 13 + gi], ref.dumps["Z"][0][:, 13 + gi], 0.05, f"{what}: decoded token {gi}")


def test_ragged_requests_odd_lengths():
    wl = synth.make_workload("tiny", n_req=5, cand_per_req=[1, 70, 3, 64, 9], seq_len=(3, 70, 129),
                             user_rows=5000, item_rows=3000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    g = _tc(GpuRun(wl, w, debug=False))
    g.run()
    ref = oracle.score(wl, w, dumps=True)
    _tokens_close(g, wl, ref, "ragged")
    assert_pcvr_close(g.out(), ref.out, "ragged")


@pytest.mark.parametrize("tc", [0, 1])
def test_sharp_softmax_rescales(tc):
    # tables ~ U(-1, 1) and tau 0.01 make the logits large: for about a tenth of the (row, head) pairs the
    # running max jumps by more than 2^8 between chunks, so O is rescaled. At this temperature the bf16
    # rounding of Q and H alone moves the decoded tokens by ~6% against the fp64 oracle, so the reference is
    # the attention recomputed in fp64 from the kernel's own bf16 Q and H: it isolates the attention kernel.
    import torch
    import cvr_ranking_model_gb300 as cvr
    tau, L = 0.01, (200, 130, 64)
    wl = synth.make_workload("tiny", n_req=3, n_cand=50, seq_len=L, user_rows=3000, item_rows=3000, table_scale=1.0)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05)
    g = GpuRun(wl, w, debug=False, tau=tau)
    g.sc.set_option(cvr.OPT_ATTENTION_TC, tc)
    g.run()
    R, B = wl.n_req, wl.n_cand
    H = g.stage(cvr.STAGE_H, (R * sum(L), 128), torch.bfloat16)
    Q = g.stage(cvr.STAGE_Q, (B, 3, 128), torch.bfloat16)
    Z = g.stage(cvr.STAGE_Z, (B, 16, 128), torch.bfloat16)
    jumps = 0
    for gi in range(3):
        goff = R * sum(L[:gi])
        ref = np.zeros((B, 128))
        for b in range(B):
            Hg = H[goff + wl.req_ids[b] * L[gi]:goff + (wl.req_ids[b] + 1) * L[gi]]
            for h in range(4):
                lg = Hg[:, 32 * h:32 * h + 32] @ Q[b, gi, 32 * h:32 * h + 32] / (tau * np.sqrt(32.0))
                run = np.maximum.accumulate([lg[c:c + 64].max() for c in range(0, L[gi], 64)])
                jumps += int(np.any(np.diff(run) * np.log2(np.e) > 8.0))
                p = np.exp(lg - lg.max())
                ref[b, 32 * h:32 * h + 32] = (p / p.sum()) @ Hg[:, 32 * h:32 * h + 32]
        rel_close(Z[:, 13 + gi], ref, 0.02, f"sharp (tcgen05={tc}): decoded token {gi}")
    assert jumps > 0, "no row's running max moved by more than 8 (log2 units): the rescale path is not covered"


def _long(**kw):
    return synth.make_workload("tiny", seq_len=(600, 1100, 1500), user_rows=3000, item_rows=3000, seq_rows=20000,
                               **kw)


def test_split_sequences_two_calls():
    wl = _long(n_req=3, n_cand=128)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    g = _tc(GpuRun(wl, w, debug=False))
    g.run()
    ref = oracle.score(wl, w, dumps=True)
    _tokens_close(g, wl, ref, "split")
    assert_pcvr_close(g.out(), ref.out, "split")
    g.run()   # the merge counters were reset: a second call gives the same result
    assert_pcvr_close(g.out(), ref.out, "split, second call")


def test_split_variable_lengths_and_ragged_tiles():
    import torch
    wl = _long(n_req=4, cand_per_req=[130, 40, 1, 90])
    w = synth.make_weights(wl.n_layers, wl.seed)
    lens = synth.make_seq_lens(wl, min_len=0, seed=9)
    lens[0] = [0, 100, 1500]   # empty group, one split used of three, every split used
    g = _tc(GpuRun(wl, w, debug=False))
    d_lens = torch.from_numpy(lens).to("cuda:0")
    r, b, o, s, out = g.dw.ptrs()
    g.sc.score_varlen(wl.n_req, wl.n_cand, r, b, o, s, d_lens.data_ptr(), out)
    ref = oracle.score(wl, w, seq_lens=lens)
    assert_pcvr_close(g.out(), ref.out, "split varlen")


def test_two_layers():
    wl = synth.make_workload("deep", n_req=3, n_cand=40, seq_len=(17, 33, 65), user_rows=1000, item_rows=1000,
                             seq_rows=10_000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    g = _tc(GpuRun(wl, w, debug=False))
    g.run()
    ref = oracle.score(wl, w)
    assert_pcvr_close(g.out(), ref.out, "two layers")


def test_prod_shape_agrees_with_default_kernel():
    wl = synth.make_workload("prod")
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    g.run()
    base = g.out()
    _tc(g).run()
    tc = g.out()
    assert np.all(np.isfinite(tc))
    # both kernels are within the oracle tolerance; against each other allow twice that
    err = np.abs(tc - base)
    assert np.all(err <= 2 * (2e-3 + 1e-2 * np.abs(base))), f"max |d| = {err.max():.3e}"
